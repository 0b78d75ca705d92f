/*
 * csa_oracle.h -- plain CPU oracle for compressed sparse attention (CSA) decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link or call this code; only the
 * tests, the smoke check and the benchmark's CPU-baseline leg use it.  It
 * shares no header, helper, table or constant with the CUDA path.
 *
 * Every floating-point quantity is carried in IEEE double.  bf16 inputs are
 * passed as their raw 16-bit patterns and widened exactly to double.
 *
 * Sources (web pages of the nvfp4-megamoe-kernel project):
 *   [Audit rewrite]  "ARCHITECTURE & MEMORY AUDIT -- Post-probe rewrite"
 *   [Audit 1M]       "ARCHITECTURE & MEMORY AUDIT -- 1M-context viability"
 *   [Part A clues]   "PART A -- Next Session Clues"
 *
 * Return codes: 0 = ok, negative = invalid argument or inconsistent input.
 */
#ifndef CSA_ORACLE_H
#define CSA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CSA_ORACLE_OK 0
#define CSA_ORACLE_EINVAL (-1)
#define CSA_ORACLE_EINDEX (-2)      /* a selected index outside [0, n_vis) */
#define CSA_ORACLE_ESWA (-3)        /* a window position no longer resident */
#define CSA_ORACLE_ESOFTMAX (-4)    /* softmax weights failed to sum to one */
#define CSA_ORACLE_ENOMEM (-5)

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int32_t csa_oracle_num_threads(void);

/* Exact widening of a bf16 bit pattern. */
double csa_oracle_bf16_to_f64(uint16_t bits);

/* Compressed blocks visible to a query at absolute position pos: the blocks
 * that strictly precede the (incomplete) block holding pos, capped by the
 * number of blocks the cache holds.  [Part A clues], section 3 (causality). */
int64_t csa_oracle_n_vis(int64_t n_comp, int64_t pos, int32_t ratio);

/* Lightning-indexer score of one compressed block for one query token:
 *   I = sum_h w[h] * max(0, q[h,:] . k[:])
 * One key per block shared by every indexer head (MQA on the indexer).
 * [Audit rewrite], F1 and F3 (eq. 16 of the DSv4 paper, section 2.3.1). */
double csa_oracle_block_score(int32_t n_ih, int32_t ihd, const uint16_t *q,
                              const float *w, const uint16_t *k);

/* Scores of every visible block for T query tokens.
 *   q_idx  [T, n_ih, ihd] bf16 bits     w_idx [T, n_ih] float
 *   k_idx  [R, ihd] bf16 bits, rows of sequence b at comp_off[b] .. comp_off[b+1]
 *   tok_seq [T], tok_pos [T], comp_off [num_seqs+1]
 *   scores [T, ld] double: entry (t, s) written for s < n_vis(t) only
 *   n_vis_out [T] (nullable) */
int32_t csa_oracle_indexer_scores(int32_t T, int32_t n_ih, int32_t ihd, int32_t ratio,
                                  int32_t num_seqs, const int32_t *tok_seq,
                                  const int64_t *tok_pos, const int64_t *comp_off,
                                  const uint16_t *q_idx, const float *w_idx,
                                  const uint16_t *k_idx, double *scores, int64_t ld,
                                  int64_t *n_vis_out);

/* Top-k selection over n scores: orders the blocks by (score descending,
 * block index ascending), keeps the first min(top_k, n), and writes them in
 * ascending block index, padding the rest of idx[0 .. top_k) with -1.
 * -0.0 and +0.0 compare equal.  [Audit rewrite], F3 (total.topk). */
int32_t csa_oracle_topk(int64_t n, const double *scores, int32_t top_k,
                        int32_t *idx, int32_t *n_sel);

/* Rows attended by token t, written as a mixed gather:
 *   rows [0, n_sel)          compressed KV rows comp_kv[comp_off[b] + idx[i]]
 *   rows [n_sel, n_sel+nswa) window positions max(0, p-window+1) .. p,
 *                            oldest first, from swa_kv[b, p mod swa_cap]
 * Both are kept even where they cover the same tokens.
 * kv_buf [T, top_k + window, hd], kv_len [T] = n_sel + nswa.
 * [Audit 1M], D3 and D5; [Part A clues], section 3 (overlap). */
int32_t csa_oracle_gather(int32_t T, int32_t hd, int32_t top_k, int32_t window,
                          int32_t ratio, int32_t num_seqs, const int32_t *tok_seq,
                          const int64_t *tok_pos, const int64_t *comp_off,
                          const int32_t *idx, const int32_t *n_sel,
                          const uint16_t *comp_kv, const uint16_t *swa_kv,
                          int32_t swa_cap, const int64_t *swa_first_pos,
                          uint16_t *kv_buf, int32_t *kv_len);

/* Shared-key-value multi-query attention over the gathered rows:
 *   l_j = scale * q[t,h,:] . row_j,  p_j = exp(l_j - m) / Z,
 *   Z   = sum_j exp(l_j - m) (+ exp(sink[h] - m) when sinks != NULL),
 *   out[t,h,:] = sum_j p_j row_j      (the same row is key and value)
 * q [T, H, hd] bf16 bits, kv_buf [T, rows_per_token, hd] bf16 bits,
 * out [T, H, hd] double.  [Audit 1M], D5 and D6. */
int32_t csa_oracle_attention(int32_t T, int32_t H, int32_t hd, int64_t rows_per_token,
                             const uint16_t *q, const uint16_t *kv_buf,
                             const int32_t *kv_len, double scale, const float *sinks,
                             double *out);

/* The whole decode step: indexer -> top-k -> mixed gather -> attention.
 * scores_out [T, ld] (nullable), idx_out [T, top_k], n_sel_out [T],
 * out [T, H, hd] double. */
int32_t csa_oracle_decode(int32_t T, int32_t num_seqs, const int32_t *tok_seq,
                          const int64_t *tok_pos, const int64_t *comp_off,
                          int32_t n_ih, int32_t ihd, int32_t hd, int32_t H,
                          int32_t top_k, int32_t window, int32_t ratio, double scale,
                          const uint16_t *q_idx, const float *w_idx,
                          const uint16_t *k_idx, const uint16_t *comp_kv,
                          const uint16_t *swa_kv, int32_t swa_cap,
                          const int64_t *swa_first_pos, const uint16_t *q,
                          const float *sinks, double *scores_out, int64_t ld,
                          int32_t *idx_out, int32_t *n_sel_out, double *out);

/* Heavily compressed attention (HCA) decode: no indexer and no selection;
 * every visible compressed row (ratio blocks, typically 128 tokens each) in
 * index order, then the window rows, then the same shared-KV attention.
 * [Audit 1M], D4 ("HCA is dense over compressed entries") and [Audit
 * rewrite] PART 2 (one HCA entry per 128 tokens).  n_vis follows the same
 * strictly-preceding rule.  out [T, H, hd] double; kv_len_out [T] (nullable). */
int32_t csa_oracle_hca_decode(int32_t T, int32_t num_seqs, const int32_t *tok_seq,
                              const int64_t *tok_pos, const int64_t *comp_off, int32_t hd,
                              int32_t H, int32_t window, int32_t ratio, double scale,
                              const uint16_t *comp_kv, const uint16_t *swa_kv, int32_t swa_cap,
                              const int64_t *swa_first_pos, const uint16_t *q,
                              const float *sinks, int32_t *kv_len_out, double *out);

/* FP4 indexer key cache.  [Audit rewrite], C4 and [Audit 1M], M1 cache the
 * indexer keys in FP4 (the paper's section 5.2.1) without fixing a format.
 * Reading: OCP MXFP4.  Elements are e2m1 (sign bit 3; exponent bits 2..1,
 * bias 1; mantissa bit 0: 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives);
 * every 32 consecutive elements share one e8m0 scale 2^(E - 127) with
 * E = floor(log2(amax of the block)) - 2 + 127, clamped to 0 .. 254 (E = 0
 * for an all-zero block).  An element is x / 2^(E-127) rounded to the
 * nearest e2m1 magnitude, ties to the even code, saturating at 6; a zero
 * magnitude is code 0 whatever the sign.
 * One key row (ihd = 128): bytes 0..63 the codes (element 2i in the low
 * nibble of byte i, element 2i+1 in the high nibble), bytes 64..67 the four
 * block scales, bytes 68..79 zero: CSA_ORACLE_FP4_ROW bytes. */
#define CSA_ORACLE_FP4_ROW 80

/* Value of one e2m1 code (low 4 bits). */
double csa_oracle_e2m1_value(uint8_t code);

/* k [R, ihd] bf16 bits -> rows [R, CSA_ORACLE_FP4_ROW]; ihd must be 128. */
int32_t csa_oracle_fp4_quantize(int64_t R, int32_t ihd, const uint16_t *k, uint8_t *rows);

/* rows -> k [R, ihd] bf16 bits.  Every MXFP4 value of a quantized bf16 key is
 * a bf16 value, so this is exact; a row whose values are not bf16 values
 * (hand-made scales out of range) returns CSA_ORACLE_EINVAL. */
int32_t csa_oracle_fp4_dequantize(int64_t R, int32_t ihd, const uint8_t *rows, uint16_t *k);

#ifdef __cplusplus
}
#endif
#endif /* CSA_ORACLE_H */
