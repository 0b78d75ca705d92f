/*
 * csa.h -- C ABI of libcsa.so: compressed sparse attention (CSA) decode on
 * NVIDIA GB300 (sm_103a).
 *
 * One CSA layer, one decode (or chunked-prefill) step, for T query tokens:
 *
 *   1. lightning indexer   I[t,s] = sum_h w[t,h] * ReLU(q^I[t,h] . K^I[s])
 *      over the compressed blocks s visible to token t;
 *   2. top-k               the top_k highest-scoring visible blocks;
 *   3. mixed gather        their compressed rows, then the sliding-window rows;
 *   4. shared-KV MQA       softmax attention of the H query heads over those
 *                          rows, each 512-wide row serving as key and value.
 *
 * Sources (web pages of the nvfp4-megamoe-kernel project):
 *   [Audit rewrite]  "ARCHITECTURE & MEMORY AUDIT -- Post-probe rewrite":
 *                    F1 (128-wide indexer keys shared by the 64 indexer heads),
 *                    F3 (the scoring formula, eq. 16 of the DSv4 paper
 *                    section 2.3.1, and the einsum 'tnd,cd->tnc'), B2 (no silent
 *                    fallback when the top-k is missing), C1 (capacity sized
 *                    by ceil(context / ratio)), C2 (pre-allocated gather buffer).
 *   [Audit 1M]       "ARCHITECTURE & MEMORY AUDIT -- 1M-context viability":
 *                    D3 (gather of selected rows + window), D5 (window kept
 *                    beside the compressed rows), D6 (attention sink),
 *                    M2 (overflow of the compressed buffer), M5 (attention that
 *                    reads rows by index with no gather buffer).
 *   [Part A clues]   "PART A -- Next Session Clues", section 3 (a query sees
 *                    only blocks strictly preceding its own; window and newest
 *                    compressed block are both attended).
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers unless marked (host).  All device buffers
 *     are owned and allocated by the caller; the library never allocates,
 *     frees or synchronises, and keeps no state between calls.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     only enqueued; results are ready when the stream reaches that point.
 *   - Host-side argument errors return before anything is launched.
 *   - Errors found by the kernels (an index out of range, a window row the
 *     ring no longer holds, an inconsistent layout) are OR-ed into the
 *     caller's device word `dev_status` (CSA_DEV_* bits; the caller zeroes it);
 *     the offending row or token is skipped, nothing traps.
 *   - bf16 is IEEE bfloat16 (uint16 storage); f32 is IEEE binary32.
 *   - Every buffer is dense row-major with the shape given; every device
 *     pointer must be 16-byte aligned.
 */
#ifndef CSA_H
#define CSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CSA_ABI_VERSION 1

typedef enum {
    CSA_OK = 0,
    CSA_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size, misaligned buffer */
    CSA_ERR_UNSUPPORTED = 2,      /* dims or device the library does not handle */
    CSA_ERR_CAPACITY = 3,         /* a buffer is smaller than the layout needs */
    CSA_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed */
    CSA_ERR_DEVICE_FAULT = 5,     /* reserved: a device-status bit was read back */
    CSA_ERR_TIMEOUT = 6,          /* reserved: a bounded device wait gave up */
    CSA_ERR_WORKSPACE = 7         /* workspace missing or smaller than csa_workspace_size */
} csa_status_t;

/* Bits OR-ed into *dev_status by the kernels. */
#define CSA_DEV_BAD_INDEX   0x01  /* idx outside [0, n_vis) for a selected slot */
#define CSA_DEV_MISSING_SWA 0x02  /* a window position below swa_first_pos */
#define CSA_DEV_BAD_LAYOUT  0x04  /* tok_seq outside [0,B), tok_pos < 0, bad comp_off */
#define CSA_DEV_CAPACITY    0x08  /* a sequence holds more blocks than max_comp_rows */
#define CSA_DEV_BAD_LENGTH  0x10  /* kv_len outside [0, top_k + window] */
#define CSA_DEV_TIMEOUT     0x20  /* a bounded wait inside a kernel gave up */
#define CSA_DEV_CHECK       0x40  /* libcsa_checks.so only: an index inside the library
                                     left its array; the access was skipped */

/* Where each query token's rows live.  Device arrays unless marked (host).
 * The library's kernels may read tok_seq, tok_pos, comp_off and
 * swa_first_pos as soon as they start, while a preceding kernel that allows
 * programmatic dependent launch may still run: these arrays must not be
 * written by such a kernel (the library's own kernels never write them; a
 * copy, or a kernel without that launch attribute, completes before the
 * next one starts).  Everything else a call reads (queries, weights, keys,
 * rows, the window ring) is read only after the preceding kernel has
 * finished. */
typedef struct {
    int32_t num_seqs;               /* (host) B >= 1 */
    int32_t num_tokens;             /* (host) T >= 0 */
    int64_t total_comp_rows;        /* (host) R = comp_off[B], rows in k_idx / comp_kv */
    int64_t max_comp_rows;          /* (host) upper bound of comp_off[b+1]-comp_off[b];
                                       sizes grids and workspace without a device read */
    const int32_t *tok_seq;         /* [T] sequence of each query token */
    const int64_t *tok_pos;         /* [T] absolute 0-based position of each query token */
    const int64_t *comp_off;        /* [B+1] block b of sequence s is row comp_off[s] + b */
    const void *swa_kv;             /* bf16 [B, swa_cap, hd]: position p at slot p % swa_cap */
    int32_t swa_cap;                /* (host) ring slots per sequence, >= window */
    const int64_t *swa_first_pos;   /* [B] oldest position the ring still holds */
} csa_layout_t;

/* Problem constants.  The library supports n_ih = 64, ihd = 128, hd = 512,
 * n_heads a multiple of 16 up to 128, 1 <= top_k <= 2048, window <= swa_cap. */
typedef struct {
    int32_t n_ih;     /* indexer heads (64) */
    int32_t ihd;      /* indexer head dim = width of the shared block key (128) */
    int32_t hd;       /* main head dim = width of a compressed / window row (512) */
    int32_t n_heads;  /* main query heads H */
    int32_t top_k;    /* selected blocks per token (1024) */
    int32_t window;   /* sliding-window rows per token (128) */
    int32_t ratio;    /* tokens per compressed block (4 for CSA) */
    float scale;      /* attention logit scale (1/sqrt(hd)) */
} csa_params_t;

/* Derived rule used by every entry point ([Part A clues], section 3):
 *   n_vis(t) = min(comp_off[b+1] - comp_off[b], floor(tok_pos[t] / ratio)),
 *   b = tok_seq[t]: token t sees blocks 0 .. n_vis(t)-1 of its sequence.
 * Window of token t: positions max(0, p - window + 1) .. p, p = tok_pos[t]. */

/* Human-readable name of a status code (static storage). */
const char *csa_status_string(csa_status_t status);

/* CSA_ABI_VERSION of the loaded library. */
int32_t csa_abi_version(void);

/* Bytes of workspace `ws` that csa_topk, csa_indexer_topk,
 * csa_sparse_mqa_decode and csa_decode need for this layout and these params
 * (one size serves all of them).
 * The workspace is device memory, 256-byte aligned, owned by the caller.
 * Its front holds per-token top-k state (16640 bytes per token) that must be
 * zero when a call starts: zero-fill the workspace once after allocating it.
 * Every call that completes without error leaves that state zero again, so
 * the workspace is reused with no memset.  Scratch data is packed against
 * the END of the buffer, so a workspace sized for the largest call (most
 * tokens, most blocks) serves every smaller call as well.  After a call that
 * returned an error or set a dev_status bit, zero the workspace again.
 * Calls that may run concurrently (different streams) need separate
 * workspaces.  Returns CSA_ERR_INVALID_ARGUMENT / CSA_ERR_UNSUPPORTED on bad
 * input. */
csa_status_t csa_workspace_size(const csa_layout_t *layout, const csa_params_t *params,
                                size_t *bytes /* (host) out */);

/* Step 1, the lightning indexer ([Audit rewrite], F1 and F3):
 *   scores[t, s] = sum_h w_idx[t,h] * max(0, sum_d q_idx[t,h,d] * k_idx[comp_off[b]+s, d])
 * for s < n_vis(t); entries s >= n_vis(t) are not written.
 *   q_idx  bf16 [T, n_ih, ihd]     w_idx f32 [T, n_ih]
 *   k_idx  bf16 [R, ihd]           scores f32 [T, ld_scores], ld_scores >= max_comp_rows.
 * Products are exact (bf16 x bf16), sums are f32 (tensor-core accumulation
 * over d, then a fixed-order sum over h).  The result does not depend on the
 * stream, launch order or other tokens. */
csa_status_t csa_indexer_scores(const csa_layout_t *layout, const csa_params_t *params,
                                const void *q_idx, const float *w_idx, const void *k_idx,
                                float *scores, int64_t ld_scores, int32_t *dev_status,
                                void *stream);

/* Step 2, top-k over the visible scores ([Audit rewrite], F3: total.topk):
 * keeps k'(t) = min(top_k, n_vis(t)) blocks ranked by (score descending,
 * block index ascending; -0.0 ties with +0.0), writes them to idx[t, 0..k')
 * in ascending block index and -1 in idx[t, k'..top_k); n_sel[t] = k'.
 *   scores f32 [T, ld_scores] (as written by csa_indexer_scores; NaN unsupported)
 *   idx    int32 [T, top_k]      n_sel int32 [T]
 * Exact: the selection is a pure function of the scores' bits. */
csa_status_t csa_topk(const csa_layout_t *layout, const csa_params_t *params,
                      const float *scores, int64_t ld_scores, int32_t *idx, int32_t *n_sel,
                      int32_t *dev_status, void *ws, size_t ws_bytes, void *stream);

/* Steps 1 and 2 in one call ([Audit rewrite], F3: the scores feed
 * total.topk): idx / n_sel exactly as csa_topk writes them for the scores
 * csa_indexer_scores computes, without handing the scores to the caller.
 * For decode batches (one query token per key tile: more than one sequence,
 * or fewer than four tokens) the selection runs inside the indexer kernel:
 * each CTA keeps the candidates of its key range on chip and the last one to
 * finish a token selects from them (an exact fallback over the token's whole
 * score row covers the inputs where the candidates cannot prove the result,
 * such as long runs of tied scores).  Other layouts run the indexer and
 * csa_topk's kernels back to back.
 *   q_idx bf16 [T, n_ih, ihd], w_idx f32 [T, n_ih], k_idx bf16 [R, ihd],
 *   idx int32 [T, top_k], n_sel int32 [T], ws as for csa_topk. */
csa_status_t csa_indexer_topk(const csa_layout_t *layout, const csa_params_t *params,
                              const void *q_idx, const float *w_idx, const void *k_idx,
                              int32_t *idx, int32_t *n_sel, int32_t *dev_status, void *ws,
                              size_t ws_bytes, void *stream);

/* Step 3, mixed gather into a caller-owned buffer ([Audit 1M], D3 and D5;
 * [Audit rewrite], C2):
 *   kv_buf[t, i]          = comp_kv[comp_off[b] + idx[t, i]],  i < n_sel[t]
 *   kv_buf[t, n_sel + j]  = swa_kv[b, x_j % swa_cap],  x_j = first + j, oldest first
 *   kv_len[t]             = n_sel[t] + (p - first + 1)
 * Both the compressed rows and the window rows are kept even where they cover
 * the same tokens.  Rows kv_buf[t, kv_len[t] ..) are left untouched.
 *   idx int32 [T, top_k], n_sel int32 [T], comp_kv bf16 [R, hd],
 *   kv_buf bf16 [T, top_k + window, hd], kv_len int32 [T].
 * An idx outside [0, n_vis(t)) sets CSA_DEV_BAD_INDEX and that row is
 * written as zeros (no clamping); a window position the ring no longer holds
 * sets CSA_DEV_MISSING_SWA and that row is written as zeros. */
csa_status_t csa_gather_mixed(const csa_layout_t *layout, const csa_params_t *params,
                              const int32_t *idx, const int32_t *n_sel, const void *comp_kv,
                              void *kv_buf, int32_t *kv_len, int32_t *dev_status,
                              void *stream);

/* Step 4, shared-KV multi-query attention over gathered rows ([Audit 1M], D5):
 *   l_j = scale * q[t,h,:] . kv_buf[t,j,:],  j < kv_len[t]
 *   out[t,h,:] = sum_j softmax_j(l) * kv_buf[t,j,:]
 * With sinks != NULL (f32 [H]), exp(sinks[h] - max) joins the softmax
 * denominator of head h ([Audit 1M], D6); NULL means no sink.
 *   q bf16 [T, H, hd], kv_buf bf16 [T, top_k + window, hd], kv_len int32 [T],
 *   out f32 [T, H, hd].  kv_len[t] = 0 gives out[t] = 0.
 * bf16 x bf16 products on tensor cores, f32 accumulation and softmax. */
csa_status_t csa_sparse_mqa_decode(int32_t num_tokens, const csa_params_t *params,
                                   const void *q, const void *kv_buf, const int32_t *kv_len,
                                   const float *sinks, float *out, int32_t *dev_status,
                                   void *ws, size_t ws_bytes, void *stream);

/* Steps 1-4 fused ([Audit 1M], M5): the indexer feeds the top-k through the
 * workspace, and attention reads the selected compressed rows by index
 * straight from comp_kv and the window rows straight from the ring; no
 * gather buffer exists.  Same inputs and outputs as the four calls above;
 * idx_out (nullable, int32 [T, top_k]) receives the selection exactly as
 * csa_topk would write it for the scores csa_indexer_scores computes. */
csa_status_t csa_decode(const csa_layout_t *layout, const csa_params_t *params,
                        const void *q_idx, const float *w_idx, const void *k_idx,
                        const void *comp_kv, const void *q, const float *sinks, float *out,
                        int32_t *idx_out, int32_t *dev_status, void *ws, size_t ws_bytes,
                        void *stream);

/* Heavily compressed attention (HCA) decode ([Audit 1M], D4: HCA layers run
 * no indexer and attend densely over every compressed entry; [Audit rewrite]
 * PART 2: one entry per 128 tokens).  Token t attends every visible block
 * 0 .. n_vis(t)-1 of its sequence (the same strictly-preceding rule, with
 * params->ratio = 128 for HCA) in index order, then its window rows, with
 * the same shared-KV attention as csa_sparse_mqa_decode; no selection and no
 * gather buffer (rows are read in place).  params->top_k is not used.
 *   comp_kv bf16 [R, hd], q bf16 [T, H, hd], sinks f32 [H] (nullable),
 *   out f32 [T, H, hd].  Workspace: csa_hca_workspace_size bytes, same
 *   contract as csa_workspace_size. */
csa_status_t csa_hca_workspace_size(const csa_layout_t *layout, const csa_params_t *params,
                                    size_t *bytes /* (host) out */);

csa_status_t csa_hca_decode(const csa_layout_t *layout, const csa_params_t *params,
                            const void *comp_kv, const void *q, const float *sinks, float *out,
                            int32_t *dev_status, void *ws, size_t ws_bytes, void *stream);

/* Sharded single-sequence decode ([Audit 1M], PART 2, "Total KV cache @ 1M
 * context": the KV cache sharded across GPUs).  One sequence (num_seqs == 1,
 * else CSA_ERR_UNSUPPORTED) whose compressed blocks are cut into contiguous
 * ranges: shard g holds blocks [lo_g, hi_g) as rows 0 .. hi_g - lo_g - 1 of
 * its own k_idx and comp_kv (the same row formats as above).  `layout` is the
 * whole sequence's layout as every other call takes it (comp_off = {0,
 * n_comp}); a shard's own caches replace k_idx / comp_kv.  One step:
 *   1. each shard: csa_shard_candidates -> its k' = min(top_k, its visible
 *      blocks) best blocks, global block indices and the scores they won on;
 *   2. exchange the candidates (all-gather), then csa_shard_merge on any
 *      device: the global top-k by (score descending, block index ascending),
 *      identical to csa_topk on the whole score row, because a block of the
 *      global top-k is among its own shard's k best;
 *   3. each shard: csa_shard_attention over its own selected rows, and one
 *      device csa_window_attention over the window rows: unnormalised
 *      partials (O scaled to m, m in log2 units, l), no sink;
 *   4. exchange the partials, then csa_shard_combine: the log-sum-exp merge,
 *      the sink (if any) in the denominator.
 * No call communicates: the exchanges are the caller's (NCCL all-gathers,
 * or plain copies on one device).  Buffers are device memory, caller-owned.
 *
 * csa_shard_workspace_size: bytes of workspace for the shard calls with this
 * range (zeroed once before first use, as for csa_decode).
 * csa_shard_candidates: cand_score f32 [T, top_k], cand_idx int32 [T, top_k]
 * (global indices, -1 past n_cand[t]), n_cand int32 [T].
 * csa_shard_merge: shard_bounds (host) int64 [G + 1], G <= 8, lo_0 <= ... <=
 * hi_{G-1}; cand_* [G][T][top_k] and n_cand [G][T] as gathered; writes idx
 * int32 [T, top_k] (global, ascending, -1 padded), n_sel [T], shard_idx int32
 * [G][T][top_k] (each shard's part of idx in its own rows, ascending) and
 * shard_nsel [G][T].  A candidate index outside [0, hi_{G-1}) sets
 * CSA_DEV_BAD_INDEX and is dropped; a count outside [0, top_k] sets
 * CSA_DEV_BAD_LENGTH and is clamped.  G * top_k <= 16384.
 * csa_shard_attention: shard_idx / shard_nsel as the merge gave them for
 * this shard ([T][top_k], [T]); part_o f32 [T, H, 512], part_ml f32 [T, H, 2].
 * csa_window_attention: the window rows of every token (from the layout's
 * ring), as a partial of the same form.
 * csa_shard_combine: num_parts partials laid out [P][T][H][512] and
 * [P][T][H][2] (P <= 256) -> out f32 [T, H, 512]; a partial with m = -inf
 * carries no rows. */
csa_status_t csa_shard_workspace_size(const csa_layout_t *layout, const csa_params_t *params,
                                      int64_t shard_lo, int64_t shard_hi,
                                      size_t *bytes /* (host) out */);

csa_status_t csa_shard_candidates(const csa_layout_t *layout, const csa_params_t *params,
                                  int64_t shard_lo, int64_t shard_hi, const void *q_idx,
                                  const float *w_idx, const void *k_idx_shard, float *cand_score,
                                  int32_t *cand_idx, int32_t *n_cand, int32_t *dev_status, void *ws,
                                  size_t ws_bytes, void *stream);

csa_status_t csa_shard_merge(int32_t num_tokens, int32_t top_k, int32_t num_shards,
                             const int64_t *shard_bounds /* (host) */, const float *cand_score,
                             const int32_t *cand_idx, const int32_t *n_cand, int32_t *idx,
                             int32_t *n_sel, int32_t *shard_idx, int32_t *shard_nsel,
                             int32_t *dev_status, void *stream);

csa_status_t csa_shard_attention(const csa_layout_t *layout, const csa_params_t *params,
                                 int64_t shard_lo, int64_t shard_hi, const int32_t *shard_idx,
                                 const int32_t *shard_nsel, const void *comp_kv_shard,
                                 const void *q, float *part_o, float *part_ml, int32_t *dev_status,
                                 void *ws, size_t ws_bytes, void *stream);

csa_status_t csa_window_attention(const csa_layout_t *layout, const csa_params_t *params,
                                  const void *q, float *part_o, float *part_ml,
                                  int32_t *dev_status, void *ws, size_t ws_bytes, void *stream);

csa_status_t csa_shard_combine(int32_t num_parts, int32_t num_tokens, int32_t n_heads,
                               const float *part_o, const float *part_ml, const float *sinks,
                               float *out, int32_t *dev_status, void *stream);

/* FP4 indexer key cache ([Audit rewrite], C4, and [Audit 1M], M1: the
 * indexer keys are cached in FP4, the paper's section 5.2.1).  The pages fix
 * no format; this library reads it as OCP MXFP4: e2m1 elements (0, 0.5, 1,
 * 1.5, 2, 3, 4, 6 and negatives), one e8m0 scale 2^(E-127) per 32 elements
 * with E = floor(log2(block amax)) - 2 + 127 (clamped to 0..254; 0 for an
 * all-zero block), elements rounded to the nearest value, ties to the even
 * code, saturating at 6, a zero stored as code 0.  One key (ihd = 128) is an
 * 80-byte row: bytes 0..63 the codes (element 2i in the low nibble of byte
 * i, 2i+1 in the high nibble), bytes 64..67 the four block scales, bytes
 * 68..79 zero (rows stay 16-byte aligned for the bulk-copy engine).
 *
 * csa_fp4_quantize_keys: k_idx bf16 [rows, 128] -> k_fp4 uint8 [rows, 80],
 * both device pointers, 16-byte aligned.  Row by row and deterministic, so a
 * cache may quantize rows as it appends them.
 *
 * csa_indexer_scores_fp4 and csa_decode_fp4: csa_indexer_scores and
 * csa_decode with the keys given as such rows (k_fp4 uint8 [R, 80]).  The
 * scores are exactly those of the bf16 indexer on the dequantized keys
 * (every MXFP4 value of a bf16 key is itself a bf16 value); the kernel reads
 * 80 bytes per key instead of 256 and expands the codes in shared memory.
 * Tokens are scored one per key tile (no grouping of prefill tokens).
 * Same errors as the bf16 calls; k_fp4 must be 16-byte aligned. */
csa_status_t csa_fp4_quantize_keys(int64_t rows, const void *k_idx, void *k_fp4, void *stream);

csa_status_t csa_indexer_scores_fp4(const csa_layout_t *layout, const csa_params_t *params,
                                    const void *q_idx, const float *w_idx, const void *k_fp4,
                                    float *scores, int64_t ld_scores, int32_t *dev_status,
                                    void *stream);

csa_status_t csa_decode_fp4(const csa_layout_t *layout, const csa_params_t *params,
                            const void *q_idx, const float *w_idx, const void *k_fp4,
                            const void *comp_kv, const void *q, const float *sinks, float *out,
                            int32_t *idx_out, int32_t *dev_status, void *ws, size_t ws_bytes,
                            void *stream);

/* csa_topk without a workspace, for callers that cannot allocate device
 * memory at all: an engine whose memory planner owns every byte of the GPU,
 * or a plug-in that is not allowed to call the allocator, cannot hand
 * csa_topk the workspace it needs.  The pages have no counterpart: this is a
 * deployment convenience, not a step of the method.
 *
 * Same arguments, results and errors as csa_topk minus ws/ws_bytes (the
 * same checks run in the same order, so a bad input gets the same code).  The
 * scratch is a fixed 260 KiB array inside libcsa.so, reserved on every GPU
 * that loads the library until the process exits; it limits a call to at
 * most 16 query tokens: more returns CSA_ERR_CAPACITY.  top_k above 2048
 * returns CSA_ERR_UNSUPPORTED, as it does for csa_topk.
 * Each token's selection runs in one thread block here, so long rows take
 * longer than with csa_topk.
 * The first call on a device looks up the array's device address (a one-time
 * set-up per device); make that first call before any stream capture.  Every
 * call reuses the same array and clears the part that must start at zero, so
 * calls that overlap on the GPU (two streams, two threads) race: serialise
 * them. */
csa_status_t csa_topk_noalloc(const csa_layout_t *layout, const csa_params_t *params,
                              const float *scores, int64_t ld_scores, int32_t *idx,
                              int32_t *n_sel, int32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* CSA_H */
