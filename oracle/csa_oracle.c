/*
 * csa_oracle.c -- plain CPU oracle for compressed sparse attention decode.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path.  It is written
 * straight from the definitions on the pages (see csa_oracle.h for the page
 * titles) with no blocking, fusion or reordering: each step is a loop over
 * the quantities the definition names, in double precision.
 *
 * Parity pins (tests/test_oracle_*.py): closed-form indexer cases, one-hot
 * head weights reducing to a matrix-vector product, brute-force top-k over
 * every subset on tiny inputs, hand-derived visibility tables, attention
 * special cases (one row, identical rows, q = 0, permutation) and dense
 * softmax attention from a library routine when top_k covers every block.
 */
#include "csa_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int32_t csa_oracle_num_threads(void) {
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}

double csa_oracle_bf16_to_f64(uint16_t bits) {
    /* bf16 is the top half of an IEEE binary32. */
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* [Part A clues], section 3: a decode query sees only the compressed blocks
 * strictly preceding its own, still incomplete, block.  The block holding
 * position pos is floor(pos / ratio); the blocks before it are
 * 0 .. floor(pos / ratio) - 1.  The cache cannot offer more than it holds. */
int64_t csa_oracle_n_vis(int64_t n_comp, int64_t pos, int32_t ratio) {
    if (pos < 0 || ratio < 1 || n_comp < 0) return -1;
    int64_t preceding = pos / ratio;
    return preceding < n_comp ? preceding : n_comp;
}

/* [Audit rewrite], F3: I[t,s] = sum_h w[t,h] * ReLU(q[t,h] . K[s]). */
double csa_oracle_block_score(int32_t n_ih, int32_t ihd, const uint16_t *q,
                              const float *w, const uint16_t *k) {
    double total = 0.0;
    for (int32_t h = 0; h < n_ih; ++h) {
        double dot = 0.0;
        for (int32_t d = 0; d < ihd; ++d)
            dot += csa_oracle_bf16_to_f64(q[(int64_t)h * ihd + d]) *
                   csa_oracle_bf16_to_f64(k[d]);
        double relu = dot > 0.0 ? dot : 0.0;
        total += (double)w[h] * relu;
    }
    return total;
}

static int check_token(int32_t t, int32_t num_seqs, const int32_t *tok_seq,
                       const int64_t *tok_pos, const int64_t *comp_off) {
    int32_t b = tok_seq[t];
    if (b < 0 || b >= num_seqs) return 0;
    if (tok_pos[t] < 0) return 0;
    if (comp_off[b + 1] < comp_off[b]) return 0;
    return 1;
}

int32_t csa_oracle_indexer_scores(int32_t T, int32_t n_ih, int32_t ihd, int32_t ratio,
                                  int32_t num_seqs, const int32_t *tok_seq,
                                  const int64_t *tok_pos, const int64_t *comp_off,
                                  const uint16_t *q_idx, const float *w_idx,
                                  const uint16_t *k_idx, double *scores, int64_t ld,
                                  int64_t *n_vis_out) {
    if (T < 0 || n_ih < 1 || ihd < 1 || ratio < 1 || num_seqs < 1) return CSA_ORACLE_EINVAL;
    for (int32_t t = 0; t < T; ++t)
        if (!check_token(t, num_seqs, tok_seq, tok_pos, comp_off)) return CSA_ORACLE_EINVAL;
    for (int32_t t = 0; t < T; ++t) {
        int32_t b = tok_seq[t];
        int64_t n_comp = comp_off[b + 1] - comp_off[b];
        int64_t nv = csa_oracle_n_vis(n_comp, tok_pos[t], ratio);
        if (nv > ld) return CSA_ORACLE_EINVAL;
        if (n_vis_out) n_vis_out[t] = nv;
        const uint16_t *qt = q_idx + (int64_t)t * n_ih * ihd;
        const float *wt = w_idx + (int64_t)t * n_ih;
        const uint16_t *kb = k_idx + comp_off[b] * (int64_t)ihd;
        double *st = scores + (int64_t)t * ld;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
        for (int64_t s = 0; s < nv; ++s)
            st[s] = csa_oracle_block_score(n_ih, ihd, qt, wt, kb + s * (int64_t)ihd);
    }
    return CSA_ORACLE_OK;
}

/* ---- top-k ------------------------------------------------------------ */

typedef struct {
    double score;
    int64_t index;
} ranked_t;

/* Order: larger score first; among equal scores the lower block index first.
 * Comparing doubles makes -0.0 and +0.0 equal, as the selection wants. */
static int rank_cmp(const void *a, const void *b) {
    const ranked_t *x = (const ranked_t *)a, *y = (const ranked_t *)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->index > y->index) - (x->index < y->index);
}

static int int32_cmp(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

int32_t csa_oracle_topk(int64_t n, const double *scores, int32_t top_k, int32_t *idx,
                        int32_t *n_sel) {
    if (n < 0 || top_k < 1) return CSA_ORACLE_EINVAL;
    for (int64_t i = 0; i < n; ++i)
        if (scores[i] != scores[i]) return CSA_ORACLE_EINVAL; /* NaN unsupported */
    int64_t kk = n < (int64_t)top_k ? n : (int64_t)top_k;
    ranked_t *r = NULL;
    if (n > 0) {
        r = (ranked_t *)malloc((size_t)n * sizeof *r);
        if (!r) return CSA_ORACLE_ENOMEM;
        for (int64_t i = 0; i < n; ++i) {
            r[i].score = scores[i];
            r[i].index = i;
        }
        qsort(r, (size_t)n, sizeof *r, rank_cmp);
    }
    for (int64_t i = 0; i < kk; ++i) idx[i] = (int32_t)r[i].index;
    qsort(idx, (size_t)kk, sizeof *idx, int32_cmp);
    for (int64_t i = kk; i < top_k; ++i) idx[i] = -1;
    *n_sel = (int32_t)kk;
    free(r);
    return CSA_ORACLE_OK;
}

/* ---- mixed gather ----------------------------------------------------- */

int32_t csa_oracle_gather(int32_t T, int32_t hd, int32_t top_k, int32_t window,
                          int32_t ratio, int32_t num_seqs, const int32_t *tok_seq,
                          const int64_t *tok_pos, const int64_t *comp_off,
                          const int32_t *idx, const int32_t *n_sel,
                          const uint16_t *comp_kv, const uint16_t *swa_kv,
                          int32_t swa_cap, const int64_t *swa_first_pos,
                          uint16_t *kv_buf, int32_t *kv_len) {
    if (T < 0 || hd < 1 || top_k < 1 || window < 1 || swa_cap < window || ratio < 1)
        return CSA_ORACLE_EINVAL;
    int64_t rows_per_token = (int64_t)top_k + window;
    for (int32_t t = 0; t < T; ++t) {
        if (!check_token(t, num_seqs, tok_seq, tok_pos, comp_off)) return CSA_ORACLE_EINVAL;
        int32_t b = tok_seq[t];
        int64_t p = tok_pos[t];
        int64_t nv = csa_oracle_n_vis(comp_off[b + 1] - comp_off[b], p, ratio);
        int32_t ns = n_sel[t];
        if (ns < 0 || ns > top_k) return CSA_ORACLE_EINDEX;
        uint16_t *dst = kv_buf + (int64_t)t * rows_per_token * hd;
        int64_t r = 0;
        for (int32_t i = 0; i < ns; ++i, ++r) {
            int32_t s = idx[(int64_t)t * top_k + i];
            if (s < 0 || (int64_t)s >= nv) return CSA_ORACLE_EINDEX;
            memcpy(dst + r * hd, comp_kv + (comp_off[b] + s) * (int64_t)hd,
                   (size_t)hd * sizeof(uint16_t));
        }
        /* Sliding window: the last `window` positions up to and including p. */
        int64_t first = p - window + 1;
        if (first < 0) first = 0;
        for (int64_t x = first; x <= p; ++x, ++r) {
            if (r >= rows_per_token) return CSA_ORACLE_EINVAL;
            if (x < swa_first_pos[b]) return CSA_ORACLE_ESWA;
            int64_t slot = x % swa_cap;
            memcpy(dst + r * hd, swa_kv + ((int64_t)b * swa_cap + slot) * hd,
                   (size_t)hd * sizeof(uint16_t));
        }
        kv_len[t] = (int32_t)r;
    }
    return CSA_ORACLE_OK;
}

/* ---- attention -------------------------------------------------------- */

int32_t csa_oracle_attention(int32_t T, int32_t H, int32_t hd, int64_t rows_per_token,
                             const uint16_t *q, const uint16_t *kv_buf,
                             const int32_t *kv_len, double scale, const float *sinks,
                             double *out) {
    if (T < 0 || H < 1 || hd < 1 || rows_per_token < 1) return CSA_ORACLE_EINVAL;
    for (int32_t t = 0; t < T; ++t)
        if (kv_len[t] < 0 || kv_len[t] > rows_per_token) return CSA_ORACLE_EINVAL;
    int32_t status = CSA_ORACLE_OK;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t th = 0; th < (int64_t)T * H; ++th) {
        int64_t t = th / H, h = th % H;
        int64_t L = kv_len[t];
        const uint16_t *qh = q + (t * H + h) * (int64_t)hd;
        const uint16_t *rows = kv_buf + t * rows_per_token * (int64_t)hd;
        double *o = out + (t * H + h) * (int64_t)hd;
        double *logit = (double *)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
        if (!logit) {
#ifdef _OPENMP
#pragma omp critical
#endif
            status = CSA_ORACLE_ENOMEM;
            continue;
        }
        /* logits: the shared row is the key */
        double m = -INFINITY;
        for (int64_t j = 0; j < L; ++j) {
            double dot = 0.0;
            for (int32_t d = 0; d < hd; ++d)
                dot += csa_oracle_bf16_to_f64(qh[d]) *
                       csa_oracle_bf16_to_f64(rows[j * hd + d]);
            logit[j] = scale * dot;
            if (logit[j] > m) m = logit[j];
        }
        if (sinks && (double)sinks[h] > m) m = (double)sinks[h];
        double z = 0.0;
        for (int64_t j = 0; j < L; ++j) z += exp(logit[j] - m);
        double zsink = sinks ? exp((double)sinks[h] - m) : 0.0;
        z += zsink;
        /* the same shared row is the value */
        for (int32_t d = 0; d < hd; ++d) o[d] = 0.0;
        double wsum = 0.0;
        for (int64_t j = 0; j < L; ++j) {
            double p = exp(logit[j] - m) / z;
            wsum += p;
            for (int32_t d = 0; d < hd; ++d) o[d] += p * csa_oracle_bf16_to_f64(rows[j * hd + d]);
        }
        /* The weights (with the sink's share) form a distribution. */
        if (z > 0.0 && fabs(wsum + zsink / z - 1.0) > 1e-9) {
#ifdef _OPENMP
#pragma omp critical
#endif
            status = CSA_ORACLE_ESOFTMAX;
        }
        free(logit);
    }
    return status;
}

/* ---- the whole step --------------------------------------------------- */

int32_t csa_oracle_decode(int32_t T, int32_t num_seqs, const int32_t *tok_seq,
                          const int64_t *tok_pos, const int64_t *comp_off,
                          int32_t n_ih, int32_t ihd, int32_t hd, int32_t H,
                          int32_t top_k, int32_t window, int32_t ratio, double scale,
                          const uint16_t *q_idx, const float *w_idx,
                          const uint16_t *k_idx, const uint16_t *comp_kv,
                          const uint16_t *swa_kv, int32_t swa_cap,
                          const int64_t *swa_first_pos, const uint16_t *q,
                          const float *sinks, double *scores_out, int64_t ld,
                          int32_t *idx_out, int32_t *n_sel_out, double *out) {
    if (T < 0 || top_k < 1 || window < 1) return CSA_ORACLE_EINVAL;
    int64_t max_vis = 0;
    for (int32_t t = 0; t < T; ++t) {
        if (!check_token(t, num_seqs, tok_seq, tok_pos, comp_off)) return CSA_ORACLE_EINVAL;
        int32_t b = tok_seq[t];
        int64_t nv = csa_oracle_n_vis(comp_off[b + 1] - comp_off[b], tok_pos[t], ratio);
        if (nv > max_vis) max_vis = nv;
    }
    int64_t lds = scores_out ? ld : (max_vis > 0 ? max_vis : 1);
    if (lds < max_vis) return CSA_ORACLE_EINVAL;
    double *scores = scores_out;
    if (!scores) {
        scores = (double *)malloc((size_t)T * (size_t)lds * sizeof(double) + 8);
        if (!scores) return CSA_ORACLE_ENOMEM;
    }
    int64_t *n_vis = (int64_t *)malloc((size_t)(T > 0 ? T : 1) * sizeof(int64_t));
    int64_t rows_per_token = (int64_t)top_k + window;
    uint16_t *kv_buf = (uint16_t *)malloc((size_t)(T > 0 ? T : 1) * (size_t)rows_per_token *
                                          (size_t)hd * sizeof(uint16_t));
    int32_t *kv_len = (int32_t *)malloc((size_t)(T > 0 ? T : 1) * sizeof(int32_t));
    int32_t st = CSA_ORACLE_ENOMEM;
    if (!n_vis || !kv_buf || !kv_len) goto done;

    st = csa_oracle_indexer_scores(T, n_ih, ihd, ratio, num_seqs, tok_seq, tok_pos, comp_off,
                                   q_idx, w_idx, k_idx, scores, lds, n_vis);
    if (st) goto done;
    for (int32_t t = 0; t < T; ++t) {
        st = csa_oracle_topk(n_vis[t], scores + (int64_t)t * lds, top_k,
                             idx_out + (int64_t)t * top_k, n_sel_out + t);
        if (st) goto done;
    }
    st = csa_oracle_gather(T, hd, top_k, window, ratio, num_seqs, tok_seq, tok_pos, comp_off,
                           idx_out, n_sel_out, comp_kv, swa_kv, swa_cap, swa_first_pos,
                           kv_buf, kv_len);
    if (st) goto done;
    st = csa_oracle_attention(T, H, hd, rows_per_token, q, kv_buf, kv_len, scale, sinks, out);
done:
    if (!scores_out) free(scores);
    free(n_vis);
    free(kv_buf);
    free(kv_len);
    return st;
}

/* ---- HCA: dense over every visible compressed row --------------------- */

int32_t csa_oracle_hca_decode(int32_t T, int32_t num_seqs, const int32_t *tok_seq,
                              const int64_t *tok_pos, const int64_t *comp_off, int32_t hd,
                              int32_t H, int32_t window, int32_t ratio, double scale,
                              const uint16_t *comp_kv, const uint16_t *swa_kv, int32_t swa_cap,
                              const int64_t *swa_first_pos, const uint16_t *q,
                              const float *sinks, int32_t *kv_len_out, double *out) {
    if (T < 0 || window < 1 || ratio < 1) return CSA_ORACLE_EINVAL;
    int64_t max_vis = 0;
    for (int32_t t = 0; t < T; ++t) {
        if (!check_token(t, num_seqs, tok_seq, tok_pos, comp_off)) return CSA_ORACLE_EINVAL;
        int32_t b = tok_seq[t];
        int64_t nv = csa_oracle_n_vis(comp_off[b + 1] - comp_off[b], tok_pos[t], ratio);
        if (nv > max_vis) max_vis = nv;
    }
    /* every visible block is "selected": the mixed gather with idx = 0..n_vis-1 */
    int32_t k_all = (int32_t)(max_vis > 0 ? max_vis : 1);
    int64_t rows_per_token = (int64_t)k_all + window;
    int32_t *idx = (int32_t *)malloc((size_t)(T > 0 ? T : 1) * (size_t)k_all * sizeof(int32_t));
    int32_t *n_sel = (int32_t *)malloc((size_t)(T > 0 ? T : 1) * sizeof(int32_t));
    int32_t *kv_len = (int32_t *)malloc((size_t)(T > 0 ? T : 1) * sizeof(int32_t));
    uint16_t *kv_buf = (uint16_t *)malloc((size_t)(T > 0 ? T : 1) * (size_t)rows_per_token *
                                          (size_t)hd * sizeof(uint16_t));
    int32_t st = CSA_ORACLE_ENOMEM;
    if (!idx || !n_sel || !kv_len || !kv_buf) goto done;
    for (int32_t t = 0; t < T; ++t) {
        int32_t b = tok_seq[t];
        int64_t nv = csa_oracle_n_vis(comp_off[b + 1] - comp_off[b], tok_pos[t], ratio);
        n_sel[t] = (int32_t)nv;
        for (int32_t i = 0; i < k_all; ++i) idx[(int64_t)t * k_all + i] = i < nv ? i : -1;
    }
    st = csa_oracle_gather(T, hd, k_all, window, ratio, num_seqs, tok_seq, tok_pos, comp_off,
                           idx, n_sel, comp_kv, swa_kv, swa_cap, swa_first_pos, kv_buf, kv_len);
    if (st) goto done;
    st = csa_oracle_attention(T, H, hd, rows_per_token, q, kv_buf, kv_len, scale, sinks, out);
    if (!st && kv_len_out)
        for (int32_t t = 0; t < T; ++t) kv_len_out[t] = kv_len[t];
done:
    free(idx);
    free(n_sel);
    free(kv_len);
    free(kv_buf);
    return st;
}

/* ------------------------------------------------------------------ FP4 keys
 * MXFP4 as read in csa_oracle.h: e2m1 elements, one e8m0 scale per 32. */
static const double kE2m1Magnitude[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double csa_oracle_e2m1_value(uint8_t code) {
    double v = kE2m1Magnitude[code & 7];
    return (code & 8) ? -v : v;
}

/* Nearest e2m1 magnitude code to v >= 0 (v already divided by the block
 * scale); of two equally near grid points the one with the even code wins;
 * beyond the largest magnitude the code saturates. */
static uint8_t e2m1_nearest(double v) {
    if (v >= kE2m1Magnitude[7]) return 7;
    uint8_t best = 0;
    double best_d = fabs(v - kE2m1Magnitude[0]);
    for (uint8_t c = 1; c < 8; ++c) {
        double d = fabs(v - kE2m1Magnitude[c]);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return best;
}

int32_t csa_oracle_fp4_quantize(int64_t R, int32_t ihd, const uint16_t *k, uint8_t *rows) {
    if (R < 0 || ihd != 128 || (R > 0 && (!k || !rows))) return CSA_ORACLE_EINVAL;
    for (int64_t r = 0; r < R; ++r) {
        uint8_t *row = rows + r * CSA_ORACLE_FP4_ROW;
        memset(row, 0, CSA_ORACLE_FP4_ROW);
        for (int b = 0; b < ihd / 32; ++b) {
            const uint16_t *x = k + r * ihd + b * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) {
                double a = fabs(csa_oracle_bf16_to_f64(x[i]));
                if (a > amax) amax = a;
            }
            int E = 0;
            if (amax > 0.0) {
                int ex;
                frexp(amax, &ex);  /* amax = f * 2^ex, f in [0.5, 1): floor(log2) = ex - 1 */
                E = (ex - 1) - 2 + 127;
                if (E < 0) E = 0;
                if (E > 254) E = 254;
            }
            row[64 + b] = (uint8_t)E;
            const double scale = ldexp(1.0, E - 127);
            for (int i = 0; i < 32; ++i) {
                double v = csa_oracle_bf16_to_f64(x[i]);
                uint8_t mag = e2m1_nearest(fabs(v) / scale);
                uint8_t code = mag == 0 ? 0 : (uint8_t)(mag | (v < 0.0 ? 8 : 0));
                int e = b * 32 + i;
                row[e / 2] |= (uint8_t)((e & 1) ? (code << 4) : code);
            }
        }
    }
    return CSA_ORACLE_OK;
}

int32_t csa_oracle_fp4_dequantize(int64_t R, int32_t ihd, const uint8_t *rows, uint16_t *k) {
    if (R < 0 || ihd != 128 || (R > 0 && (!k || !rows))) return CSA_ORACLE_EINVAL;
    for (int64_t r = 0; r < R; ++r) {
        const uint8_t *row = rows + r * CSA_ORACLE_FP4_ROW;
        for (int e = 0; e < ihd; ++e) {
            uint8_t code = (uint8_t)((e & 1) ? (row[e / 2] >> 4) : (row[e / 2] & 15));
            double v = csa_oracle_e2m1_value(code) * ldexp(1.0, (int)row[64 + e / 32] - 127);
            float f = (float)v;
            uint32_t u;
            memcpy(&u, &f, sizeof u);
            if ((double)f != v || (u & 0xFFFFu) != 0) return CSA_ORACLE_EINVAL;
            k[r * ihd + e] = (uint16_t)(u >> 16);
        }
    }
    return CSA_ORACLE_OK;
}
