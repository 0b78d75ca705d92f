// csa_api.cu -- the C ABI of libcsa.so (declared in include/csa.h).
//
// Host side only: argument validation, the workspace plan, tensor-map
// encoding and kernel launches.  Nothing here allocates, frees or
// synchronises; every device buffer belongs to the caller.
#include <cudaTypedefs.h>
#include <math.h>
#include <mutex>

#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

WsPlan make_plan(int64_t T, int64_t max_comp_rows, const csa_params_t &p, int64_t rows_max_in) {
    WsPlan w;
    w.T = T;
    w.top_k = p.top_k;
    w.H = p.n_heads;
    w.ld = ((max_comp_rows > 0 ? max_comp_rows : 1) + 3) / 4 * 4;
    topk_grid(T, max_comp_rows, &w.topk_chunk, &w.topk_per_tok);
    // Attention: a token's row slots (the window starts at a multiple of 4)
    // in chunks of kTcChunk; splits per token so that about one CTA per SM
    // runs, each a whole number of chunks, at most 128 (at HCA's 130 chunks, 65
    // CTAs of two chunks beat 130 of one: 15.9 against 17.9 us; the combine
    // itself takes up to 256).
    const int64_t rows_max =
        rows_max_in >= 0 ? rows_max_in : static_cast<int64_t>(p.top_k) + p.window;
    const int64_t comp_max = rows_max > p.window ? rows_max - p.window : 0;
    const int64_t slots = ((comp_max + 3) & ~int64_t(3)) + p.window;
    const int64_t chunks = (slots + kTcChunk - 1) / kTcChunk;
    const int64_t groups = (p.n_heads + kTcHeads - 1) / kTcHeads;
    int64_t splits = kAttnCtas / ((T > 0 ? T : 1) * groups);
    if (splits > chunks) splits = chunks;
    if (splits > 128) splits = 128;
    if (splits < 1) splits = 1;
    const int64_t per = (chunks + splits - 1) / splits;
    w.rows_split = static_cast<int32_t>(per * kTcChunk);
    w.splits = static_cast<int32_t>((slots + w.rows_split - 1) / w.rows_split);
    // Still few CTAs (one long-context token): 2 or 4 CTAs per split, each
    // computing the split's weights in full and accumulating and writing
    // only its share of the 512 output columns.
    const int64_t ctas = static_cast<int64_t>(w.splits) * (T > 0 ? T : 1) * groups;
    w.dparts = ctas * 4 <= kAttnCtas ? 4 : (ctas * 2 <= kAttnCtas ? 2 : 1);
    const size_t A = 256;
    const size_t Tz = static_cast<size_t>(T > 0 ? T : 0);
    w.state_bytes = Tz * kStateWords * 4;
    size_t off = 0;
    w.off_scores = off;  off = align_up(off + Tz * w.ld * 4, A);
    w.off_slots = off;
    if (w.topk_per_tok > 1) off = align_up(off + Tz * w.topk_per_tok * w.topk_chunk * 8, A);
    w.off_slot_cnt = off; off = align_up(off + Tz * w.topk_per_tok * 4, A);
    w.off_idx = off;     off = align_up(off + Tz * p.top_k * 4, A);
    w.off_nsel = off;    off = align_up(off + Tz * 4, A);
    w.off_part_o = off;
    if (w.splits > 1) off = align_up(off + Tz * w.splits * w.H * kHD * 4, A);
    w.off_part_ml = off;
    if (w.splits > 1) off = align_up(off + Tz * w.splits * w.H * 2 * 4, A);
    // the decode indexer's folded selection: one candidate slot per (token,
    // CTA owning part of it), at most grid + tokens of them (sized for up to
    // kFusedMaxTokens tokens, so the size only grows with T)
    w.fslots = kMaxIdxCtas + static_cast<int32_t>(Tz < size_t(kFusedMaxTokens) ? Tz : kFusedMaxTokens);
    w.fcap = 2 * p.top_k + 96;
    w.off_fcand = off;   off = align_up(off + size_t(w.fslots) * w.fcap * 8, A);
    w.off_fmeta = off;   off = align_up(off + size_t(w.fslots) * 16, A);
    w.off_shard = off;   off = align_up(off + (Tz + 2) * 8, A);
    w.data_bytes = off;
    w.total = w.state_bytes + w.data_bytes + A;
    return w;
}

// Start of the data area: packed against the end of the caller's workspace.
static uint8_t *data_base(void *ws, size_t ws_bytes, const WsPlan &plan) {
    const size_t off = (ws_bytes - plan.data_bytes) & ~static_cast<size_t>(255);
    return static_cast<uint8_t *>(ws) + off;
}

// ---------------------------------------------------------------- driver entry point

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static void resolve_encode() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
}

CUresult encode_tensor_map_2d_bf16(CUtensorMap *map, const void *base, uint64_t inner,
                                   uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                                   uint32_t box_outer) {
    resolve_encode();
    if (!g_encode) return CUDA_ERROR_NOT_SUPPORTED;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_tensor_map_2d_u8(CUtensorMap *map, const void *base, uint64_t inner_bytes,
                                 uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
    resolve_encode();
    if (!g_encode) return CUDA_ERROR_NOT_SUPPORTED;
    cuuint64_t dims[2] = {inner_bytes, outer};
    cuuint64_t strides[1] = {inner_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// ---------------------------------------------------------------- device check

static int g_dev_ok[64];          // 0 unknown, 1 ok, -1 unsupported
static int g_dev_sms[64];
static std::mutex g_dev_mu;

csa_status_t current_device(int *sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CSA_ERR_CUDA;
    if (dev < 0 || dev >= 64) return CSA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_dev_ok[dev] == 0) {
        int major = 0, minor = 0, n = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return CSA_ERR_CUDA;
        // Kernels are built for sm_103a only.
        g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
        g_dev_sms[dev] = n;
    }
    if (g_dev_ok[dev] < 0) return CSA_ERR_UNSUPPORTED;
    *sms = g_dev_sms[dev];
    return CSA_OK;
}

// ---------------------------------------------------------------- validation

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

csa_status_t check_params(const csa_params_t *p) {
    if (!p) return CSA_ERR_INVALID_ARGUMENT;
    if (p->n_ih != kNIH || p->ihd != kIHD || p->hd != kHD) return CSA_ERR_UNSUPPORTED;
    if (p->n_heads < kHeadGroup || p->n_heads > 128 || p->n_heads % kHeadGroup) return CSA_ERR_UNSUPPORTED;
    if (p->top_k < 1) return CSA_ERR_INVALID_ARGUMENT;
    if (p->top_k > kMaxTopK) return CSA_ERR_UNSUPPORTED;
    if (p->window < 1 || p->ratio < 1) return CSA_ERR_INVALID_ARGUMENT;
    if (!isfinite(p->scale)) return CSA_ERR_INVALID_ARGUMENT;
    return CSA_OK;
}

csa_status_t check_layout(const csa_layout_t *L, const csa_params_t *p, bool need_swa) {
    if (!L) return CSA_ERR_INVALID_ARGUMENT;
    if (L->num_seqs < 1 || L->num_tokens < 0) return CSA_ERR_INVALID_ARGUMENT;
    if (L->total_comp_rows < 0 || L->max_comp_rows < 0) return CSA_ERR_INVALID_ARGUMENT;
    if (L->max_comp_rows > L->total_comp_rows) return CSA_ERR_INVALID_ARGUMENT;
    if (L->total_comp_rows >= (int64_t(1) << 31)) return CSA_ERR_UNSUPPORTED;
    if (L->num_tokens > 0 && (!L->tok_seq || !L->tok_pos || !L->comp_off))
        return CSA_ERR_INVALID_ARGUMENT;
    // indexer work units: one token, or 4 tokens of a single sequence
    const int64_t units = (L->num_seqs == 1 && L->num_tokens >= 4) ? (L->num_tokens + 3) / 4
                                                                   : L->num_tokens;
    if (units > 4096) return CSA_ERR_UNSUPPORTED;
    if (need_swa && L->num_tokens > 0) {
        if (!L->swa_kv || !L->swa_first_pos) return CSA_ERR_INVALID_ARGUMENT;
        if (!aligned16(L->swa_kv)) return CSA_ERR_INVALID_ARGUMENT;
        if (L->swa_cap < p->window) return CSA_ERR_CAPACITY;
    }
    return CSA_OK;
}

}  // namespace csa

using namespace csa;

static csa_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

static csa_status_t check_ws(const WsPlan &plan, void *ws, size_t ws_bytes) {
    if (plan.total > 0 && !ws) return CSA_ERR_WORKSPACE;
    if (ws_bytes < plan.total) return CSA_ERR_WORKSPACE;
    if (ws && (reinterpret_cast<uintptr_t>(ws) & 255u)) return CSA_ERR_INVALID_ARGUMENT;
    return CSA_OK;
}

#define CSA_TRY(x)                          \
    do {                                    \
        csa_status_t _s = (x);              \
        if (_s != CSA_OK) return _s;        \
    } while (0)

extern "C" {

const char *csa_status_string(csa_status_t s) {
    switch (s) {
        case CSA_OK: return "CSA_OK";
        case CSA_ERR_INVALID_ARGUMENT: return "CSA_ERR_INVALID_ARGUMENT";
        case CSA_ERR_UNSUPPORTED: return "CSA_ERR_UNSUPPORTED";
        case CSA_ERR_CAPACITY: return "CSA_ERR_CAPACITY";
        case CSA_ERR_CUDA: return "CSA_ERR_CUDA";
        case CSA_ERR_DEVICE_FAULT: return "CSA_ERR_DEVICE_FAULT";
        case CSA_ERR_TIMEOUT: return "CSA_ERR_TIMEOUT";
        case CSA_ERR_WORKSPACE: return "CSA_ERR_WORKSPACE";
    }
    return "CSA_ERR_UNKNOWN";
}

int32_t csa_abi_version(void) { return CSA_ABI_VERSION; }

csa_status_t csa_workspace_size(const csa_layout_t *layout, const csa_params_t *params,
                                size_t *bytes) {
    if (!bytes) return CSA_ERR_INVALID_ARGUMENT;
    CSA_TRY(check_params(params));
    if (!layout) return CSA_ERR_INVALID_ARGUMENT;
    if (layout->num_tokens < 0 || layout->max_comp_rows < 0) return CSA_ERR_INVALID_ARGUMENT;
    *bytes = make_plan(layout->num_tokens, layout->max_comp_rows, *params).total;
    return CSA_OK;
}

// Tokens are scored one per key tile (decode batches): the prefill grouping
// of four tokens of one sequence per tile does not apply.
static bool one_token_per_tile(const csa_layout_t &L) {
    return !(L.num_seqs == 1 && L.num_tokens >= 4);
}

static csa_status_t indexer_scores_impl(const csa_layout_t *layout, const csa_params_t *params,
                                        const void *q_idx, const float *w_idx, const void *k_idx,
                                        float *scores, int64_t ld_scores, int32_t *dev_status,
                                        void *stream, bool fp4) {
    CSA_TRY(check_params(params));
    CSA_TRY(check_layout(layout, params, false));
    if (layout->num_tokens == 0) return CSA_OK;
    if (!q_idx || !w_idx || !scores || !dev_status) return CSA_ERR_INVALID_ARGUMENT;
    if (layout->total_comp_rows > 0 && !k_idx) return CSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q_idx) || (k_idx && !aligned16(k_idx))) return CSA_ERR_INVALID_ARGUMENT;
    if (ld_scores < layout->max_comp_rows || ld_scores < 1) return CSA_ERR_CAPACITY;
    int sms = 0;
    CSA_TRY(current_device(&sms));
    Launch lc{static_cast<cudaStream_t>(stream), sms};
    if (one_token_per_tile(*layout) && decode_indexer_fits(*layout, sms, false))
        return cuda_status(launch_decode_indexer(lc, *layout, *params, q_idx, w_idx, k_idx, scores,
                                                 ld_scores, dev_status, nullptr, fp4));
    return cuda_status(launch_indexer(lc, *layout, *params, q_idx, w_idx, k_idx, scores,
                                      ld_scores, nullptr, dev_status, fp4));
}

csa_status_t csa_indexer_scores(const csa_layout_t *layout, const csa_params_t *params,
                                const void *q_idx, const float *w_idx, const void *k_idx,
                                float *scores, int64_t ld_scores, int32_t *dev_status,
                                void *stream) {
    return indexer_scores_impl(layout, params, q_idx, w_idx, k_idx, scores, ld_scores,
                               dev_status, stream, false);
}

csa_status_t csa_indexer_scores_fp4(const csa_layout_t *layout, const csa_params_t *params,
                                    const void *q_idx, const float *w_idx, const void *k_fp4,
                                    float *scores, int64_t ld_scores, int32_t *dev_status,
                                    void *stream) {
    return indexer_scores_impl(layout, params, q_idx, w_idx, k_fp4, scores, ld_scores,
                               dev_status, stream, true);
}

csa_status_t csa_fp4_quantize_keys(int64_t rows, const void *k_idx, void *k_fp4, void *stream) {
    if (rows < 0) return CSA_ERR_INVALID_ARGUMENT;
    if (rows == 0) return CSA_OK;
    if (!k_idx || !k_fp4 || !aligned16(k_idx) || !aligned16(k_fp4)) return CSA_ERR_INVALID_ARGUMENT;
    int sms = 0;
    CSA_TRY(current_device(&sms));
    Launch lc{static_cast<cudaStream_t>(stream), sms};
    return cuda_status(launch_fp4_quantize(lc, rows, k_idx, k_fp4));
}

csa_status_t csa_topk(const csa_layout_t *layout, const csa_params_t *params, const float *scores,
                      int64_t ld_scores, int32_t *idx, int32_t *n_sel, int32_t *dev_status,
                      void *ws, size_t ws_bytes, void *stream) {
    CSA_TRY(check_params(params));
    CSA_TRY(check_layout(layout, params, false));
    if (layout->num_tokens == 0) return CSA_OK;
    if (!scores || !idx || !n_sel || !dev_status) return CSA_ERR_INVALID_ARGUMENT;
    if (ld_scores < layout->max_comp_rows || ld_scores < 1) return CSA_ERR_CAPACITY;
    const WsPlan plan = make_plan(layout->num_tokens, layout->max_comp_rows, *params);
    CSA_TRY(check_ws(plan, ws, ws_bytes));
    int sms = 0;
    CSA_TRY(current_device(&sms));
    Launch lc{static_cast<cudaStream_t>(stream), sms};
    uint8_t *w = data_base(ws, ws_bytes, plan);
    TopkWs tw{static_cast<uint32_t *>(ws), reinterpret_cast<uint64_t *>(w + plan.off_slots),
              reinterpret_cast<uint32_t *>(w + plan.off_slot_cnt)};
    return cuda_status(launch_topk(lc, *layout, *params, scores, ld_scores, tw, false, idx, n_sel,
                                   dev_status));
}

csa_status_t csa_gather_mixed(const csa_layout_t *layout, const csa_params_t *params,
                              const int32_t *idx, const int32_t *n_sel, const void *comp_kv,
                              void *kv_buf, int32_t *kv_len, int32_t *dev_status, void *stream) {
    CSA_TRY(check_params(params));
    CSA_TRY(check_layout(layout, params, true));
    if (layout->num_tokens == 0) return CSA_OK;
    if (!idx || !n_sel || !kv_buf || !kv_len || !dev_status) return CSA_ERR_INVALID_ARGUMENT;
    if (layout->total_comp_rows > 0 && !comp_kv) return CSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(kv_buf) || (comp_kv && !aligned16(comp_kv))) return CSA_ERR_INVALID_ARGUMENT;
    int sms = 0;
    CSA_TRY(current_device(&sms));
    Launch lc{static_cast<cudaStream_t>(stream), sms};
    RowSource R{};
    R.fused = kRowsSelected;
    R.rows_per_token = params->top_k + params->window;
    R.L = *layout;
    R.ratio = params->ratio;
    R.window = params->window;
    R.top_k = params->top_k;
    R.idx = idx;
    R.n_sel = n_sel;
    R.comp_kv = comp_kv;
    return cuda_status(launch_gather(lc, R, layout->num_tokens, kv_buf, kv_len, dev_status));
}

csa_status_t csa_sparse_mqa_decode(int32_t num_tokens, const csa_params_t *params, const void *q,
                                   const void *kv_buf, const int32_t *kv_len, const float *sinks,
                                   float *out, int32_t *dev_status, void *ws, size_t ws_bytes,
                                   void *stream) {
    CSA_TRY(check_params(params));
    if (num_tokens < 0) return CSA_ERR_INVALID_ARGUMENT;
    if (num_tokens == 0) return CSA_OK;
    if (!q || !kv_buf || !kv_len || !out || !dev_status) return CSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(kv_buf) || !aligned16(out)) return CSA_ERR_INVALID_ARGUMENT;
    const WsPlan plan = make_plan(num_tokens, 0, *params);
    CSA_TRY(check_ws(plan, ws, ws_bytes));
    int sms = 0;
    CSA_TRY(current_device(&sms));
    Launch lc{static_cast<cudaStream_t>(stream), sms};
    RowSource R{};
    R.fused = kRowsGathered;
    R.kv_buf = kv_buf;
    R.kv_len = kv_len;
    R.rows_per_token = params->top_k + params->window;
    uint8_t *w = data_base(ws, ws_bytes, plan);
    return cuda_status(launch_attention_tc(lc, R, num_tokens, *params, plan, q, sinks, out,
                                        reinterpret_cast<float *>(w + plan.off_part_o),
                                        reinterpret_cast<float *>(w + plan.off_part_ml),
                                        dev_status));
}

// Steps 1 and 2: the selection of every token into idx / nsel.  Decode
// batches go through the decode indexer with the selection folded in; other
// layouts (prefill chunks, FP4 keys, very large batches) through the indexer
// and the separate top-k.
static cudaError_t select_blocks(const Launch &lc, const csa_layout_t &L, const csa_params_t &p,
                                 const WsPlan &plan, uint8_t *w, uint32_t *state,
                                 const void *q_idx, const float *w_idx, const void *k_idx,
                                 int32_t *idx, int32_t *nsel, int32_t *dev_status, bool fp4) {
    float *scores = reinterpret_cast<float *>(w + plan.off_scores);
    if (one_token_per_tile(L) && decode_indexer_fits(L, lc.sm_count, true)) {
        FusedTopk f;
        f.state = state;
        f.cand = reinterpret_cast<uint64_t *>(w + plan.off_fcand);
        f.meta = reinterpret_cast<uint4 *>(w + plan.off_fmeta);
        f.slots = plan.fslots;
        f.cap = plan.fcap;
        f.idx = idx;
        f.n_sel = nsel;
        return launch_decode_indexer(lc, L, p, q_idx, w_idx, k_idx, scores, plan.ld, dev_status, &f,
                                     fp4);
    }
    const bool fuse = indexer_fuses_hist(L);
    cudaError_t e = launch_indexer(lc, L, p, q_idx, w_idx, k_idx, scores, plan.ld,
                                   fuse ? state : nullptr, dev_status, fp4);
    if (e != cudaSuccess) return e;
    TopkWs tw{state, reinterpret_cast<uint64_t *>(w + plan.off_slots),
              reinterpret_cast<uint32_t *>(w + plan.off_slot_cnt)};
    return launch_topk(lc, L, p, scores, plan.ld, tw, fuse, idx, nsel, dev_status);
}

csa_status_t csa_indexer_topk(const csa_layout_t *layout, const csa_params_t *params,
                              const void *q_idx, const float *w_idx, const void *k_idx,
                              int32_t *idx, int32_t *n_sel, int32_t *dev_status, void *ws,
                              size_t ws_bytes, void *stream) {
    CSA_TRY(check_params(params));
    CSA_TRY(check_layout(layout, params, false));
    if (layout->num_tokens == 0) return CSA_OK;
    if (!q_idx || !w_idx || !idx || !n_sel || !dev_status) return CSA_ERR_INVALID_ARGUMENT;
    if (layout->total_comp_rows > 0 && !k_idx) return CSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q_idx) || (k_idx && !aligned16(k_idx))) return CSA_ERR_INVALID_ARGUMENT;
    const WsPlan plan = make_plan(layout->num_tokens, layout->max_comp_rows, *params);
    CSA_TRY(check_ws(plan, ws, ws_bytes));
    int sms = 0;
    CSA_TRY(current_device(&sms));
    Launch lc{static_cast<cudaStream_t>(stream), sms};
    uint8_t *w = data_base(ws, ws_bytes, plan);
    return cuda_status(select_blocks(lc, *layout, *params, plan, w, static_cast<uint32_t *>(ws),
                                     q_idx, w_idx, k_idx, idx, n_sel, dev_status, false));
}

static csa_status_t decode_impl(const csa_layout_t *layout, const csa_params_t *params,
                                const void *q_idx, const float *w_idx, const void *k_idx,
                                const void *comp_kv, const void *q, const float *sinks, float *out,
                                int32_t *idx_out, int32_t *dev_status, void *ws, size_t ws_bytes,
                                void *stream, bool fp4) {
    CSA_TRY(check_params(params));
    CSA_TRY(check_layout(layout, params, true));
    if (layout->num_tokens == 0) return CSA_OK;
    if (!q_idx || !w_idx || !q || !out || !dev_status) return CSA_ERR_INVALID_ARGUMENT;
    if (layout->total_comp_rows > 0 && (!k_idx || !comp_kv)) return CSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q_idx) || !aligned16(q) || !aligned16(out) ||
        (k_idx && !aligned16(k_idx)) || (comp_kv && !aligned16(comp_kv)))
        return CSA_ERR_INVALID_ARGUMENT;
    const WsPlan plan = make_plan(layout->num_tokens, layout->max_comp_rows, *params);
    CSA_TRY(check_ws(plan, ws, ws_bytes));
    int sms = 0;
    CSA_TRY(current_device(&sms));
    Launch lc{static_cast<cudaStream_t>(stream), sms};
    uint8_t *w = data_base(ws, ws_bytes, plan);
    uint32_t *state = static_cast<uint32_t *>(ws);
    int32_t *idx = idx_out ? idx_out : reinterpret_cast<int32_t *>(w + plan.off_idx);
    int32_t *nsel = reinterpret_cast<int32_t *>(w + plan.off_nsel);
    cudaError_t e = select_blocks(lc, *layout, *params, plan, w, state, q_idx, w_idx, k_idx, idx,
                                  nsel, dev_status, fp4);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
    RowSource R{};
    R.fused = kRowsSelected;
    R.rows_per_token = params->top_k + params->window;
    R.L = *layout;
    R.ratio = params->ratio;
    R.window = params->window;
    R.top_k = params->top_k;
    R.idx = idx;
    R.n_sel = nsel;
    R.comp_kv = comp_kv;
    return cuda_status(launch_attention_tc(lc, R, layout->num_tokens, *params, plan, q, sinks, out,
                                        reinterpret_cast<float *>(w + plan.off_part_o),
                                        reinterpret_cast<float *>(w + plan.off_part_ml),
                                        dev_status, true));
}

csa_status_t csa_decode(const csa_layout_t *layout, const csa_params_t *params, const void *q_idx,
                        const float *w_idx, const void *k_idx, const void *comp_kv, const void *q,
                        const float *sinks, float *out, int32_t *idx_out, int32_t *dev_status,
                        void *ws, size_t ws_bytes, void *stream) {
    return decode_impl(layout, params, q_idx, w_idx, k_idx, comp_kv, q, sinks, out, idx_out,
                       dev_status, ws, ws_bytes, stream, false);
}

csa_status_t csa_decode_fp4(const csa_layout_t *layout, const csa_params_t *params,
                            const void *q_idx, const float *w_idx, const void *k_fp4,
                            const void *comp_kv, const void *q, const float *sinks, float *out,
                            int32_t *idx_out, int32_t *dev_status, void *ws, size_t ws_bytes,
                            void *stream) {
    return decode_impl(layout, params, q_idx, w_idx, k_fp4, comp_kv, q, sinks, out, idx_out,
                       dev_status, ws, ws_bytes, stream, true);
}

static int64_t hca_rows_max(const csa_layout_t *L, const csa_params_t *p) {
    return (L->max_comp_rows > 0 ? L->max_comp_rows : 0) + p->window;
}

csa_status_t csa_hca_workspace_size(const csa_layout_t *layout, const csa_params_t *params,
                                    size_t *bytes) {
    if (!bytes || !layout) return CSA_ERR_INVALID_ARGUMENT;
    CSA_TRY(check_params(params));
    if (layout->num_tokens < 0 || layout->max_comp_rows < 0) return CSA_ERR_INVALID_ARGUMENT;
    *bytes = make_plan(layout->num_tokens, 0, *params, hca_rows_max(layout, params)).total;
    return CSA_OK;
}

csa_status_t csa_hca_decode(const csa_layout_t *layout, const csa_params_t *params,
                            const void *comp_kv, const void *q, const float *sinks, float *out,
                            int32_t *dev_status, void *ws, size_t ws_bytes, void *stream) {
    CSA_TRY(check_params(params));
    CSA_TRY(check_layout(layout, params, true));
    if (layout->num_tokens == 0) return CSA_OK;
    if (!q || !out || !dev_status) return CSA_ERR_INVALID_ARGUMENT;
    if (layout->total_comp_rows > 0 && !comp_kv) return CSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(out) || (comp_kv && !aligned16(comp_kv)))
        return CSA_ERR_INVALID_ARGUMENT;
    const WsPlan plan = make_plan(layout->num_tokens, 0, *params, hca_rows_max(layout, params));
    CSA_TRY(check_ws(plan, ws, ws_bytes));
    int sms = 0;
    CSA_TRY(current_device(&sms));
    Launch lc{static_cast<cudaStream_t>(stream), sms};
    uint8_t *w = data_base(ws, ws_bytes, plan);
    RowSource R{};
    R.fused = kRowsAllVisible;
    R.rows_per_token = static_cast<int32_t>(hca_rows_max(layout, params));
    R.L = *layout;
    R.ratio = params->ratio;
    R.window = params->window;
    R.top_k = params->top_k;
    R.comp_kv = comp_kv;
    return cuda_status(launch_attention_tc(lc, R, layout->num_tokens, *params, plan, q, sinks, out,
                                        reinterpret_cast<float *>(w + plan.off_part_o),
                                        reinterpret_cast<float *>(w + plan.off_part_ml),
                                        dev_status));
}

// ---------------------------------------------------------------- sharded decode

// A shard's range of one sequence's blocks: [lo, hi), the shard's caches
// holding hi - lo rows.
static csa_status_t check_shard(const csa_layout_t *layout, int64_t lo, int64_t hi) {
    if (layout->num_seqs != 1) return CSA_ERR_UNSUPPORTED;
    if (lo < 0 || hi < lo || hi > (int64_t(1) << 31) - 1) return CSA_ERR_INVALID_ARGUMENT;
    return CSA_OK;
}

// The shard's layout in the workspace (device arrays written by a kernel).
static csa_layout_t shard_layout(const Launch &lc, const csa_layout_t &L, const csa_params_t &p,
                                 const WsPlan &plan, uint8_t *w, int64_t lo, int64_t hi,
                                 int32_t *status, cudaError_t *err) {
    int64_t *pos = reinterpret_cast<int64_t *>(w + plan.off_shard);
    int64_t *off = pos + (plan.T > 0 ? plan.T : 0);
    *err = launch_shard_layout(lc, L, p.ratio, lo, hi, pos, off, status);
    csa_layout_t S = L;
    S.tok_pos = pos;
    S.comp_off = off;
    S.num_seqs = 1;
    S.total_comp_rows = hi - lo;
    S.max_comp_rows = hi - lo;
    return S;
}

csa_status_t csa_shard_workspace_size(const csa_layout_t *layout, const csa_params_t *params,
                                      int64_t shard_lo, int64_t shard_hi, size_t *bytes) {
    if (!bytes || !layout) return CSA_ERR_INVALID_ARGUMENT;
    CSA_TRY(check_params(params));
    if (layout->num_tokens < 0) return CSA_ERR_INVALID_ARGUMENT;
    CSA_TRY(check_shard(layout, shard_lo, shard_hi));
    const size_t a = make_plan(layout->num_tokens, shard_hi - shard_lo, *params).total;
    const size_t b = make_plan(layout->num_tokens, 0, *params).total;   // the window's partial
    *bytes = a > b ? a : b;
    return CSA_OK;
}

csa_status_t csa_shard_candidates(const csa_layout_t *layout, const csa_params_t *params,
                                  int64_t shard_lo, int64_t shard_hi, const void *q_idx,
                                  const float *w_idx, const void *k_idx_shard, float *cand_score,
                                  int32_t *cand_idx, int32_t *n_cand, int32_t *dev_status, void *ws,
                                  size_t ws_bytes, void *stream) {
    CSA_TRY(check_params(params));
    CSA_TRY(check_layout(layout, params, false));
    CSA_TRY(check_shard(layout, shard_lo, shard_hi));
    if (layout->num_tokens == 0) return CSA_OK;
    if (!q_idx || !w_idx || !cand_score || !cand_idx || !n_cand || !dev_status)
        return CSA_ERR_INVALID_ARGUMENT;
    if (shard_hi > shard_lo && !k_idx_shard) return CSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q_idx) || (k_idx_shard && !aligned16(k_idx_shard))) return CSA_ERR_INVALID_ARGUMENT;
    const int64_t nb = shard_hi - shard_lo;
    const WsPlan plan = make_plan(layout->num_tokens, nb, *params);
    CSA_TRY(check_ws(plan, ws, ws_bytes));
    int sms = 0;
    CSA_TRY(current_device(&sms));
    Launch lc{static_cast<cudaStream_t>(stream), sms};
    uint8_t *w = data_base(ws, ws_bytes, plan);
    cudaError_t e = cudaSuccess;
    if (nb == 0)   // a shard without blocks has no candidates
        return cuda_status(launch_shard_candidates(lc, layout->num_tokens, params->top_k,
                                                   shard_lo, nullptr, 0, nullptr, nullptr,
                                                   cand_score, cand_idx, n_cand));
    const csa_layout_t S = shard_layout(lc, *layout, *params, plan, w, shard_lo, shard_hi,
                                        dev_status, &e);
    if (e != cudaSuccess) return cuda_status(e);
    // every visible block's score (the candidates carry them), then the local top-k
    float *scores = reinterpret_cast<float *>(w + plan.off_scores);
    if (one_token_per_tile(S) && decode_indexer_fits(S, sms, false))
        e = launch_decode_indexer(lc, S, *params, q_idx, w_idx, k_idx_shard, scores, plan.ld,
                                  dev_status, nullptr);
    else
        e = launch_indexer(lc, S, *params, q_idx, w_idx, k_idx_shard, scores, plan.ld, nullptr,
                           dev_status, false);
    if (e != cudaSuccess) return cuda_status(e);
    int32_t *idx = reinterpret_cast<int32_t *>(w + plan.off_idx);
    int32_t *nsel = reinterpret_cast<int32_t *>(w + plan.off_nsel);
    TopkWs tw{static_cast<uint32_t *>(ws), reinterpret_cast<uint64_t *>(w + plan.off_slots),
              reinterpret_cast<uint32_t *>(w + plan.off_slot_cnt)};
    e = launch_topk(lc, S, *params, scores, plan.ld, tw, false, idx, nsel, dev_status);
    if (e != cudaSuccess) return cuda_status(e);
    return cuda_status(launch_shard_candidates(lc, layout->num_tokens, params->top_k, shard_lo,
                                               scores, plan.ld, idx, nsel, cand_score, cand_idx,
                                               n_cand));
}

csa_status_t csa_shard_merge(int32_t num_tokens, int32_t top_k, int32_t num_shards,
                             const int64_t *shard_bounds, const float *cand_score,
                             const int32_t *cand_idx, const int32_t *n_cand, int32_t *idx,
                             int32_t *n_sel, int32_t *shard_idx, int32_t *shard_nsel,
                             int32_t *dev_status, void *stream) {
    if (num_tokens < 0 || top_k < 1 || num_shards < 1 || !shard_bounds) return CSA_ERR_INVALID_ARGUMENT;
    if (num_shards > kMaxShards || top_k > 2048) return CSA_ERR_UNSUPPORTED;
    for (int g = 0; g < num_shards; ++g)
        if (shard_bounds[g] < 0 || shard_bounds[g + 1] < shard_bounds[g]) return CSA_ERR_INVALID_ARGUMENT;
    if (shard_bounds[num_shards] > (int64_t(1) << 31) - 1) return CSA_ERR_INVALID_ARGUMENT;
    if (num_tokens == 0) return CSA_OK;
    if (!cand_score || !cand_idx || !n_cand || !idx || !n_sel || !shard_idx || !shard_nsel ||
        !dev_status)
        return CSA_ERR_INVALID_ARGUMENT;
    int sms = 0;
    CSA_TRY(current_device(&sms));
    Launch lc{static_cast<cudaStream_t>(stream), sms};
    ShardMergeArgs A{};
    A.T = num_tokens;
    A.top_k = top_k;
    A.G = num_shards;
    for (int g = 0; g <= num_shards; ++g) A.bounds[g] = shard_bounds[g];
    A.cand_score = cand_score;
    A.cand_idx = cand_idx;
    A.n_cand = n_cand;
    A.idx = idx;
    A.n_sel = n_sel;
    A.shard_idx = shard_idx;
    A.shard_nsel = shard_nsel;
    A.status = dev_status;
    return cuda_status(launch_shard_merge(lc, A));
}

csa_status_t csa_shard_attention(const csa_layout_t *layout, const csa_params_t *params,
                                 int64_t shard_lo, int64_t shard_hi, const int32_t *shard_idx,
                                 const int32_t *shard_nsel, const void *comp_kv_shard,
                                 const void *q, float *part_o, float *part_ml, int32_t *dev_status,
                                 void *ws, size_t ws_bytes, void *stream) {
    CSA_TRY(check_params(params));
    CSA_TRY(check_layout(layout, params, false));
    CSA_TRY(check_shard(layout, shard_lo, shard_hi));
    if (layout->num_tokens == 0) return CSA_OK;
    if (!shard_idx || !shard_nsel || !q || !part_o || !part_ml || !dev_status)
        return CSA_ERR_INVALID_ARGUMENT;
    if (shard_hi > shard_lo && !comp_kv_shard) return CSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(part_o) || (comp_kv_shard && !aligned16(comp_kv_shard)))
        return CSA_ERR_INVALID_ARGUMENT;
    const int64_t nb = shard_hi - shard_lo;
    const WsPlan plan = make_plan(layout->num_tokens, nb, *params);
    CSA_TRY(check_ws(plan, ws, ws_bytes));
    int sms = 0;
    CSA_TRY(current_device(&sms));
    Launch lc{static_cast<cudaStream_t>(stream), sms};
    uint8_t *w = data_base(ws, ws_bytes, plan);
    cudaError_t e = cudaSuccess;
    const csa_layout_t S = shard_layout(lc, *layout, *params, plan, w, shard_lo, shard_hi,
                                        dev_status, &e);
    if (e != cudaSuccess) return cuda_status(e);
    RowSource R{};
    R.fused = kRowsSelected;
    R.rows_per_token = params->top_k;
    R.L = S;
    R.ratio = params->ratio;
    R.window = params->window;
    R.top_k = params->top_k;
    R.idx = shard_idx;
    R.n_sel = shard_nsel;
    R.comp_kv = comp_kv_shard;
    R.no_window = 1;
    return cuda_status(launch_attention_tc(lc, R, layout->num_tokens, *params, plan, q, nullptr,
                                           part_o, reinterpret_cast<float *>(w + plan.off_part_o),
                                           reinterpret_cast<float *>(w + plan.off_part_ml),
                                           dev_status, false, part_ml));
}

csa_status_t csa_window_attention(const csa_layout_t *layout, const csa_params_t *params,
                                  const void *q, float *part_o, float *part_ml,
                                  int32_t *dev_status, void *ws, size_t ws_bytes, void *stream) {
    CSA_TRY(check_params(params));
    CSA_TRY(check_layout(layout, params, true));
    if (layout->num_seqs != 1) return CSA_ERR_UNSUPPORTED;
    if (layout->num_tokens == 0) return CSA_OK;
    if (!q || !part_o || !part_ml || !dev_status) return CSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(part_o)) return CSA_ERR_INVALID_ARGUMENT;
    const WsPlan plan = make_plan(layout->num_tokens, 0, *params, params->window);
    CSA_TRY(check_ws(plan, ws, ws_bytes));
    int sms = 0;
    CSA_TRY(current_device(&sms));
    Launch lc{static_cast<cudaStream_t>(stream), sms};
    uint8_t *w = data_base(ws, ws_bytes, plan);
    RowSource R{};
    R.fused = kRowsSelected;
    R.rows_per_token = params->window;
    R.L = *layout;
    R.ratio = params->ratio;
    R.window = params->window;
    R.top_k = params->top_k;
    R.no_selected = 1;
    return cuda_status(launch_attention_tc(lc, R, layout->num_tokens, *params, plan, q, nullptr,
                                           part_o, reinterpret_cast<float *>(w + plan.off_part_o),
                                           reinterpret_cast<float *>(w + plan.off_part_ml),
                                           dev_status, false, part_ml));
}

csa_status_t csa_shard_combine(int32_t num_parts, int32_t num_tokens, int32_t n_heads,
                               const float *part_o, const float *part_ml, const float *sinks,
                               float *out, int32_t *dev_status, void *stream) {
    if (num_parts < 1 || num_tokens < 0 || n_heads < 1) return CSA_ERR_INVALID_ARGUMENT;
    if (num_parts > 256 || n_heads > 128) return CSA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return CSA_OK;
    if (!part_o || !part_ml || !out || !dev_status) return CSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(part_o) || !aligned16(out)) return CSA_ERR_INVALID_ARGUMENT;
    int sms = 0;
    CSA_TRY(current_device(&sms));
    Launch lc{static_cast<cudaStream_t>(stream), sms};
    return cuda_status(launch_partials_combine(lc, num_parts, num_tokens, n_heads, part_o, part_ml,
                                               sinks, out, dev_status));
}

}  // extern "C"
