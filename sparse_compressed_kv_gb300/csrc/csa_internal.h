// csa_internal.h -- host-side plumbing shared by the library's translation
// units: workspace plan, launch context and the per-kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "csa.h"

namespace csa {

// Device-independent grid targets (sized for ~150-SM parts).
constexpr int kTargetCtas = 296;
constexpr int kTcChunk = 64;     // rows per chunk of the tensor-core attention
constexpr int kTcHeads = 64;     // heads per tensor-core attention CTA
constexpr int kAttnCtas = 148;   // attention CTAs to aim for (about one per SM)
constexpr int kHeadGroup = 16;   // n_heads must be a multiple of this
constexpr int kMaxFilterChunk = 4096;  // scores per top-k filter CTA (multi-CTA mode)
constexpr int kMaxPerTok = 512;        // top-k filter CTAs per token

// Decode indexer (one query token per key tile), with or without the top-k
// folded in (csa_indexer_topk.cu).  Key ranges are cut in units of kBoxRows
// keys (the TMA box height), so CTAs get equal shares to within one unit.
constexpr int kBoxRows = 32;
constexpr int kMaxIdxCtas = 192;       // grid cap of the decode indexer
constexpr int kDecMaxTokens = 1024;    // tokens the decode indexer takes
constexpr int kFusedMaxTokens = 512;   // tokens the fused selection takes
constexpr int kSegKeysMax = 8192;      // keys one CTA keeps on chip for its local selection

struct WsPlan {
    int64_t T = 0;
    int64_t ld = 0;          // row stride of the workspace score matrix
    int32_t top_k = 0;
    int32_t H = 0;
    int32_t topk_chunk = 0;  // scores per top-k filter CTA
    int32_t topk_per_tok = 1;  // top-k filter CTAs per token (1: one CTA owns the row)
    int32_t splits = 1;      // attention splits per token
    int32_t rows_split = 0;  // rows per attention split (multiple of kTcChunk)
    int32_t dparts = 1;      // attention CTAs per split and head group (1, 2 or 4), one column range each
    // Layout: [per-token state | ... free ... | data].  The state slots sit at
    // the front at offsets that depend only on the token index; the data
    // regions are packed against the end of the caller's workspace, so no
    // call's data ever lands on a state slot of a call with more tokens.
    size_t state_bytes = 0;
    size_t off_scores = 0, off_slots = 0, off_slot_cnt = 0;   // offsets inside the data area
    size_t off_idx = 0, off_nsel = 0, off_part_o = 0, off_part_ml = 0;
    size_t off_fcand = 0, off_fmeta = 0;  // fused selection: candidate slots and their headers
    size_t off_shard = 0;                 // a shard's layout: token positions [T], offsets [2]
    int32_t fslots = 0;                   // candidate slots (grid cap + tokens)
    int32_t fcap = 0;                     // entries per candidate slot
    size_t data_bytes = 0;
    size_t total = 0;        // state + data + alignment slack
};

// Host-side argument checks shared by the entry points (csa_api.cu).  Each
// returns CSA_OK or the csa_status_t the entry point reports.
csa_status_t check_params(const csa_params_t *p);
csa_status_t check_layout(const csa_layout_t *L, const csa_params_t *p, bool need_swa);
// The current device is an sm_103 part; *sms = its SM count (cached per device).
csa_status_t current_device(int *sms);

// rows_max: most rows any token attends (top_k + window for CSA; for HCA,
// every visible block + window); < 0 means top_k + window.
WsPlan make_plan(int64_t T, int64_t max_comp_rows, const csa_params_t &p, int64_t rows_max = -1);

struct Launch {
    cudaStream_t stream;
    int sm_count;
};

// Top-k workspace pieces (device pointers).  With slots == nullptr the top-k
// runs one CTA per token and needs only the state.
struct TopkWs {
    uint32_t *state;     // [T][kStateWords]: histogram + counters, zero on entry and exit
    uint64_t *slots;     // [T][per_tok][chunk] filter output (multi-CTA mode)
    uint32_t *slot_cnt;  // [T][per_tok]
};

// Shape of the top-k filter grid for T tokens of at most max_comp_rows blocks.
void topk_grid(int64_t T, int64_t max_comp_rows, int32_t *chunk, int32_t *per_tok);

// Fused selection of the decode indexer: where its candidates go and where
// the selection lands (device pointers).
struct FusedTopk {
    uint32_t *state;       // [T][kStateWords] per-token state (its ticket word is used)
    uint64_t *cand;        // [slots][cap] (key << 32 | block) candidates, ascending block
    uint4 *meta;           // [slots] count, bound, overflow, length
    int32_t slots, cap;
    int32_t *idx;          // [T][top_k]
    int32_t *n_sel;        // [T]
};

// The decode indexer (bf16 keys, one token per key tile) takes this layout:
// at most kDecMaxTokens tokens; with the fused selection, at most
// kFusedMaxTokens and at most kSegKeysMax keys per CTA.
bool decode_indexer_fits(const csa_layout_t &L, int sm_count, bool fused);

// Scores of every visible block (fused == nullptr), or the top-k selection
// as well (scores then go to the workspace, for the exact fallback).
cudaError_t launch_decode_indexer(const Launch &lc, const csa_layout_t &L, const csa_params_t &p,
                                  const void *q_idx, const float *w_idx, const void *k_idx,
                                  float *scores, int64_t ld, int32_t *status,
                                  const FusedTopk *fused, bool fp4 = false);

// Where attention rows come from.
enum RowMode { kRowsGathered = 0, kRowsSelected = 1, kRowsAllVisible = 2 };

struct RowSource {
    int fused;                     // RowMode: gathered buffer / selected indices / every
                                   // visible block (HCA), the last two plus the window ring
    const void *kv_buf;            // gathered: bf16 [T][rows_per_token][hd]
    const int32_t *kv_len;         // gathered: [T]
    int32_t rows_per_token;        // top_k + window
    csa_layout_t L;                // fused
    int32_t ratio, window, top_k;  // fused
    const int32_t *idx;            // fused: [T][top_k]
    const int32_t *n_sel;          // fused: [T]
    const void *comp_kv;           // fused: bf16 [R][hd]
    int32_t no_window;             // selected rows only (a shard's partial)
    int32_t no_selected;           // window rows only (the window's partial)
};

// Sharded single-sequence decode (csa_shard.cu).
constexpr int kMaxShards = 8;

struct ShardMergeArgs {
    int32_t T, top_k, G;
    int32_t npad, kpad;                    // set by the launcher
    int64_t bounds[kMaxShards + 1];        // shard g holds blocks [bounds[g], bounds[g+1])
    const float *cand_score;               // [G][T][top_k]
    const int32_t *cand_idx;               // [G][T][top_k] global block indices
    const int32_t *n_cand;                 // [G][T]
    int32_t *idx;                          // [T][top_k] global, ascending
    int32_t *n_sel;                        // [T]
    int32_t *shard_idx;                    // [G][T][top_k] shard rows, ascending
    int32_t *shard_nsel;                   // [G][T]
    int32_t *status;
};

cudaError_t launch_shard_layout(const Launch &lc, const csa_layout_t &L, int32_t ratio,
                                int64_t lo, int64_t hi, int64_t *tok_pos_out,
                                int64_t *comp_off_out, int32_t *status);
cudaError_t launch_shard_candidates(const Launch &lc, int32_t T, int32_t top_k, int64_t lo,
                                    const float *scores, int64_t ld, const int32_t *idx,
                                    const int32_t *n_sel, float *cand_score, int32_t *cand_idx,
                                    int32_t *n_cand);
size_t shard_merge_smem(int G, int top_k);
cudaError_t launch_shard_merge(const Launch &lc, ShardMergeArgs A);

// k_idx: bf16 [R, 128] keys, or, with fp4, MXFP4 rows [R, 80] (csa.h).
cudaError_t launch_indexer(const Launch &lc, const csa_layout_t &L, const csa_params_t &p,
                           const void *q_idx, const float *w_idx, const void *k_idx,
                           float *scores, int64_t ld, uint32_t *state, int32_t *status,
                           bool fp4 = false);

// bf16 keys [R, 128] -> MXFP4 rows [R, 80].
cudaError_t launch_fp4_quantize(const Launch &lc, int64_t rows, const void *k_idx, void *k_fp4);

// True when csa_decode's indexer can fold the pass-1 histogram of the top-k
// into its epilogue (one token per indexer unit).
bool indexer_fuses_hist(const csa_layout_t &L);

cudaError_t launch_topk(const Launch &lc, const csa_layout_t &L, const csa_params_t &p,
                        const float *scores, int64_t ld, const TopkWs &ws, bool hist_ready,
                        int32_t *idx, int32_t *n_sel, int32_t *status);

cudaError_t launch_gather(const Launch &lc, const RowSource &src, int32_t T, void *kv_buf,
                          int32_t *kv_len, int32_t *status);

// Shared-KV attention on the tensor cores (csa_attention_tc.cu): grid
// (splits, ceil(H / 64), T), partials merged by a combine kernel when a
// token has several splits.  With raw_ml set the result is the unnormalised
// partial instead (out: O [T][H][512] scaled to the running maximum m,
// raw_ml: (m in log2 units, l) [T][H][2]; no sink).
cudaError_t launch_attention_tc(const Launch &lc, const RowSource &src, int32_t T,
                                const csa_params_t &p, const WsPlan &plan, const void *q,
                                const float *sinks, float *out, float *part_o, float *part_ml,
                                int32_t *status, bool early_q = false, float *raw_ml = nullptr);

// Log-sum-exp merge of P partials laid out [P][T][H][512] and [P][T][H][2]
// into out [T][H][512] (with the sinks, if given, in the denominator).
cudaError_t launch_partials_combine(const Launch &lc, int32_t P, int32_t T, int32_t H,
                                    const float *part_o, const float *part_ml, const float *sinks,
                                    float *out, int32_t *status);

// Launch helper: programmatic dependent launch on, so each kernel's prologue
// may overlap the previous kernel's tail (kernels wait with griddepcontrol).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Dynamic shared memory limit, and the largest shared-memory carveout for
// every kernel of the library: all kernels then run under one L1/shared
// split, so an SM never has to drain and reconfigure between them.
template <typename K>
cudaError_t set_kernel_smem(K kernel, size_t dyn_bytes) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         static_cast<int>(cudaSharedmemCarveoutMaxShared));
    if (e != cudaSuccess) return e;
    if (dyn_bytes > 48 * 1024)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(dyn_bytes));
    return e;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
CUresult encode_tensor_map_2d_bf16(CUtensorMap *map, const void *base, uint64_t inner,
                                   uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                                   uint32_t box_outer);
// Dense byte rows of inner_bytes each, no swizzle.
CUresult encode_tensor_map_2d_u8(CUtensorMap *map, const void *base, uint64_t inner_bytes,
                                 uint64_t outer, uint32_t box_inner, uint32_t box_outer);

}  // namespace csa
