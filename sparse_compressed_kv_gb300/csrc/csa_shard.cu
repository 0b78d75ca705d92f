// csa_shard.cu -- one sequence's compressed blocks sharded into contiguous
// ranges, each range on its own device.
//
// ("ARCHITECTURE & MEMORY AUDIT -- 1M-context viability", PART 2, "Total KV
// cache @ 1M context": the KV cache sharded across the GPUs.)  Shard g holds
// blocks [lo_g, hi_g) of the sequence as rows 0 .. hi_g - lo_g - 1 of its own
// key and row caches.  A decode step then runs as
//   1. per shard: scores of its visible blocks and their local top-k
//      (csa_shard_candidates: k candidates with their scores);
//   2. one exchange (the candidates of every shard), then the global top-k
//      with the single-device rule, score descending, block index ascending
//      (csa_shard_merge): a block of the global top-k is in its own shard's
//      top-k, so the merge sees every block it needs;
//   3. per shard: attention over its own selected rows, and on one device
//      over the window rows, each emitting an unnormalised partial (O, m, l)
//      (csa_shard_attention, csa_window_attention);
//   4. one exchange of the partials and one log-sum-exp combine
//      (csa_shard_combine).
// This file holds the shard's view of the layout (a device-side rewrite of
// the token positions and block offsets, so the single-device kernels run on
// a shard unchanged), the candidate list and the merge.
#include <math.h>

#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {
namespace {

// The shard's layout: one sequence whose blocks are the shard's rows, and
// per token a position p' with floor(p' / ratio) = the number of the shard's
// blocks the token sees, n' = clamp(n_vis - lo, 0, hi - lo), so that
// token_view on the rewritten layout yields n' visible blocks at rows 0..n'-1.
__global__ void shard_layout_kernel(const csa_layout_t L, int32_t ratio, int64_t lo, int64_t hi,
                                    int64_t *tok_pos_out, int64_t *comp_off_out, int32_t *status) {
    // (no early start for the next kernel: the decode indexer reads the layout
    // this kernel writes before it waits for the preceding grid)
    pdl_wait();
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t == 0) {
        comp_off_out[0] = 0;
        comp_off_out[1] = hi - lo;
    }
    if (t >= L.num_tokens) return;
    const TokenView v = token_view(L, ratio, t);
    int64_t nl = 0;
    if (v.bad & CSA_DEV_BAD_LAYOUT) {
        raise_status(status, v.bad);
    } else {
        if (v.bad) raise_status(status, v.bad);
        nl = v.n_vis - lo;
        nl = nl < 0 ? 0 : nl;
        nl = nl < hi - lo ? nl : hi - lo;
    }
    tok_pos_out[t] = nl * ratio;
}

// Candidates of the shard: its local selection with global block indices and
// the scores they were selected on; entries past the count hold -1 / -inf.
// n_sel == nullptr: an empty shard (no candidates).
__global__ void shard_candidates_kernel(int32_t T, int32_t top_k, int64_t lo, const float *scores,
                                        int64_t ld, const int32_t *idx, const int32_t *n_sel,
                                        float *cand_score, int32_t *cand_idx, int32_t *n_cand) {
    pdl_wait();
    pdl_launch_dependents();
    const int t = blockIdx.y;
    if (t >= T) return;
    const int n = n_sel ? n_sel[t] : 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) n_cand[t] = n;
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < top_k; j += gridDim.x * blockDim.x) {
        const int64_t o = static_cast<int64_t>(t) * top_k + j;
        if (j < n) {
            const int32_t s = idx[o];
            cand_idx[o] = static_cast<int32_t>(lo + s);
            cand_score[o] = scores[static_cast<int64_t>(t) * ld + s];
        } else {
            cand_idx[o] = -1;
            cand_score[o] = -INFINITY;
        }
    }
}

constexpr int kMergeThreads = 1024;

// Bitonic sort of n (a power of two) 64-bit keys in shared memory, descending.
__device__ void bitonic_desc(uint64_t *a, int n) {
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const int p = i ^ j;
                if (p > i) {
                    const uint64_t x = a[i], y = a[p];
                    // descending within blocks whose bit k is clear, ascending otherwise
                    const bool desc = (i & k) == 0;
                    if (desc ? x < y : x > y) {
                        a[i] = y;
                        a[p] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
}

// One CTA per token: the k' = min(top_k, candidates) best of every shard's
// candidates by (score descending, block index ascending), as the ascending
// block list idx and, per shard, its part of that list in local rows.
__global__ void __launch_bounds__(kMergeThreads) shard_merge_kernel(const ShardMergeArgs A) {
    pdl_wait();
    pdl_launch_dependents();
    extern __shared__ uint64_t mkeys[];   // [npad]
    __shared__ int32_t tot_s;      // valid candidates
    __shared__ int32_t cnt_s[kMaxShards];
    const int t = blockIdx.x;
    const int T = A.T, K = A.top_k, G = A.G;
    if (threadIdx.x == 0) {
        for (int g = 0; g < G; ++g) {
            int c = A.n_cand[static_cast<int64_t>(g) * T + t];
            if (c < 0 || c > K) {
                raise_status(A.status, CSA_DEV_BAD_LENGTH);
                c = c < 0 ? 0 : K;
            }
            cnt_s[g] = c;
        }
        tot_s = 0;
    }
    __syncthreads();
    const int npad = A.npad;
    // key = score key << 32 | (2^32 - 1 - block): larger is better, and at
    // equal scores the lower block index is larger
    for (int i = threadIdx.x; i < npad; i += blockDim.x) mkeys[i] = 0;
    __syncthreads();
    int base = 0, valid = 0;
    for (int g = 0; g < G; ++g) {
        const int c = cnt_s[g];
        const int64_t o = (static_cast<int64_t>(g) * T + t) * K;
        for (int j = threadIdx.x; j < c; j += blockDim.x) {
            const int32_t b = A.cand_idx[o + j];
            const bool ok = b >= 0 && b < A.bounds[G];
            if (!ok) raise_status(A.status, CSA_DEV_BAD_INDEX);   // dropped (its key stays 0)
            if (ok && CSA_CHECK(base + j < npad, A.status)) {
                mkeys[base + j] = (static_cast<uint64_t>(score_key(A.cand_score[o + j])) << 32) |
                                  (0xffffffffu - static_cast<uint32_t>(b));
                ++valid;
            }
        }
        base += c;
    }
    if (valid) atomicAdd(&tot_s, valid);
    __syncthreads();
    bitonic_desc(mkeys, npad);
    const int tot = tot_s;
    const int kk = tot < K ? tot : K;
    // the selected blocks, ascending, in the kpad words after the keys
    // (entries past kk pad with the largest value, so they sort last)
    uint32_t *sel = reinterpret_cast<uint32_t *>(mkeys + npad);   // [kpad] after the keys
    const int kpad = A.kpad;
    for (int i = threadIdx.x; i < kpad; i += blockDim.x)
        sel[i] = i < kk ? 0xffffffffu - static_cast<uint32_t>(mkeys[i] & 0xffffffffu) : 0xffffffffu;
    __syncthreads();
    // ascending bitonic sort of the kpad block indices
    for (int k = 2; k <= kpad; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < kpad; i += blockDim.x) {
                const int p = i ^ j;
                if (p > i) {
                    const uint32_t x = sel[i], y = sel[p];
                    const bool asc = (i & k) == 0;
                    if (asc ? x > y : x < y) {
                        sel[i] = y;
                        sel[p] = x;
                    }
                }
            }
            __syncthreads();
        }
    int32_t *out = A.idx + static_cast<int64_t>(t) * K;
    for (int i = threadIdx.x; i < K; i += blockDim.x) out[i] = i < kk ? static_cast<int32_t>(sel[i]) : -1;
    if (threadIdx.x == 0) A.n_sel[t] = kk;
    // each shard's blocks form one run of the ascending list
    for (int g = 0; g < G; ++g) {
        const int64_t lo = A.bounds[g], hi = A.bounds[g + 1];
        if (threadIdx.x == 0) cnt_s[g] = 0;
        __syncthreads();
        int mine = 0;
        for (int i = threadIdx.x; i < kk; i += blockDim.x) mine += static_cast<int64_t>(sel[i]) < lo ? 1 : 0;
        if (mine) atomicAdd(&cnt_s[g], mine);
        __syncthreads();
        const int first = cnt_s[g];
        __syncthreads();
        int32_t *so = A.shard_idx + (static_cast<int64_t>(g) * T + t) * K;
        int n = 0;
        // the run's length: entries in [lo, hi) (all after `first`)
        for (int i = threadIdx.x; i < kk; i += blockDim.x) {
            const int64_t b = sel[i];
            n += (b >= lo && b < hi) ? 1 : 0;
        }
        if (threadIdx.x == 0) cnt_s[g] = 0;
        __syncthreads();
        if (n) atomicAdd(&cnt_s[g], n);
        __syncthreads();
        const int len = cnt_s[g];
        for (int i = threadIdx.x; i < K; i += blockDim.x)
            so[i] = i < len ? static_cast<int32_t>(static_cast<int64_t>(sel[first + i]) - lo) : -1;
        if (threadIdx.x == 0) A.shard_nsel[static_cast<int64_t>(g) * T + t] = len;
        __syncthreads();
    }
}

int pow2_at_least(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

}  // namespace

cudaError_t launch_shard_layout(const Launch &lc, const csa_layout_t &L, int32_t ratio,
                                int64_t lo, int64_t hi, int64_t *tok_pos_out,
                                int64_t *comp_off_out, int32_t *status) {
    const int T = L.num_tokens;
    const unsigned blocks = static_cast<unsigned>((T + 255) / 256 > 0 ? (T + 255) / 256 : 1);
    return launch_pdl(shard_layout_kernel, dim3(blocks), dim3(256), 0, lc.stream, L, ratio, lo, hi,
                      tok_pos_out, comp_off_out, status);
}

cudaError_t launch_shard_candidates(const Launch &lc, int32_t T, int32_t top_k, int64_t lo,
                                    const float *scores, int64_t ld, const int32_t *idx,
                                    const int32_t *n_sel, float *cand_score, int32_t *cand_idx,
                                    int32_t *n_cand) {
    if (T <= 0) return cudaSuccess;
    const unsigned bx = static_cast<unsigned>((top_k + 255) / 256);
    return launch_pdl(shard_candidates_kernel, dim3(bx, T), dim3(256), 0, lc.stream, T, top_k, lo,
                      scores, ld, idx, n_sel, cand_score, cand_idx, n_cand);
}

size_t shard_merge_smem(int G, int top_k) {
    return static_cast<size_t>(pow2_at_least(G * top_k)) * 8 + static_cast<size_t>(pow2_at_least(top_k)) * 4;
}

cudaError_t launch_shard_merge(const Launch &lc, ShardMergeArgs A) {
    if (A.T <= 0) return cudaSuccess;
    A.npad = pow2_at_least(A.G * A.top_k);
    A.kpad = pow2_at_least(A.top_k);
    const size_t smem = shard_merge_smem(A.G, A.top_k);
    cudaError_t e = set_kernel_smem(shard_merge_kernel, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(shard_merge_kernel, dim3(A.T), dim3(kMergeThreads), smem, lc.stream, A);
}

}  // namespace csa
