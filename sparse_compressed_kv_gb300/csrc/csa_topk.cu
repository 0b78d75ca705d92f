// csa_topk.cu -- exact top-k over the visible indexer scores.
//
// ("ARCHITECTURE & MEMORY AUDIT -- Post-probe rewrite", F3: the top_k best
// compressed blocks per query, tk = min(top_k, n_comp).)
//
// Ranking: score descending, block index ascending; -0.0 ties with +0.0.
// Output: the k' = min(top_k, n_vis) selected blocks in ascending index.
//
// Radix select on the order-preserving 32-bit key of each score:
//   digit 1 = key[31:21]  histogram built by the indexer epilogue (csa_decode)
//                          or by score_hist_kernel (csa_topk);
//   filter (many CTAs per token): blocks whose digit 1 exceeds the threshold
//                          digit are certainly selected; blocks equal to it are
//                          candidates;
//   resolve (the last CTA of each token, by atomic ticket): digits 2 and 3
//                          over the candidates give the exact k-th key; ties at
//                          that key are taken in ascending index order; a
//                          bitmap over the index range emits the set sorted.
// The result is a pure function of the score bits: no step depends on the
// order in which CTAs or atomics run.  The kernel that consumes a counter
// resets it, so the workspace is left zeroed for the next call.
#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

constexpr int kSelThreads = 512;
constexpr int kBitmapBits = 1 << 18;  // index window emitted per bitmap pass (32 KiB)
constexpr int kStagedCand = kBitmapBits / 64;  // candidates that fit in the bitmap's space

struct SelectParams {
    csa_layout_t L;
    int32_t ratio;
    int32_t top_k;
    const float *scores;
    int64_t ld;
    uint32_t *state;      // [T][kStateWords]: digit-1 histogram, then TokCounters
    int32_t *sel;         // [T][top_k]
    uint64_t *cand;       // [T][cap]
    int32_t cap;
    int32_t chunk;        // scores per filter CTA
    int32_t local_hist;   // one CTA per token builds digit 1 itself
    int32_t *idx_out;     // [T][top_k]
    int32_t *nsel_out;    // [T]
    int32_t *status;
};

// ---------------------------------------------------------------- helpers

// Block-wide exclusive scan of one value per thread (kSelThreads threads).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *warp_tmp,
                                                    uint32_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tmp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        uint32_t x = lane < nw ? warp_tmp[lane] : 0u;
        uint32_t xi = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, xi, o);
            if (lane >= o) xi += y;
        }
        if (lane < nw) warp_tmp[lane] = xi - x;
        if (lane == nw - 1 && total) *total = xi;
    }
    __syncthreads();
    uint32_t r = warp_tmp[warp] + incl - v;
    __syncthreads();
    return r;
}

// Given a histogram h[0..nbins) and a rank k >= 1 counted from the top,
// find the digit d with count(> d) < k <= count(>= d).  Writes d and
// count(> d).  nbins is a multiple of blockDim.x.
__device__ void find_threshold_digit(const uint32_t *h, int nbins, uint32_t k, uint32_t *warp_tmp,
                                     int32_t *d_out, uint32_t *gt_out) {
    const int per = nbins / blockDim.x;
    // thread i owns bins [nbins - (i+1)*per, nbins - i*per): thread 0 owns the top bins
    const int hi = nbins - threadIdx.x * per;
    uint32_t local = 0;
    for (int b = hi - 1; b >= hi - per; --b) local += h[b];
    uint32_t above = block_excl_scan(local, warp_tmp, nullptr);  // count in bins >= hi
    uint32_t run = above;
    for (int b = hi - 1; b >= hi - per; --b) {
        const uint32_t c = h[b];
        if (run < k && run + c >= k) {
            *d_out = b;
            *gt_out = run;
        }
        run += c;
    }
    __syncthreads();
}

__device__ __forceinline__ void warp_append(bool pred, uint32_t *counter, uint32_t limit,
                                            int32_t *buf_i32, uint64_t *buf_u64, uint64_t val,
                                            int32_t ival) {
    const unsigned m = __ballot_sync(0xffffffffu, pred);
    if (!m) return;
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(m) - 1;
    uint32_t base = 0;
    if (lane == leader) base = atomicAdd(counter, static_cast<uint32_t>(__popc(m)));
    base = __shfl_sync(0xffffffffu, base, leader);
    if (pred) {
        const uint32_t pos = base + __popc(m & ((1u << lane) - 1u));
        if (pos < limit) {
            if (buf_i32) buf_i32[pos] = ival;
            else buf_u64[pos] = val;
        }
    }
}

// ---------------------------------------------------------------- digit-1 histogram

__global__ void __launch_bounds__(256) score_hist_kernel(const SelectParams P) {
    __shared__ uint32_t h[kD1Bins];
    pdl_wait();
    const int t = blockIdx.y;
    for (int i = threadIdx.x; i < kD1Bins; i += blockDim.x) h[i] = 0;
    __syncthreads();
    const TokenView v = token_view(P.L, P.ratio, t);
    const int64_t n = v.n_vis;
    const int64_t b0 = static_cast<int64_t>(blockIdx.x) * P.chunk;
    const int64_t b1 = min(n, b0 + P.chunk);
    const float *sc = P.scores + static_cast<int64_t>(t) * P.ld;
    for (int64_t i = b0 + threadIdx.x; i < b1; i += blockDim.x)
        atomicAdd(&h[score_key(sc[i]) >> kD1Shift], 1u);
    __syncthreads();
    uint32_t *gh = P.state + static_cast<int64_t>(t) * kStateWords;
    for (int i = threadIdx.x; i < kD1Bins; i += blockDim.x)
        if (h[i]) atomicAdd(&gh[i], h[i]);
    pdl_launch_dependents();
}

// ---------------------------------------------------------------- filter + resolve

struct SelectSmem {
    uint32_t h[kD1Bins];          // digit histograms (reused per pass)
    uint32_t warp_tmp[32];
    uint32_t bitmap[kBitmapBits / 32];
    int32_t sel[kMaxTopK];        // selected indices (unordered until emitted)
    uint32_t nsel;
    int32_t d;                    // threshold digit of the current pass
    uint32_t gt;                  // count strictly above the threshold digit
    uint32_t total;
    uint32_t last;
    uint32_t tie_taken;
};

__global__ void __launch_bounds__(kSelThreads) select_kernel(const SelectParams P) {
    extern __shared__ uint8_t smem_raw[];
    SelectSmem &S = *reinterpret_cast<SelectSmem *>(smem_raw);
    const int t = blockIdx.y;
    const int tid = threadIdx.x;

    pdl_wait();

    const TokenView v = token_view(P.L, P.ratio, t);
    if (v.bad && blockIdx.x == 0 && tid == 0) raise_status(P.status, v.bad);
    const int64_t n = v.n_vis;
    const uint32_t kk = static_cast<uint32_t>(min(static_cast<int64_t>(P.top_k), n));
    const float *sc = P.scores + static_cast<int64_t>(t) * P.ld;
    uint32_t *gh = P.state + static_cast<int64_t>(t) * kStateWords;
    TokCounters *cnt = reinterpret_cast<TokCounters *>(gh + kD1Bins);

    // ---- digit-1 histogram and threshold (every CTA of the token)
    if (kk > 0 && kk < n) {
        if (P.local_hist) {
            for (int i = tid; i < kD1Bins; i += blockDim.x) S.h[i] = 0;
            __syncthreads();
            for (int64_t i = tid; i < n; i += blockDim.x) atomicAdd(&S.h[score_key(sc[i]) >> kD1Shift], 1u);
        } else {
            for (int i = tid; i < kD1Bins; i += blockDim.x) S.h[i] = __ldcg(&gh[i]);
        }
        __syncthreads();
        find_threshold_digit(S.h, kD1Bins, kk, S.warp_tmp, &S.d, &S.gt);
        const uint32_t d1 = static_cast<uint32_t>(S.d);

        // ---- filter this CTA's slice of the index range
        const int64_t b0 = P.local_hist ? 0 : static_cast<int64_t>(blockIdx.x) * P.chunk;
        const int64_t b1 = P.local_hist ? n : min(n, b0 + P.chunk);
        int32_t *selg = P.sel + static_cast<int64_t>(t) * P.top_k;
        uint64_t *candg = P.cand + static_cast<int64_t>(t) * P.cap;
        for (int64_t base = b0; base < b1; base += blockDim.x) {
            const int64_t i = base + tid;
            uint32_t key = 0, dg = 0;
            const bool in = i < b1;
            if (in) {
                key = score_key(__ldcg(&sc[i]));
                dg = key >> kD1Shift;
            }
            warp_append(in && dg > d1, &cnt->sel, static_cast<uint32_t>(P.top_k), selg, nullptr, 0,
                        static_cast<int32_t>(i));
            warp_append(in && dg == d1, &cnt->cand, static_cast<uint32_t>(P.cap), nullptr, candg,
                        (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(i), 0);
        }
    }

    // ---- last CTA of this token resolves
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(&cnt->ticket, 1u);
        S.last = (prev == gridDim.x - 1) ? 1u : 0u;
    }
    __syncthreads();
    if (!S.last) {
        pdl_launch_dependents();
        return;
    }
    __threadfence();

    int32_t *out = P.idx_out + static_cast<int64_t>(t) * P.top_k;
    if (kk == 0 || kk == n) {
        // nothing to rank: none visible, or every visible block fits
        for (int i = tid; i < P.top_k; i += blockDim.x) out[i] = i < static_cast<int>(kk) ? i : -1;
    } else {
        const uint32_t d1 = static_cast<uint32_t>(S.d);
        const uint32_t gt1 = S.gt;
        const uint32_t ncand = __ldcg(&cnt->cand);
        const bool overflow = ncand > static_cast<uint32_t>(P.cap);
        const int32_t *selg = P.sel + static_cast<int64_t>(t) * P.top_k;
        const uint64_t *candg = P.cand + static_cast<int64_t>(t) * P.cap;
        for (uint32_t i = tid; i < gt1; i += blockDim.x) S.sel[i] = __ldcg(&selg[i]);
        if (tid == 0) S.nsel = gt1;
        uint32_t need = kk - gt1;   // >= 1, all from digit-1 bin d1
        uint32_t prefix = d1;       // key bits fixed so far (top bits)
        int fixed = kD1Bits;        // how many top bits are fixed
        // Candidate source: the compacted list staged in shared memory (it
        // fits in the bitmap's space, which is only needed later), the list
        // in global memory when it is longer, or the whole row on overflow.
        const int64_t m = overflow ? n : static_cast<int64_t>(ncand);
        const bool staged = !overflow && ncand <= static_cast<uint32_t>(kStagedCand);
        uint64_t *cs = reinterpret_cast<uint64_t *>(S.bitmap);
        if (staged) {
            for (uint32_t i = tid; i < ncand; i += blockDim.x) cs[i] = __ldcg(&candg[i]);
            __syncthreads();
        }
        auto cand_key = [&](int64_t i, uint32_t &key, int64_t &index) {
            if (overflow) {
                key = score_key(__ldcg(&sc[i]));
                index = i;
            } else {
                const uint64_t c = staged ? cs[i] : __ldcg(&candg[i]);
                key = static_cast<uint32_t>(c >> 32);
                index = static_cast<int64_t>(c & 0xffffffffu);
            }
        };
        // ---- digits 2 and 3 among keys matching the fixed prefix
        for (int pass = 0; pass < 2; ++pass) {
            const int bits = pass == 0 ? kD2Bits : kD2Shift;
            const int shift = 32 - fixed - bits;
            const uint32_t mask = (1u << bits) - 1u;
            for (int i = tid; i < kD1Bins; i += blockDim.x) S.h[i] = 0;
            __syncthreads();
            for (int64_t i = tid; i < m; i += blockDim.x) {
                uint32_t key;
                int64_t index;
                cand_key(i, key, index);
                if ((key >> (32 - fixed)) == prefix) atomicAdd(&S.h[(key >> shift) & mask], 1u);
            }
            __syncthreads();
            find_threshold_digit(S.h, kD1Bins, need, S.warp_tmp, &S.d, &S.gt);
            need -= S.gt;
            prefix = (prefix << bits) | static_cast<uint32_t>(S.d);
            fixed += bits;
        }
        // prefix is now the full k-th key tau; need = how many keys equal to tau are taken
        const uint32_t tau = prefix;
        const uint32_t eq = S.h[S.d];
        // every key > tau among the candidates is selected
        for (int64_t base = 0; base < m; base += blockDim.x) {
            const int64_t i = base + tid;
            uint32_t key = 0;
            int64_t index = 0;
            if (i < m) cand_key(i, key, index);
            const bool take = i < m && (key >> (32 - kD1Bits)) == d1 && (key > tau || (key == tau && need == eq));
            const unsigned bm = __ballot_sync(0xffffffffu, take);
            if (bm) {
                const int lane = tid & 31;
                const int leader = __ffs(bm) - 1;
                uint32_t pos = 0;
                if (lane == leader) pos = atomicAdd(&S.nsel, static_cast<uint32_t>(__popc(bm)));
                pos = __shfl_sync(0xffffffffu, pos, leader);
                if (take) {
                    const uint32_t q = pos + __popc(bm & ((1u << lane) - 1u));
                    if (q < static_cast<uint32_t>(kMaxTopK)) S.sel[q] = static_cast<int32_t>(index);
                }
            }
        }
        __syncthreads();
        if (need != eq) {
            // ties straddle the cut: take the `need` lowest indices with key == tau,
            // scanning the row in index order.
            if (tid == 0) S.tie_taken = 0;
            __syncthreads();
            for (int64_t base = 0; base < n; base += blockDim.x) {
                const int64_t i = base + tid;
                const bool hit = i < n && score_key(__ldcg(&sc[i])) == tau;
                const uint32_t before = block_excl_scan(hit ? 1u : 0u, S.warp_tmp, &S.total);
                const uint32_t taken = S.tie_taken;
                if (hit && taken + before < need) S.sel[S.nsel + taken + before] = static_cast<int32_t>(i);
                __syncthreads();
                if (tid == 0) S.tie_taken = taken + S.total;
                __syncthreads();
                if (S.tie_taken >= need) break;
            }
            if (tid == 0) S.nsel += need;
            __syncthreads();
        }
        // ---- emit in ascending index through a bitmap of the index range
        const uint32_t ns = S.nsel;  // == kk
        uint32_t written = 0;
        for (int64_t w0 = 0; w0 < n; w0 += kBitmapBits) {
            const int64_t wlen = min(static_cast<int64_t>(kBitmapBits), n - w0);
            const int nwords = static_cast<int>((wlen + 31) >> 5);
            for (int i = tid; i < nwords; i += blockDim.x) S.bitmap[i] = 0;
            __syncthreads();
            for (uint32_t i = tid; i < ns; i += blockDim.x) {
                const int64_t x = S.sel[i];
                if (x >= w0 && x < w0 + wlen) atomicOr(&S.bitmap[(x - w0) >> 5], 1u << ((x - w0) & 31));
            }
            __syncthreads();
            const int per = (nwords + blockDim.x - 1) / blockDim.x;
            const int wb = min(nwords, static_cast<int>(tid) * per), we = min(nwords, wb + per);
            uint32_t c = 0;
            for (int i = wb; i < we; ++i) c += __popc(S.bitmap[i]);
            uint32_t pos = written + block_excl_scan(c, S.warp_tmp, &S.total);
            for (int i = wb; i < we; ++i) {
                uint32_t bits = S.bitmap[i];
                while (bits) {
                    const int b = __ffs(bits) - 1;
                    bits &= bits - 1;
                    if (pos < kk) out[pos] = static_cast<int32_t>(w0 + (static_cast<int64_t>(i) << 5) + b);
                    ++pos;
                }
            }
            written += S.total;
            __syncthreads();
        }
        for (int i = kk + tid; i < P.top_k; i += blockDim.x) out[i] = -1;
        if (written != kk && tid == 0) raise_status(P.status, CSA_DEV_BAD_INDEX);
    }
    if (tid == 0) P.nsel_out[t] = static_cast<int32_t>(kk);
    // ---- leave the workspace zeroed for the next call
    if (!P.local_hist)
        for (int i = tid; i < kD1Bins; i += blockDim.x) gh[i] = 0;
    if (tid == 0) {
        cnt->sel = 0;
        cnt->cand = 0;
        cnt->ticket = 0;
    }
    pdl_launch_dependents();
}

cudaError_t launch_topk(const Launch &lc, const csa_layout_t &L, const csa_params_t &p,
                        const float *scores, int64_t ld, const TopkWs &ws, bool hist_ready,
                        int32_t *idx, int32_t *n_sel, int32_t *status) {
    const int T = L.num_tokens;
    if (T <= 0) return cudaSuccess;
    SelectParams P;
    P.L = L;
    P.ratio = p.ratio;
    P.top_k = p.top_k;
    P.scores = scores;
    P.ld = ld;
    P.state = ws.state;
    P.sel = ws.sel;
    P.cand = ws.cand;
    P.cap = ws.cap;
    P.idx_out = idx;
    P.nsel_out = n_sel;
    P.status = status;
    const int64_t maxn = L.max_comp_rows > 0 ? L.max_comp_rows : 1;
    // CTAs per token: enough to cover ~2 waves in total, each with >= 1024 scores.
    int64_t want = (2 * static_cast<int64_t>(lc.sm_count) + T - 1) / T;
    int64_t chunk = (maxn + want - 1) / want;
    chunk = ((chunk + 1023) / 1024) * 1024;
    if (chunk < 1024) chunk = 1024;
    const int64_t per_tok = (maxn + chunk - 1) / chunk;
    P.chunk = static_cast<int32_t>(chunk);
    P.local_hist = (per_tok == 1 && !hist_ready) ? 1 : 0;
    cudaError_t e;
    if (!hist_ready && !P.local_hist) {
        e = launch_pdl(score_hist_kernel, dim3(static_cast<unsigned>(per_tok), T), dim3(256), 0,
                       lc.stream, P);
        if (e != cudaSuccess) return e;
    }
    const size_t smem = sizeof(SelectSmem);
    e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_pdl(select_kernel, dim3(static_cast<unsigned>(per_tok), T), dim3(kSelThreads),
                      smem, lc.stream, P);
}

}  // namespace csa
