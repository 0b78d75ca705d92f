// csa_indexer.cu -- lightning indexer on the 5th-generation tensor cores.
//
//   score[t, s] = sum_h w[t,h] * ReLU(q^I[t,h,:] . K^I[s,:])
//
// ("ARCHITECTURE & MEMORY AUDIT -- Post-probe rewrite", F1 and F3: one
// 128-wide key per compressed block, shared by all 64 indexer heads.)
//
// The contraction is run "swap-AB": A = 128 compressed keys x 128 (the
// streamed operand, M = 128), B = the query heads of G tokens x 128 (N = 64G),
// so the f32 accumulator in TMEM holds one key per lane and one head per
// column.  The epilogue thread that owns a lane applies ReLU, the head weights
// and the head sum in registers: no cross-thread reduction.
//
// Persistent CTAs own contiguous ranges of (unit, key tile) work, where a unit
// is G consecutive query tokens of one sequence.  Warp roles:
//   warp 0      TMA producer: keys (4-stage ring, evict-first) and queries
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer
//   warps 2..5  epilogue: tcgen05.ld -> ReLU . w -> sum_h -> scores (+histogram)
// Accumulators are double-buffered in TMEM so the epilogue of tile i overlaps
// the MMAs of tile i+1.
#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

template <int G>
struct IdxCfg {
    static constexpr int kN = 64 * G;                     // MMA N (heads x tokens)
    static constexpr int kStages = 4;                     // key ring depth
    static constexpr int kABox = kTileKeys * 64 * 2;      // one 64-column box of keys: 16 KiB
    static constexpr int kABytes = 2 * kABox;             // one key tile: 32 KiB
    static constexpr int kBBox = kN * 64 * 2;
    static constexpr int kBBytes = 2 * kBBox;             // queries of one unit
    static constexpr int kTmemCols = 2 * kN;              // two accumulators (power of two)
    static constexpr int kMaxUnits = 4096;
    // Epilogue warps: one per TMEM lane quarter; with several tokens per tile
    // two per quarter, each taking half of the tokens.
    static constexpr int kEpiWarps = G >= 2 ? 8 : 4;
    static constexpr int kThreads = 64 + 32 * kEpiWarps;
    static constexpr int kBarBytes = (2 * kStages + 6) * 8;
    static constexpr size_t kSmemMain = size_t(kStages) * kABytes + kBBytes;
    static size_t smem_bytes(bool hist) {
        size_t s = 1024 /* alignment slack */ + kSmemMain + kBarBytes + 16 /* tmem holder */ +
                   (kMaxUnits + 4) * 4 /* prefix */;
        if (hist) s += 2 * kD1Bins * 4;
        return s;
    }
};

struct IndexerParams {
    csa_layout_t L;
    int32_t ratio;
    int32_t num_units;
    const float *w_idx;
    float *scores;
    int64_t ld;
    uint32_t *state;  // [T][kStateWords] when the digit-1 histogram is fused
    int32_t *status;
    int32_t w_vec;    // w_idx 16-byte aligned: four weights per load
};

__device__ __forceinline__ int find_unit(const int32_t *prefix, int n, int u) {
    int lo = 0, hi = n;  // invariant: prefix[lo] <= u < prefix[hi]
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (prefix[mid] <= u) lo = mid;
        else hi = mid;
    }
    return lo;
}

template <int G, bool kHist>
__global__ void __launch_bounds__(IdxCfg<G>::kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                   const IndexerParams P) {
    using C = IdxCfg<G>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + C::kStages * C::kABytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kSmemMain);
    uint64_t *a_full = bars;
    uint64_t *a_empty = bars + C::kStages;
    uint64_t *b_full = bars + 2 * C::kStages;
    uint64_t *b_empty = b_full + 1;
    uint64_t *acc_full = b_full + 2;   // [2]
    uint64_t *acc_empty = b_full + 4;  // [2]
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 2 * C::kStages + 6);
    int32_t *prefix = reinterpret_cast<int32_t *>(tmem_holder + 4);
    uint32_t *hist_s = reinterpret_cast<uint32_t *>(prefix + C::kMaxUnits + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int T = P.L.num_tokens;
    const int nu = P.num_units;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&a_full[s], 1);
            mbar_init(&a_empty[s], 1);
        }
        mbar_init(b_full, 1);
        mbar_init(b_empty, 1);
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 32 * C::kEpiWarps);
        }
        mbar_fence_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_q);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, C::kTmemCols);
        tmem_relinquish();
    }
    if (kHist)
        for (int i = threadIdx.x; i < 2 * kD1Bins; i += blockDim.x) hist_s[i] = 0;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    // Inputs may come from the preceding grid in the stream.
    pdl_wait();

    // Tiles per unit -> exclusive prefix over units.
    if (threadIdx.x == 0) prefix[0] = 0;
    for (int u = threadIdx.x; u < nu; u += blockDim.x) {
        int64_t nv = 0;
        int bad = 0;
        for (int g = 0; g < G; ++g) {
            int t = u * G + g;
            if (t < T) {
                TokenView v = token_view(P.L, P.ratio, t);
                bad |= v.bad;
                nv = v.n_vis > nv ? v.n_vis : nv;
            }
        }
        if (bad && blockIdx.x == 0) raise_status(P.status, bad);
        prefix[u + 1] = static_cast<int32_t>((nv + kTileKeys - 1) / kTileKeys);
    }
    __syncthreads();
    if (warp == 0) {
        int seg = (nu + 31) >> 5;
        int beg = min(nu, lane * seg), end = min(nu, beg + seg);
        int sum = 0;
        for (int i = beg; i < end; ++i) {
            sum += prefix[i + 1];
            prefix[i + 1] = sum;
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        int excl = incl - sum;
        for (int i = beg; i < end; ++i) prefix[i + 1] += excl;
    }
    __syncthreads();

    const int U = prefix[nu];
    const int u0 = static_cast<int>(static_cast<int64_t>(U) * blockIdx.x / gridDim.x);
    const int u1 = static_cast<int>(static_cast<int64_t>(U) * (blockIdx.x + 1) / gridDim.x);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0 && u0 < u1) {
            // One token per tile (decode): every key is read once, keep it
            // out of the way.  Several tokens per tile (prefill): every unit
            // of the sequence re-reads the same keys, keep them in L2.
            const uint64_t pol_k = G > 1 ? policy_evict_last() : policy_evict_first();
            const uint64_t pol_q = G > 1 ? policy_evict_normal() : policy_evict_last();
            int unit = find_unit(prefix, nu, u0), cur = -1;
            uint32_t gsw = 0;
            int64_t row_base = 0;
            int it = 0;
            for (int u = u0; u < u1; ++u, ++it) {
                while (u >= prefix[unit + 1]) ++unit;
                if (unit != cur) {
                    if (!mbar_wait(b_empty, (gsw & 1u) ^ 1u, P.status)) break;
                    mbar_arrive_expect_tx(b_full, C::kBBytes);
                    const int y = unit * G * 64;
                    tma_load_2d(sB, &tm_q, 0, y, b_full, pol_q);
                    tma_load_2d(sB + C::kBBox, &tm_q, 64, y, b_full, pol_q);
                    row_base = token_view(P.L, P.ratio, unit * G).off;
                    cur = unit;
                    ++gsw;
                }
                const int j = u - prefix[unit];
                const int stage = it % C::kStages;
                const uint32_t ph = static_cast<uint32_t>(it / C::kStages) & 1u;
                if (!mbar_wait(&a_empty[stage], ph ^ 1u, P.status)) break;
                mbar_arrive_expect_tx(&a_full[stage], C::kABytes);
                const int32_t row0 = static_cast<int32_t>(row_base + static_cast<int64_t>(j) * kTileKeys);
                uint8_t *dst = sA + stage * C::kABytes;
                tma_load_2d(dst, &tm_k, 0, row0, &a_full[stage], pol_k);
                tma_load_2d(dst + C::kABox, &tm_k, 64, row0, &a_full[stage], pol_k);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0 && u0 < u1) {
            constexpr uint32_t idesc = idesc_bf16_f32<kTileKeys, C::kN>();
            int unit = find_unit(prefix, nu, u0), cur = -1;
            uint32_t gsw = 0;
            int it = 0;
            const uint32_t a_base = smem_addr(sA);
            const uint32_t b_base = smem_addr(sB);
            for (int u = u0; u < u1; ++u, ++it) {
                while (u >= prefix[unit + 1]) ++unit;
                if (unit != cur) {
                    if (!mbar_wait(b_full, gsw & 1u, P.status)) break;
                    cur = unit;
                    ++gsw;
                }
                const int acc = it & 1;
                if (!mbar_wait(&acc_empty[acc], (static_cast<uint32_t>(it >> 1) & 1u) ^ 1u, P.status))
                    break;
                const int stage = it % C::kStages;
                const uint32_t ph = static_cast<uint32_t>(it / C::kStages) & 1u;
                if (!mbar_wait(&a_full[stage], ph, P.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::kN);
                const uint32_t a_st = a_base + stage * C::kABytes;
#pragma unroll
                for (int kk = 0; kk < kIHD / 16; ++kk) {
                    const uint32_t a_addr = a_st + (kk >> 2) * C::kABox + (kk & 3) * 32;
                    const uint32_t b_addr = b_base + (kk >> 2) * C::kBBox + (kk & 3) * 32;
                    umma_bf16(d_tmem, sw128_kmajor_desc(a_addr), sw128_kmajor_desc(b_addr), idesc,
                              kk > 0 ? 1u : 0u);
                }
                umma_commit(&a_empty[stage]);
                umma_commit(&acc_full[acc]);
                if (u + 1 == u1 || u + 1 >= prefix[unit + 1]) umma_commit(b_empty);
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        // No barrier inside this loop: a warp that gives up on a wait must not
        // strand the others.  Head weights are read through the read-only
        // cache (one broadcast address per warp-load, four weights per load
        // when aligned); the histogram keeps two per-unit slots in shared
        // memory and sends later units straight to global memory.  With two
        // warps per TMEM lane quarter, each takes half of the unit's tokens.
        constexpr int kGPer = C::kEpiWarps == 8 ? G / 2 : G;
        const uint64_t pol_sc = G > 1 ? policy_evict_first() : 0ull;
        const int gbeg = C::kEpiWarps == 8 ? ((warp - 2) >> 2) * kGPer : 0;
        const int ep = threadIdx.x - 64;
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const int first_unit = (u0 < u1) ? find_unit(prefix, nu, u0) : 0;
        int unit = first_unit, cur = -1, it = 0;
        int64_t nv[kGPer];
#pragma unroll
        for (int g = 0; g < kGPer; ++g) nv[g] = 0;
        for (int u = u0; u < u1; ++u, ++it) {
            while (u >= prefix[unit + 1]) ++unit;
            if (unit != cur) {
#pragma unroll
                for (int g = 0; g < kGPer; ++g) {
                    const int t = unit * G + gbeg + g;
                    nv[g] = t < T ? token_view(P.L, P.ratio, t).n_vis : 0;
                }
                cur = unit;
            }
            const int acc = it & 1;
            const bool ok = mbar_wait(&acc_full[acc], static_cast<uint32_t>(it >> 1) & 1u, P.status);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const int j = u - prefix[unit];
            const int64_t s = static_cast<int64_t>(j) * kTileKeys + row;
            // every TMEM load of the tile first, one wait, then the math
            float v[kGPer][4][16];
#pragma unroll
            for (int gi = 0; gi < kGPer; ++gi) {
                const uint32_t col = tmem_base + lane_addr +
                                     static_cast<uint32_t>(acc * C::kN + (gbeg + gi) * 64);
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) tmem_ld16(col + c4 * 16, v[gi][c4]);
            }
            tmem_wait_ld();
            // the accumulator is in registers: hand it back to the MMA warp
            // before the math
            tc_fence_before();
            mbar_arrive(&acc_empty[acc]);
#pragma unroll
            for (int gi = 0; gi < kGPer; ++gi) {
                const int g = gbeg + gi;
                const int t = unit * G + g;
                if (t >= T) continue;  // warp-uniform
                const float *wt = P.w_idx + static_cast<int64_t>(t) * kNIH;
                float part[4] = {0.f, 0.f, 0.f, 0.f};  // four short chains, summed in order
                if (P.w_vec) {
                    const float4 *wt4 = reinterpret_cast<const float4 *>(wt);
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                        for (int i = 0; i < 16; i += 4) {
                            const float4 w4 = __ldg(wt4 + (c4 * 16 + i) / 4);
                            part[c4] = fmaf(w4.x, fmaxf(v[gi][c4][i + 0], 0.f), part[c4]);
                            part[c4] = fmaf(w4.y, fmaxf(v[gi][c4][i + 1], 0.f), part[c4]);
                            part[c4] = fmaf(w4.z, fmaxf(v[gi][c4][i + 2], 0.f), part[c4]);
                            part[c4] = fmaf(w4.w, fmaxf(v[gi][c4][i + 3], 0.f), part[c4]);
                        }
                } else {
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            part[c4] = fmaf(__ldg(wt + c4 * 16 + i), fmaxf(v[gi][c4][i], 0.f), part[c4]);
                }
                const float score = (part[0] + part[1]) + (part[2] + part[3]);
                if (s < nv[gi]) {
                    float *dst = P.scores + static_cast<int64_t>(t) * P.ld + s;
                    // prefill rows (GBs) stream through L2 without displacing the keys
                    if (G > 1) st_global_hint(dst, score, pol_sc);
                    else *dst = score;
                    if (kHist) {
                        const uint32_t bin = score_key(score) >> kD1Shift;
                        const int slot = unit - first_unit;
                        if (slot < 2) atomicAdd(&hist_s[slot * kD1Bins + bin], 1u);
                        else atomicAdd(&P.state[static_cast<int64_t>(t) * kStateWords + bin], 1u);
                    }
                }
            }
        }
        if (kHist && u0 < u1) {
            named_bar_sync(1, 32 * C::kEpiWarps);
            const int last_unit = find_unit(prefix, nu, u1 - 1);
            const int nslots = min(2, last_unit - first_unit + 1);
            for (int sl = 0; sl < nslots; ++sl) {
                uint32_t *gh = P.state + static_cast<int64_t>(first_unit + sl) * kStateWords;
                for (int i = ep; i < kD1Bins; i += 128) {
                    const uint32_t c = hist_s[sl * kD1Bins + i];
                    if (c) atomicAdd(&gh[i], c);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    pdl_launch_dependents();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

bool indexer_fuses_hist(const csa_layout_t &L) {
    // one token per unit, and a top-k that filters with several CTAs per token
    if (L.num_seqs == 1 && L.num_tokens >= 4) return false;
    int32_t chunk = 0, per_tok = 0;
    topk_grid(L.num_tokens, L.max_comp_rows, &chunk, &per_tok);
    return per_tok > 1;
}

template <int G, bool kHist>
static cudaError_t launch_g(const Launch &lc, const CUtensorMap &tk, const CUtensorMap &tq,
                            const IndexerParams &P, int64_t tiles_bound) {
    using C = IdxCfg<G>;
    const size_t smem = C::smem_bytes(kHist);
    auto kern = indexer_kernel<G, kHist>;
    cudaError_t e = set_kernel_smem(kern, smem);
    if (e != cudaSuccess) return e;
    int64_t grid = tiles_bound < lc.sm_count ? tiles_bound : lc.sm_count;
    if (grid < 1) grid = 1;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(C::kThreads), smem, lc.stream,
                      tk, tq, P);
}

cudaError_t launch_indexer(const Launch &lc, const csa_layout_t &L, const csa_params_t &p,
                           const void *q_idx, const float *w_idx, const void *k_idx,
                           float *scores, int64_t ld, uint32_t *state, int32_t *status) {
    const int T = L.num_tokens;
    if (T <= 0 || L.total_comp_rows <= 0 || L.max_comp_rows <= 0) return cudaSuccess;
    const int G = (L.num_seqs == 1 && T >= 4) ? 4 : 1;
    const bool fuse_hist = state != nullptr;
    if (fuse_hist && G != 1) return cudaErrorInvalidValue;

    CUtensorMap tk, tq;
    if (encode_tensor_map_2d_bf16(&tk, k_idx, kIHD, static_cast<uint64_t>(L.total_comp_rows),
                                  kIHD * 2, 64, kTileKeys) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (encode_tensor_map_2d_bf16(&tq, q_idx, kIHD, static_cast<uint64_t>(T) * kNIH, kIHD * 2, 64,
                                  64 * G) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    IndexerParams P;
    P.L = L;
    P.ratio = p.ratio;
    P.num_units = (T + G - 1) / G;
    P.w_idx = w_idx;
    P.scores = scores;
    P.ld = ld;
    P.state = state;
    P.status = status;
    P.w_vec = reinterpret_cast<uintptr_t>(w_idx) % 16 == 0 ? 1 : 0;  // rows are 256 B apart
    const int64_t tiles_bound =
        static_cast<int64_t>(P.num_units) * ((L.max_comp_rows + kTileKeys - 1) / kTileKeys);
    if (G == 4) return launch_g<4, false>(lc, tk, tq, P, tiles_bound);
    if (fuse_hist) return launch_g<1, true>(lc, tk, tq, P, tiles_bound);
    return launch_g<1, false>(lc, tk, tq, P, tiles_bound);
}

}  // namespace csa
