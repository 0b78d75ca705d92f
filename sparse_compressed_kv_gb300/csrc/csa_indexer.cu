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

template <int G, bool kFp4 = false>
struct IdxCfg {
    static constexpr int kN = 64 * G;                     // MMA N (heads x tokens)
    // bf16 key ring: filled by TMA (bf16 keys) or by the converter warps
    // (FP4 keys, which arrive in a deeper ring of their own)
    static constexpr int kStages = kFp4 ? 2 : 4;
    static constexpr int kABox = kTileKeys * 64 * 2;      // one 64-column box of keys: 16 KiB
    static constexpr int kABytes = 2 * kABox;             // one key tile: 32 KiB
    static constexpr int kBBox = kN * 64 * 2;
    static constexpr int kBBytes = 2 * kBBox;             // queries of one unit
    // TMEM accumulators: enough tiles in flight that the hand-back of an
    // accumulator (MMA done -> epilogue loads -> release) stays hidden
    static constexpr int kAcc = G == 1 ? 4 : 2;
    static constexpr int kTmemCols = kAcc * kN;           // a power of two <= 512
    static constexpr int kMaxUnits = 4096;
    // Epilogue: two warps per TMEM lane quarter.  One token per tile: the
    // two groups of four take alternate tiles (each owns one of the two
    // accumulators); several tokens per tile: each group takes half of them.
    static constexpr int kEpiWarps = G >= 2 ? 8 : 4;
    static constexpr bool kTileSplit = G == 1 && kEpiWarps == 8;
    // FP4 keys: 80-byte rows (64 code bytes, 4 scales, 12 zero) in a ring of
    // their own, expanded to bf16 by four converter warps (one row each lane)
    static constexpr int kFRow = 80;
    static constexpr int kFBytes = kTileKeys * kFRow;   // one FP4 key tile: 10 KiB
    static constexpr int kFStages = kFp4 ? 8 : 0;
    static constexpr int kConvWarps = kFp4 ? 8 : 0;  // two lanes per key row
    static constexpr int kThreads = 64 + 32 * (kEpiWarps + kConvWarps);
    static constexpr int kBarBytes = (2 * kStages + 2 + 2 * kAcc + 2 * kFStages) * 8;
    static constexpr size_t kSmemMain =
        size_t(kStages) * kABytes + kBBytes + size_t(kFStages) * kFBytes;
    static size_t smem_bytes(bool hist) {
        size_t s = 1024 /* alignment slack */ + kSmemMain + kBarBytes + 16 /* tmem holder */ +
                   (kMaxUnits + 4) * 4 /* prefix */;
        if (hist) s += 2 * kD1Bins * 4;
        if (kFp4) s += 256 * 8;  // code-pair table
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

// bf16 bits of one e2m1 code (OCP definition: sign bit 3, exponent bits
// 2..1 with bias 1, mantissa bit 0): 0.5 is 2^-1; e >= 1 is 2^(e-1) times
// 1 + m/2.
__device__ __forceinline__ uint32_t e2m1_bf16_bits(uint32_t code) {
    const uint32_t e = (code >> 1) & 3u, m = code & 1u;
    const uint32_t mag = e == 0 ? (m ? 0x3F00u : 0u) : (((126u + e) << 7) | (m << 6));
    return mag | ((code & 8u) << 12);
}

// Table entry for one code byte: its two values as bf16x2 (low nibble in
// the low half) at scale 1, and a mask of the halves that are not zero.
__device__ __forceinline__ uint2 fp4_pair_entry(uint32_t byte) {
    const uint32_t lo = byte & 15u, hi = byte >> 4;
    uint2 r;
    r.x = e2m1_bf16_bits(lo) | (e2m1_bf16_bits(hi) << 16);
    r.y = ((lo & 7u) ? 0x0000FFFFu : 0u) | ((hi & 7u) ? 0xFFFF0000u : 0u);
    return r;
}

// Two codes times the block scale 2^(E-127), as bf16x2.  For E in 2 .. 252
// the product only moves the exponent fields of the nonzero halves (no half
// leaves the normal range); other scales go through f32, still exactly.
__device__ __forceinline__ uint32_t fp4_expand_pair(const uint2 *lut, uint32_t byte, uint32_t E) {
    const uint2 t = lut[byte];
    if (E >= 2u && E <= 252u) {
        const int sh = static_cast<int>(E) - 127;
        const uint32_t d = static_cast<uint32_t>(sh >= 0 ? sh : -sh) * 0x00800080u;
        return sh >= 0 ? t.x + (d & t.y) : t.x - (d & t.y);
    }
    const float scale = ldexpf(1.0f, static_cast<int>(E) - 127);
    const float a = __uint_as_float((t.x & 0xFFFFu) << 16) * scale;
    const float b = __uint_as_float(t.x & 0xFFFF0000u) * scale;
    return pack_bf16x2(a, b);
}

__device__ __forceinline__ int find_unit(const int32_t *prefix, int n, int u) {
    int lo = 0, hi = n;  // invariant: prefix[lo] <= u < prefix[hi]
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (prefix[mid] <= u) lo = mid;
        else hi = mid;
    }
    return lo;
}

template <int G, bool kHist, bool kFp4>
__global__ void __launch_bounds__(IdxCfg<G, kFp4>::kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                   const IndexerParams P) {
    using C = IdxCfg<G, kFp4>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_smem<1024>(smem_raw);
    uint8_t *sA = smem;
    uint8_t *sB = smem + C::kStages * C::kABytes;
    uint8_t *sF = sB + C::kBBytes;  // FP4 key ring (FP4 only)
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kSmemMain);
    uint64_t *a_full = bars;
    uint64_t *a_empty = bars + C::kStages;
    uint64_t *b_full = bars + 2 * C::kStages;
    uint64_t *b_empty = b_full + 1;
    uint64_t *acc_full = b_full + 2;           // [kAcc]
    uint64_t *acc_empty = acc_full + C::kAcc;  // [kAcc]
    uint64_t *f_full = acc_empty + C::kAcc;    // [kFStages]
    uint64_t *f_empty = f_full + C::kFStages;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(
        bars + 2 * C::kStages + 2 + 2 * C::kAcc + 2 * C::kFStages);
    int32_t *prefix = reinterpret_cast<int32_t *>(tmem_holder + 4);
    uint32_t *hist_s = reinterpret_cast<uint32_t *>(prefix + C::kMaxUnits + 4);
    uint2 *pair_lut = reinterpret_cast<uint2 *>(hist_s + (kHist ? 2 * kD1Bins : 0));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int T = P.L.num_tokens;
    const int nu = P.num_units;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&a_full[s], kFp4 ? C::kConvWarps : 1);
            mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < C::kFStages; ++s) {
            mbar_init(&f_full[s], 1);
            mbar_init(&f_empty[s], C::kConvWarps);
        }
        mbar_init(b_full, 1);
        mbar_init(b_empty, 1);
        for (int a = 0; a < C::kAcc; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], C::kTileSplit ? 128 : 32 * C::kEpiWarps);
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
    // One sequence, one unit: while the layout is read, warm L2 with this
    // CTA's first key tiles as they fall when the sequence starts at row 0 and
    // fills the cache.  A guess: a layout that says otherwise costs bandwidth,
    // never data (nothing is read from this warming).
    if (threadIdx.x == 0 && nu == 1 && P.L.num_seqs == 1) {
        const int Us = static_cast<int>((P.L.max_comp_rows + kTileKeys - 1) / kTileKeys);
        const int s0 = static_cast<int>(static_cast<int64_t>(Us) * blockIdx.x / gridDim.x);
        const int s1 = static_cast<int>(static_cast<int64_t>(Us) * (blockIdx.x + 1) / gridDim.x);
        for (int u = s0; u < s1 && u < s0 + 4; ++u) {
            if constexpr (kFp4) {
                tma_prefetch_l2_2d(&tm_k, 0, u * kTileKeys);
            } else {
                tma_prefetch_l2_2d(&tm_k, 0, u * kTileKeys);
                tma_prefetch_l2_2d(&tm_k, 64, u * kTileKeys);
            }
        }
    }

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
                const int32_t row0 = static_cast<int32_t>(row_base + static_cast<int64_t>(j) * kTileKeys);
                if constexpr (kFp4) {
                    // 128 rows of 80 bytes into the FP4 ring (the converters
                    // fill the bf16 ring from it)
                    const int fs = it % C::kFStages;
                    const uint32_t fph = static_cast<uint32_t>(it / C::kFStages) & 1u;
                    if (!mbar_wait(&f_empty[fs], fph ^ 1u, P.status)) break;
                    mbar_arrive_expect_tx(&f_full[fs], C::kFBytes);
                    tma_load_2d(sF + fs * C::kFBytes, &tm_k, 0, row0, &f_full[fs], pol_k);
                } else {
                    const int stage = it % C::kStages;
                    const uint32_t ph = static_cast<uint32_t>(it / C::kStages) & 1u;
                    if (!mbar_wait(&a_empty[stage], ph ^ 1u, P.status)) break;
                    mbar_arrive_expect_tx(&a_full[stage], C::kABytes);
                    uint8_t *dst = sA + stage * C::kABytes;
                    tma_load_2d(dst, &tm_k, 0, row0, &a_full[stage], pol_k);
                    tma_load_2d(dst + C::kABox, &tm_k, 64, row0, &a_full[stage], pol_k);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0 && u0 < u1) {
            constexpr uint32_t idesc = idesc_bf16_f32<kTileKeys, C::kN>();
            int unit = find_unit(prefix, nu, u0), cur = -1;
            uint32_t gsw = 0;
            int it = 0;
            // descriptors built once, stepped by byte offset / 16 (shared
            // addresses stay below 256 KiB: the start-address field never carries)
            const uint64_t a_desc = sw128_kmajor_desc(smem_addr(sA));
            const uint64_t b_desc = sw128_kmajor_desc(smem_addr(sB));
            for (int u = u0; u < u1; ++u, ++it) {
                while (u >= prefix[unit + 1]) ++unit;
                if (unit != cur) {
                    if (!mbar_wait(b_full, gsw & 1u, P.status)) break;
                    cur = unit;
                    ++gsw;
                }
                const int acc = it % C::kAcc;
                if (!mbar_wait(&acc_empty[acc], (static_cast<uint32_t>(it / C::kAcc) & 1u) ^ 1u,
                               P.status))
                    break;
                const int stage = it % C::kStages;
                const uint32_t ph = static_cast<uint32_t>(it / C::kStages) & 1u;
                if (!mbar_wait(&a_full[stage], ph, P.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::kN);
                const uint64_t a_st = a_desc + static_cast<uint64_t>((stage * C::kABytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < kIHD / 16; ++kk) {
                    const uint32_t a_off = (kk >> 2) * C::kABox + (kk & 3) * 32;
                    const uint32_t b_off = (kk >> 2) * C::kBBox + (kk & 3) * 32;
                    umma_bf16(d_tmem, a_st + (a_off >> 4), b_desc + (b_off >> 4), idesc, kk > 0 ? 1u : 0u);
                }
                umma_commit(&a_empty[stage]);
                umma_commit(&acc_full[acc]);
                if (u + 1 == u1 || u + 1 >= prefix[unit + 1]) umma_commit(b_empty);
            }
        }
    } else if (warp < 2 + C::kEpiWarps) {
        // ------------------------------------------------ epilogue
        // No barrier inside this loop: a warp that gives up on a wait must not
        // strand the others.  Head weights are read through the read-only
        // cache (one broadcast address per warp-load, four weights per load
        // when aligned); the histogram keeps two per-unit slots in shared
        // memory and sends later units straight to global memory.  Group
        // `grp` (four warps, one per TMEM lane quarter) takes alternate tiles
        // (kTileSplit: the even or the odd ones) or half of each tile's tokens.
        constexpr bool kTokenSplit = C::kEpiWarps == 8 && !C::kTileSplit;
        constexpr int kGPer = kTokenSplit ? G / 2 : G;
        const uint64_t pol_sc = G > 1 ? policy_evict_first() : 0ull;
        const int grp = (warp - 2) >> 2;
        const int gbeg = kTokenSplit ? grp * kGPer : 0;
        const int tstep = C::kTileSplit ? 2 : 1;
        const int ep = threadIdx.x - 64;
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const int first_unit = (u0 < u1) ? find_unit(prefix, nu, u0) : 0;
        int unit = first_unit, cur = -1;
        int it = C::kTileSplit ? grp : 0;
        int64_t nv[kGPer];
#pragma unroll
        for (int g = 0; g < kGPer; ++g) nv[g] = 0;
        for (int u = u0 + it; u < u1; u += tstep, it += tstep) {
            while (u >= prefix[unit + 1]) ++unit;
            if (unit != cur) {
#pragma unroll
                for (int g = 0; g < kGPer; ++g) {
                    const int t = unit * G + gbeg + g;
                    nv[g] = t < T ? token_view(P.L, P.ratio, t).n_vis : 0;
                }
                cur = unit;
            }
            const int acc = it % C::kAcc;
            const bool ok = mbar_wait(&acc_full[acc], static_cast<uint32_t>(it / C::kAcc) & 1u, P.status);
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
                for (int i = ep; i < kD1Bins; i += 32 * C::kEpiWarps) {
                    const uint32_t c = hist_s[sl * kD1Bins + i];
                    if (c) atomicAdd(&gh[i], c);
                }
            }
        }
    } else if constexpr (kFp4) {
        // ------------------------------------------------ FP4 converter
        // Two lanes per key row of the tile, one per 64-column half: the
        // 80-byte row becomes 128 bf16 values in the 128-byte-swizzled K-major
        // layout the MMA reads (what TMA writes for bf16 keys: 16-byte chunk c
        // of row r at c ^ (r & 7)).
        // Every MXFP4 value is a bf16 value, so the expansion is exact.  Two
        // codes at a time through a 256-entry shared-memory table; the block
        // scale then moves the exponent fields.
        const int ct = threadIdx.x - 32 * (2 + C::kEpiWarps);  // 0 .. 255
        const int cr = ct & 127;      // key row of the tile
        const int half = ct >> 7;     // columns 64*half .. 64*half+63: blocks 2*half, 2*half+1
        for (int b = ct; b < 256; b += 32 * C::kConvWarps) pair_lut[b] = fp4_pair_entry(b);
        named_bar_sync(2, 32 * C::kConvWarps);
        const uint32_t sw = static_cast<uint32_t>(cr & 7);
        int it = 0;
        for (int u = u0; u < u1; ++u, ++it) {
            const int fs = it % C::kFStages;
            const uint32_t fph = static_cast<uint32_t>(it / C::kFStages) & 1u;
            const int as = it % C::kStages;
            const uint32_t aph = static_cast<uint32_t>(it / C::kStages) & 1u;
            const bool ok = mbar_wait(&f_full[fs], fph, P.status) &&
                            mbar_wait(&a_empty[as], aph ^ 1u, P.status);
            if (!__all_sync(0xffffffffu, ok)) break;
            const uint8_t *src = sF + fs * C::kFBytes + cr * C::kFRow;
            uint4 code[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) code[k] = reinterpret_cast<const uint4 *>(src)[2 * half + k];
            const uint32_t scales = *reinterpret_cast<const uint32_t *>(src + 64);
            uint8_t *dbox = sA + as * C::kABytes + half * C::kABox + cr * 128;
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
                const uint32_t E = (scales >> (8 * (2 * half + bb))) & 0xFFu;
                const uint32_t words[4] = {code[bb].x, code[bb].y, code[bb].z, code[bb].w};
                if (E >= 2u && E <= 252u) {
                    // the scale moves exponent fields only: add (or subtract)
                    // |E - 127| in both halves of every nonzero pair entry
                    const int sh = static_cast<int>(E) - 127;
                    const uint32_t d = static_cast<uint32_t>(sh >= 0 ? sh : -sh) * 0x00800080u;
                    const uint32_t neg = sh < 0 ? 0xFFFFFFFFu : 0u;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t o[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint2 t = pair_lut[(words[k] >> (8 * q)) & 0xFFu];
                            const uint32_t m = d & t.y;
                            o[q] = t.x + ((m ^ neg) - neg);  // +m, or -m in two's complement
                        }
                        const uint32_t chunk = static_cast<uint32_t>(bb * 4 + k);
                        *reinterpret_cast<uint4 *>(dbox + ((chunk ^ sw) << 4)) =
                            make_uint4(o[0], o[1], o[2], o[3]);
                    }
                } else {
#pragma unroll 1
                    for (int k = 0; k < 4; ++k) {
                        uint4 o;
                        o.x = fp4_expand_pair(pair_lut, words[k] & 0xFFu, E);
                        o.y = fp4_expand_pair(pair_lut, (words[k] >> 8) & 0xFFu, E);
                        o.z = fp4_expand_pair(pair_lut, (words[k] >> 16) & 0xFFu, E);
                        o.w = fp4_expand_pair(pair_lut, words[k] >> 24, E);
                        const uint32_t chunk = static_cast<uint32_t>(bb * 4 + k);
                        *reinterpret_cast<uint4 *>(dbox + ((chunk ^ sw) << 4)) = o;
                    }
                }
            }
            // the MMA reads these bytes through the async proxy
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&a_full[as]);
                mbar_arrive(&f_empty[fs]);
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

template <int G, bool kHist, bool kFp4>
static cudaError_t launch_g(const Launch &lc, const CUtensorMap &tk, const CUtensorMap &tq,
                            const IndexerParams &P, int64_t tiles_bound) {
    using C = IdxCfg<G, kFp4>;
    const size_t smem = C::smem_bytes(kHist);
    auto kern = indexer_kernel<G, kHist, kFp4>;
    cudaError_t e = set_kernel_smem(kern, smem);
    if (e != cudaSuccess) return e;
    int64_t grid = tiles_bound < lc.sm_count ? tiles_bound : lc.sm_count;
    if (grid < 1) grid = 1;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(C::kThreads), smem, lc.stream,
                      tk, tq, P);
}

cudaError_t launch_indexer(const Launch &lc, const csa_layout_t &L, const csa_params_t &p,
                           const void *q_idx, const float *w_idx, const void *k_idx,
                           float *scores, int64_t ld, uint32_t *state, int32_t *status,
                           bool fp4) {
    const int T = L.num_tokens;
    if (T <= 0 || L.total_comp_rows <= 0 || L.max_comp_rows <= 0) return cudaSuccess;
    // FP4 keys: one token per tile (the converter ring is sized for it)
    const int G = (!fp4 && L.num_seqs == 1 && T >= 4) ? 4 : 1;
    const bool fuse_hist = state != nullptr;
    if (fuse_hist && G != 1) return cudaErrorInvalidValue;

    CUtensorMap tk, tq;
    const CUresult ek =
        fp4 ? encode_tensor_map_2d_u8(&tk, k_idx, 80, static_cast<uint64_t>(L.total_comp_rows), 80,
                                      kTileKeys)
            : encode_tensor_map_2d_bf16(&tk, k_idx, kIHD, static_cast<uint64_t>(L.total_comp_rows),
                                        kIHD * 2, 64, kTileKeys);
    if (ek != CUDA_SUCCESS) return cudaErrorInvalidValue;
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
    if (fp4) {
        if (fuse_hist) return launch_g<1, true, true>(lc, tk, tq, P, tiles_bound);
        return launch_g<1, false, true>(lc, tk, tq, P, tiles_bound);
    }
    if (G == 4) return launch_g<4, false, false>(lc, tk, tq, P, tiles_bound);
    if (fuse_hist) return launch_g<1, true, false>(lc, tk, tq, P, tiles_bound);
    return launch_g<1, false, false>(lc, tk, tq, P, tiles_bound);
}

}  // namespace csa
