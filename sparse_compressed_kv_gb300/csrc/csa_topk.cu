// csa_topk.cu -- exact top-k over the visible indexer scores.
//
// ("ARCHITECTURE & MEMORY AUDIT -- Post-probe rewrite", F3: the top_k best
// compressed blocks per query, tk = min(top_k, n_comp).)
//
// Ranking: score descending, block index ascending; -0.0 ties with +0.0.
// Output: the k' = min(top_k, n_vis) selected blocks in ascending index.
//
// Radix select on the order-preserving 32-bit key of each score:
//   digit 1 = key[31:21]  histogram built by the indexer epilogue (csa_decode),
//                          by score_hist_kernel (csa_topk), or, with one CTA
//                          per token, by that CTA itself;
//   filter                 every CTA of a token finds the threshold digit d1
//                          and compacts, with a block-wide scan, the entries
//                          (key, index) whose digit 1 is >= d1 into its own
//                          output slot: no shared counters, no contention;
//   resolve                the last CTA of the token (atomic ticket) reads
//                          the slot counts, the digit-2 histogram and every
//                          slot's first line in one round trip and stages the
//                          entries in shared memory in index order; digit-1
//                          winners are in; digit 2 comes from its histogram,
//                          and the few keys that share digits 1 and 2 with the
//                          k-th are ranked by one warp (a digit-3 histogram
//                          when they are more than 32), which gives the exact
//                          k-th key; ties at that key are taken in ascending
//                          index order; an ordered compaction emits the set.
// The result is a pure function of the score bits.  The kernel that consumes
// the per-token state (histogram, ticket) zeroes it for the next call.
#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

constexpr int kSelThreads = 512;
constexpr int kStageCap = 8192;        // entries staged in shared memory (64 KiB)
static_assert(kStageCap % (kSelThreads / 32) == 0, "per-warp staging runs");
constexpr int kMaxPerThread = kMaxFilterChunk / kSelThreads;
static_assert(kD2Bins == 4 * kSelThreads, "the resolver holds four digit-2 bins per thread");

// Resolver: the first kSpec entries of each of the first kSpecSlots slots (one
// 128-byte line, the part a filter CTA has just written) are read together
// with the slot counts: 16 bytes (two entries) per thread, eight threads per
// line, so each warp load covers four whole lines.
constexpr int kSpec = 16;
constexpr int kSpecLanes = kSpec / 2;                      // threads per slot line
constexpr int kSpecRounds = 4;                             // lines per thread
constexpr int kSpecSlots = kSelThreads / kSpecLanes * kSpecRounds;   // 256

struct SelectParams {
    csa_layout_t L;
    int32_t ratio;
    int32_t top_k;
    const float *scores;
    int64_t ld;
    uint32_t *state;      // [T][kStateWords]: digit-1 histogram, then TokCounters
    uint64_t *slots;      // [T][per_tok][chunk] (key << 32 | index), multi-CTA mode
    uint32_t *slot_cnt;   // [T][per_tok]
    int32_t chunk;        // scores per filter CTA
    int32_t per_tok;      // filter CTAs per token
    int32_t local_hist;   // one CTA per token builds digit 1 itself
    int32_t *idx_out;     // [T][top_k]
    int32_t *nsel_out;    // [T]
    int32_t *status;
};

// ---------------------------------------------------------------- helpers

// Block-wide exclusive scan of one value per thread, with one barrier: each
// warp scans its lanes and publishes its total in buf[warp]; after the
// barrier every warp reads all totals (a lane each) and sums those of the
// warps before its own in one warp reduction.  The reads of buf come after
// the barrier, so two scans with no barrier between them must use different
// buffers.  Thread 0 gets the block total in *total.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *buf, uint32_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) buf[warp] = incl;
    __syncthreads();
    const int nw = blockDim.x >> 5;
    const uint32_t x = lane < nw ? buf[lane] : 0u;
    const uint32_t before = __reduce_add_sync(0xffffffffu, lane < warp ? x : 0u);
    if (total && warp == 0) {
        const uint32_t all = __reduce_add_sync(0xffffffffu, x);
        if (lane == 0) *total = all;
    }
    return before + incl - v;
}

// Exclusive block scan of three counters packed in one 64-bit word: bits
// 42..63, 22..41 and 0..21, each of whose block totals fits its field (so no
// field carries into the next).  The warps scan the packed word; the sums of
// the warp totals before each warp are three 32-bit warp reductions.  One
// barrier; thread 0 gets the block total in *total.
constexpr int kPackA = 42, kPackB = 22;
constexpr uint32_t kMaskB = (1u << (kPackA - kPackB)) - 1u, kMaskC = (1u << kPackB) - 1u;
// every field's block total is at most the entries of one token's slots
static_assert(static_cast<int64_t>(kMaxPerTok) * kMaxFilterChunk <= kMaskC &&
                  static_cast<int64_t>(kMaxPerTok) * kMaxFilterChunk / 8 + kMaxPerTok <= kMaskB &&
                  kMaxPerTok <= kSelThreads,
              "packed resolver scan fields");
__device__ __forceinline__ uint64_t block_excl_scan3(uint64_t v, uint64_t *buf, uint64_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) buf[warp] = incl;
    __syncthreads();
    const int nw = blockDim.x >> 5;
    const uint64_t x = lane < nw ? buf[lane] : 0ull;
    auto sum3 = [](uint64_t y) {
        const uint32_t a = __reduce_add_sync(0xffffffffu, static_cast<uint32_t>(y >> kPackA));
        const uint32_t b = __reduce_add_sync(0xffffffffu, static_cast<uint32_t>(y >> kPackB) & kMaskB);
        const uint32_t c = __reduce_add_sync(0xffffffffu, static_cast<uint32_t>(y) & kMaskC);
        return (static_cast<uint64_t>(a) << kPackA) | (static_cast<uint64_t>(b) << kPackB) | c;
    };
    const uint64_t before = sum3(lane < warp ? x : 0ull);
    if (total && warp == 0) {
        const uint64_t all = sum3(x);
        if (lane == 0) *total = all;
    }
    return before + incl - v;
}

// Given a histogram h[0..kBins) in shared memory and a rank k >= 1 counted
// from the top, find the digit d with count(> d) < k <= count(>= d).  Writes
// d and count(> d).  Thread i holds the kBins / kSelThreads bins just below
// kBins - i * per (thread 0 the top ones), read as one vector.  Ends with a
// barrier after its last read of warp_tmp.
template <int kBins>
__device__ __forceinline__ void find_threshold_digit(const uint32_t *h, uint32_t k, uint32_t *warp_tmp,
                                                     int32_t *d_out, uint32_t *gt_out) {
    constexpr int per = kBins / kSelThreads;
    static_assert(kBins % kSelThreads == 0 && (per == 2 || per == 4), "bins per thread");
    const int hb = per * (kSelThreads - 1 - static_cast<int>(threadIdx.x));
    uint32_t v[per];
    if constexpr (per == 4) {
        const uint4 q = *reinterpret_cast<const uint4 *>(h + hb);
        v[0] = q.x;
        v[1] = q.y;
        v[2] = q.z;
        v[3] = q.w;
    } else {
        const uint2 q = *reinterpret_cast<const uint2 *>(h + hb);
        v[0] = q.x;
        v[1] = q.y;
    }
    uint32_t local = 0;
#pragma unroll
    for (int j = 0; j < per; ++j) local += v[j];
    uint32_t run = block_excl_scan(local, warp_tmp, nullptr);  // count in bins above hb + per - 1
#pragma unroll
    for (int j = per - 1; j >= 0; --j) {
        if (run < k && run + v[j] >= k) {
            *d_out = hb + j;
            *gt_out = run;
        }
        run += v[j];
    }
    __syncthreads();
}

// Shared-memory histogram increment, aggregated over the lanes of a warp that
// hit the same bin (scores cluster in few bins: plain atomics would serialise).
__device__ __forceinline__ void smem_hist_add(uint32_t *h, uint32_t bin, bool active) {
    const unsigned act = __ballot_sync(0xffffffffu, active);
    if (!active) return;
    const unsigned peers = __match_any_sync(act, bin);
    const int lane = threadIdx.x & 31;
    if (lane == __ffs(peers) - 1) atomicAdd(&h[bin], static_cast<uint32_t>(__popc(peers)));
}

// ---------------------------------------------------------------- digit-1 histogram

__global__ void __launch_bounds__(256) score_hist_kernel(const SelectParams P) {
    __shared__ uint32_t h[kD1Bins];
    __shared__ int64_t n_vis;
    pdl_wait();
    pdl_launch_dependents();
    const int t = blockIdx.y;
    for (int i = threadIdx.x; i < kD1Bins; i += blockDim.x) h[i] = 0;
    if (threadIdx.x == 0) n_vis = token_view(P.L, P.ratio, t).n_vis;   // one reader, shared
    __syncthreads();
    const int64_t n = n_vis;
    const int64_t b0 = static_cast<int64_t>(blockIdx.x) * P.chunk;
    const int64_t b1 = min(n, b0 + P.chunk);
    const float *sc = P.scores + static_cast<int64_t>(t) * P.ld;
    for (int64_t base = b0; base < b1; base += blockDim.x) {
        const int64_t i = base + threadIdx.x;
        smem_hist_add(h, i < b1 ? score_key(sc[i]) >> kD1Shift : 0u, i < b1);
    }
    __syncthreads();
    uint32_t *gh = P.state + static_cast<int64_t>(t) * kStateWords;
    for (int i = threadIdx.x; i < kD1Bins; i += blockDim.x)
        if (h[i]) atomicAdd(&gh[i], h[i]);
}

// ---------------------------------------------------------------- filter + resolve

struct SelectSmem {
    uint32_t h[kD1Bins];           // digit-1 histogram, then digit-3 histogram
    uint32_t h2[kD2Bins];          // digit-2 histogram of the threshold bin
    uint32_t warp_tmp[2 * 32];     // block scans: per-warp totals, two buffers
    uint64_t warp_tmp64[32];       // the one 64-bit scan
    uint64_t total64;
    uint64_t stage[kStageCap];     // entries (key << 32 | index), ascending index
    uint32_t prefix[kMaxPerTok + 1];
    uint32_t gprefix[kMaxPerTok + 1];  // staging groups of up to 8 entries per slot
    uint32_t wcount[32];           // one-CTA mode: entries per warp range
    uint32_t nstage;
    uint32_t overflow;
    int32_t d;                     // threshold digit of the current pass
    uint32_t gt;                   // count strictly above the threshold digit
    uint32_t last;
    int64_t n_vis;                 // the token's visible blocks
    uint32_t cand[32];             // keys sharing digits 1 and 2 with the k-th, when <= 32
    uint32_t ncand;
    uint32_t tau, need3, eq3;      // the k-th key, ties to take, ties in all
};

// Two CTAs per SM: the filter grid (about two CTAs per SM) runs in one wave.
__global__ void __launch_bounds__(kSelThreads, 2) select_kernel(const SelectParams P) {
    extern __shared__ uint8_t smem_raw[];
    SelectSmem &S = *reinterpret_cast<SelectSmem *>(align_smem<16>(smem_raw));
    const int t = blockIdx.y;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    constexpr int kWarps = kSelThreads / 32;

    pdl_wait();
    pdl_launch_dependents();

    uint32_t *gh = P.state + static_cast<int64_t>(t) * kStateWords;   // digit-1 histogram
    uint32_t *gh2 = gh + kD1Bins;                                       // digit-2 histogram
    TokCounters *cnt = reinterpret_cast<TokCounters *>(gh2 + kD2Bins);
    // the histogram's address depends only on t: load it while the token's
    // layout is being read
    uint32_t hreg[kD1Bins / kSelThreads];
    if (!P.local_hist)
#pragma unroll
        for (int u = 0; u < kD1Bins / kSelThreads; ++u) hreg[u] = __ldcg(&gh[u * kSelThreads + tid]);
    // Multi-CTA mode: this CTA's slice [c0, c0 + chunk) is loaded now too, in
    // coalesced warp spans (lane l of warp w holds index c0 + w*W + q*32 + l),
    // bounded by the row capacity; entries past the visible count are masked
    // once the layout is read.
    const int span = ((P.chunk + kWarps - 1) / kWarps + 31) & ~31;  // W, at most 32 * kMaxPerThread
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * P.chunk;
    const int64_t wbase = c0 + static_cast<int64_t>(warp) * span + lane;
    uint32_t keys[kMaxPerThread];
    if (!P.local_hist) {
        const int64_t cend = min(c0 + P.chunk, P.L.max_comp_rows);
        const float *row = P.scores + static_cast<int64_t>(t) * P.ld;
#pragma unroll
        for (int q = 0; q < kMaxPerThread; ++q) {
            const int64_t i = wbase + q * 32;
            keys[q] = (q * 32 < span && i < cend) ? score_key(__ldcg(row + i)) : 0u;
        }
    }
    // The token's record: one thread reads it (every thread of every CTA
    // reading the same few lines would queue thousands of requests on them)
    // and the barrier below shares it.
    if (tid == 0) {
        const TokenView v = token_view(P.L, P.ratio, t);
        if (v.bad && blockIdx.x == 0) raise_status(P.status, v.bad);
        S.n_vis = v.n_vis;
    }
    if (!P.local_hist)
#pragma unroll
        for (int u = 0; u < kD1Bins / kSelThreads; ++u) S.h[u * kSelThreads + tid] = hreg[u];
    __syncthreads();
    const int64_t n = S.n_vis;
    const uint32_t kk = static_cast<uint32_t>(min(static_cast<int64_t>(P.top_k), n));
    const float *sc = P.scores + static_cast<int64_t>(t) * P.ld;
    const bool rank = kk > 0 && kk < n;

    // ---- digit-1 threshold (every CTA of the token) and this CTA's entries
    if (rank) {
        if (P.local_hist) {
            for (int i = tid; i < kD1Bins; i += blockDim.x) S.h[i] = 0;
            for (int i = tid; i < kD2Bins; i += blockDim.x) S.h2[i] = 0;
            __syncthreads();
            // every lane runs the same number of iterations: the warp-wide
            // collectives inside smem_hist_add need the whole warp
            for (int64_t base = 0; base < n; base += blockDim.x) {
                const int64_t i = base + tid;
                smem_hist_add(S.h, i < n ? score_key(__ldcg(&sc[i])) >> kD1Shift : 0u, i < n);
            }
            __syncthreads();
        }
        find_threshold_digit<kD1Bins>(S.h, kk, S.warp_tmp, &S.d, &S.gt);
        const uint32_t d1 = static_cast<uint32_t>(S.d);

        if (P.local_hist) {
            // One CTA owns the row.  Warp w compacts its contiguous index range
            // in order into its own part of the staging area (ballot + popc),
            // and histograms digit 2 of the threshold bin.
            constexpr int kPerWarpCap = kStageCap / kWarps;
            const int64_t span = (n + kWarps - 1) / kWarps;
            const int64_t w0 = min(n, static_cast<int64_t>(warp) * span);
            const int64_t w1 = min(n, w0 + span);
            uint32_t cntw = 0;
            uint64_t *buf = S.stage + warp * kPerWarpCap;
            for (int64_t base = w0; base < w1; base += 32) {
                const int64_t i = base + lane;
                uint32_t key = 0;
                if (i < w1) key = score_key(__ldcg(&sc[i]));
                const uint32_t dg = key >> kD1Shift;
                const bool keep = i < w1 && dg >= d1;
                const unsigned m = __ballot_sync(0xffffffffu, keep);
                const uint32_t p = cntw + __popc(m & ((1u << lane) - 1u));
                if (keep && p < static_cast<uint32_t>(kPerWarpCap))
                    buf[p] = (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(i);
                smem_hist_add(S.h2, (key >> kD2Shift) & (kD2Bins - 1), i < w1 && dg == d1);
                cntw += __popc(m);
            }
            if (lane == 0) S.wcount[warp] = cntw;
            __syncthreads();
            if (tid == 0) {
                uint32_t tot = 0, of = 0;
                for (int w = 0; w < kWarps; ++w) {
                    of |= S.wcount[w] > static_cast<uint32_t>(kPerWarpCap);
                    S.prefix[w] = tot;
                    tot += S.wcount[w];
                }
                S.nstage = tot;
                S.overflow = of;
            }
            __syncthreads();
            if (!S.overflow) {
                // pack the per-warp runs into one ascending list (in place: each
                // run moves to a lower or equal offset, processed warp by warp)
                for (int w = 1; w < kWarps; ++w) {
                    const uint32_t c = S.wcount[w];
                    uint64_t v0 = 0;
                    for (uint32_t j0 = 0; j0 < c; j0 += blockDim.x) {
                        const uint32_t j = j0 + tid;
                        if (j < c) v0 = S.stage[w * kPerWarpCap + j];
                        __syncthreads();
                        if (j < c && CSA_CHECK(S.prefix[w] + j < kStageCap, P.status))
                            S.stage[S.prefix[w] + j] = v0;
                        __syncthreads();
                    }
                }
            }
        } else {
            // This CTA's slice, already in registers: in index order (warp,
            // q, lane), so a ballot per q and the warps' totals place every
            // kept entry.
            const int64_t b1 = min(n, c0 + P.chunk);
            const unsigned lt = (1u << lane) - 1u;
            uint32_t wt = 0;
#pragma unroll
            for (int q = 0; q < kMaxPerThread; ++q) {
                const bool ok = q * 32 < span && wbase + q * 32 < b1;
                const uint32_t dg = keys[q] >> kD1Shift;
                wt += __popc(__ballot_sync(0xffffffffu, ok && dg >= d1));
                if (ok && dg == d1) atomicAdd(&gh2[(keys[q] >> kD2Shift) & (kD2Bins - 1)], 1u);
            }
            if (lane == 0) S.wcount[warp] = wt;
            __syncthreads();
            uint32_t pos = 0, total = 0;
            for (int w = 0; w < kWarps; ++w) {
                const uint32_t x = S.wcount[w];
                pos += w < warp ? x : 0u;
                total += x;
            }
            uint64_t *slot = P.slots + (static_cast<int64_t>(t) * P.per_tok + blockIdx.x) * P.chunk;
#pragma unroll
            for (int q = 0; q < kMaxPerThread; ++q) {
                const bool keep = q * 32 < span && wbase + q * 32 < b1 && (keys[q] >> kD1Shift) >= d1;
                const unsigned m = __ballot_sync(0xffffffffu, keep);
                if (keep && CSA_CHECK(pos + __popc(m & lt) < static_cast<uint32_t>(P.chunk), P.status))
                    slot[pos + __popc(m & lt)] = (static_cast<uint64_t>(keys[q]) << 32) |
                                                 static_cast<uint32_t>(wbase + q * 32);
                pos += __popc(m);
            }
            if (tid == 0) P.slot_cnt[static_cast<int64_t>(t) * P.per_tok + blockIdx.x] = total;
        }
    }

    // ---- the last CTA of this token resolves
    if (!P.local_hist) {
        __syncthreads();
        if (tid == 0) {
            // release: every thread's slot writes (ordered before this by the
            // barrier) are visible to whoever takes the last ticket; acquire:
            // the last CTA then sees every other CTA's (the barrier below
            // carries it to the other threads)
            uint32_t prev;
            asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                         : "=r"(prev)
                         : "l"(&cnt->ticket)
                         : "memory");
            S.last = (prev == gridDim.x - 1) ? 1u : 0u;
        }
        __syncthreads();
        if (!S.last) return;
    }

    int32_t *out = P.idx_out + static_cast<int64_t>(t) * P.top_k;
    if (!rank) {
        // nothing to rank: none visible, or every visible block fits
        for (int i = tid; i < P.top_k; i += blockDim.x) out[i] = i < static_cast<int>(kk) ? i : -1;
    } else {
        const uint32_t d1 = static_cast<uint32_t>(S.d);
        uint32_t need = kk - S.gt;   // >= 1, all from digit-1 bin d1
        bool d2_found = false;
        bool gathered = false;       // the digit-1/2 bin's keys were collected while staging
        uint32_t pre22 = 0;
        if (!P.local_hist) {
            // One round trip: the slot counts, the digit-2 histogram and the
            // first kSpec entries of every slot, read before their counts are
            // known (entries past a slot's count are dropped below).
            const int pt = P.per_tok;
            const uint64_t *base = P.slots + static_cast<int64_t>(t) * pt * P.chunk;
            const uint32_t c = tid < pt ? __ldcg(&P.slot_cnt[static_cast<int64_t>(t) * pt + tid]) : 0u;
            // thread i holds digit-2 bins hb .. hb+3 (thread 0 the top four)
            const int hb = kD2Bins - 4 * (tid + 1);
            const uint4 h2v = __ldcg(reinterpret_cast<const uint4 *>(gh2 + hb));
            // entries se0, se0 + 1 of slots ssl0 + u * kSpecStride
            constexpr int kSpecStride = kSelThreads / kSpecLanes;
            const int ssl0 = tid / kSpecLanes;
            const uint32_t se0 = (tid % kSpecLanes) * 2;
            ulonglong2 sv[kSpecRounds];
#pragma unroll
            for (int u = 0; u < kSpecRounds; ++u) {
                const int sl = ssl0 + u * kSpecStride;
                sv[u] = sl < pt ? __ldcg(reinterpret_cast<const ulonglong2 *>(
                                      base + static_cast<int64_t>(sl) * P.chunk + se0))
                                : make_ulonglong2(0ull, 0ull);
            }
            *reinterpret_cast<uint4 *>(&S.h2[hb]) = h2v;
            // One scan gives the entry offsets, the offsets of the groups of
            // up to 8 entries the guesses did not cover, and the digit-2
            // counts above each thread's bins.
            const uint32_t spec = tid < pt && tid < kSpecSlots ? min(c, static_cast<uint32_t>(kSpec)) : 0u;
            const uint64_t packed = (static_cast<uint64_t>(c) << kPackA) |
                                    (static_cast<uint64_t>((c - spec + 7) / 8) << kPackB) |
                                    (h2v.x + h2v.y + h2v.z + h2v.w);
            const uint64_t off = block_excl_scan3(packed, S.warp_tmp64, &S.total64);
            if (tid < pt) {
                S.prefix[tid] = static_cast<uint32_t>(off >> kPackA);
                S.gprefix[tid] = static_cast<uint32_t>(off >> kPackB) & kMaskB;
            }
            {
                // digit 2: the bin where the count from the top reaches need
                uint32_t run = static_cast<uint32_t>(off) & kMaskC;
                const uint32_t hv[4] = {h2v.w, h2v.z, h2v.y, h2v.x};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (run < need && run + hv[j] >= need) {
                        S.d = hb + 3 - j;
                        S.gt = run;
                    }
                    run += hv[j];
                }
            }
            if (tid == 0) {
                const uint64_t tot = S.total64;
                S.prefix[pt] = static_cast<uint32_t>(tot >> kPackA);
                S.gprefix[pt] = static_cast<uint32_t>(tot >> kPackB) & kMaskB;
                S.nstage = static_cast<uint32_t>(tot >> kPackA);
                S.overflow = (tot >> kPackA) > static_cast<uint64_t>(kStageCap);
                S.ncand = 0;
            }
            __syncthreads();
            d2_found = true;
            need -= S.gt;
            pre22 = (d1 << kD2Bits) | static_cast<uint32_t>(S.d);
            // The entries sharing digits 1 and 2 with the k-th key number
            // h2[d2]; when they fit one warp their keys are collected as the
            // entries are staged, and one warp finds the k-th key among them.
            gathered = !S.overflow && S.h2[S.d] <= 32u;
            auto collect = [&](uint64_t e) {
                const uint32_t key = static_cast<uint32_t>(e >> 32);
                if ((key >> kD2Shift) == pre22) {
                    const uint32_t at = atomicAdd(&S.ncand, 1u);
                    if (at < 32u) S.cand[at] = key;
                }
            };
            if (!S.overflow) {
#pragma unroll
                for (int u = 0; u < kSpecRounds; ++u) {
                    const int sl = ssl0 + u * kSpecStride;
                    if (sl < pt) {
                        const uint32_t cnt = S.prefix[sl + 1] - S.prefix[sl];
                        uint64_t *dst = S.stage + S.prefix[sl];
                        if (!CSA_CHECK(S.prefix[sl] + cnt <= static_cast<uint32_t>(kStageCap), P.status))
                            continue;
                        if (se0 < cnt) {
                            dst[se0] = sv[u].x;
                            if (gathered) collect(sv[u].x);
                        }
                        if (se0 + 1 < cnt) {
                            dst[se0 + 1] = sv[u].y;
                            if (gathered) collect(sv[u].y);
                        }
                    }
                }
                // the rest: one group per thread, its slot by one search over
                // the group offsets, up to eight independent loads in flight
                const uint32_t ng = S.gprefix[pt];
                for (uint32_t g = tid; g < ng; g += blockDim.x) {
                    int lo = 0, hi = pt;  // the last slot with gprefix[lo] <= g
                    while (hi - lo > 1) {
                        const int mid = (lo + hi) >> 1;
                        if (S.gprefix[mid] <= g) lo = mid;
                        else hi = mid;
                    }
                    const uint32_t cnt = S.prefix[lo + 1] - S.prefix[lo];
                    const uint32_t sp = lo < kSpecSlots ? min(cnt, static_cast<uint32_t>(kSpec)) : 0u;
                    const uint32_t e0 = sp + (g - S.gprefix[lo]) * 8;
                    const uint64_t *src = base + static_cast<int64_t>(lo) * P.chunk + e0;
                    uint64_t *dst = S.stage + S.prefix[lo] + e0;
                    if (!CSA_CHECK(S.prefix[lo] + cnt <= static_cast<uint32_t>(kStageCap), P.status))
                        continue;
                    uint64_t val[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) val[u] = e0 + u < cnt ? __ldcg(src + u) : 0ull;
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (e0 + u < cnt) {
                            dst[u] = val[u];
                            if (gathered) collect(val[u]);
                        }
                }
            }
        }
        __syncthreads();
        // Entries in ascending index order: the staged list, or, when it did
        // not fit, the whole row filtered by digit 1.
        const bool staged = !S.overflow;
        const int64_t m = staged ? static_cast<int64_t>(S.nstage) : n;
        auto entry = [&](int64_t i, uint32_t &key, int64_t &index) {
            if (staged) {
                const uint64_t c = S.stage[i];
                key = static_cast<uint32_t>(c >> 32);
                index = static_cast<int64_t>(c & 0xffffffffu);
            } else {
                key = score_key(__ldcg(&sc[i]));
                index = i;
            }
        };
        // ---- the k-th key tau: the need-th largest of the entries that
        // share digits 1 and 2 with it
        uint32_t tau, eq;
        if (gathered) {
            // one warp, a key per lane: its rank among the collected keys
            if (warp == 0) {
                const uint32_t nc = min(S.ncand, 32u);
                const uint32_t key = static_cast<uint32_t>(lane) < nc ? S.cand[lane] : 0u;
                uint32_t above = 0, same = 0;
                // rolled: this code runs once per launch, and every
                // instruction of it is fetched cold
#pragma unroll 1
                for (uint32_t j = 0; j < nc; ++j) {
                    const uint32_t o = __shfl_sync(0xffffffffu, key, static_cast<int>(j));
                    above += o > key ? 1u : 0u;
                    same += o == key ? 1u : 0u;
                }
                const bool hit = static_cast<uint32_t>(lane) < nc && above < need && need <= above + same;
                const unsigned hm = __ballot_sync(0xffffffffu, hit);
                const int src = hm ? __ffs(hm) - 1 : 0;
                const uint32_t tk = __shfl_sync(0xffffffffu, key, src);
                const uint32_t ta = __shfl_sync(0xffffffffu, above, src);
                const uint32_t ts = __shfl_sync(0xffffffffu, same, src);
                if (lane == 0) {
                    S.tau = tk;
                    S.need3 = need - ta;
                    S.eq3 = ts;
                }
            }
            __syncthreads();
            tau = S.tau;
            need = S.need3;
            eq = S.eq3;
        } else {
            // digit 2 from its histogram (if not found yet), then digit 3
            // over the entries that share digits 1 and 2
            if (!d2_found) {
                find_threshold_digit<kD2Bins>(S.h2, need, S.warp_tmp, &S.d, &S.gt);
                need -= S.gt;
                pre22 = (d1 << kD2Bits) | static_cast<uint32_t>(S.d);
            }
            for (int i = tid; i < kD3Bins; i += blockDim.x) S.h[i] = 0;
            __syncthreads();
            for (int64_t i = tid; i < m; i += blockDim.x) {
                uint32_t key;
                int64_t index;
                entry(i, key, index);
                if ((key >> kD2Shift) == pre22) atomicAdd(&S.h[key & (kD3Bins - 1)], 1u);
            }
            __syncthreads();
            find_threshold_digit<kD3Bins>(S.h, need, S.warp_tmp, &S.d, &S.gt);
            need -= S.gt;
            tau = (pre22 << kD2Shift) | static_cast<uint32_t>(S.d);
            eq = S.h[S.d];
        }
        // ---- ordered compaction: every key above tau, then the `need`
        // lowest-index keys equal to tau; thread-contiguous runs keep order
        const int64_t run = (m + blockDim.x - 1) / blockDim.x;
        const int64_t r0 = min(m, static_cast<int64_t>(tid) * run), r1 = min(m, r0 + run);
        uint32_t tie_before = 0;
        if (need != eq) {
            uint32_t ties = 0;
            for (int64_t i = r0; i < r1; ++i) {
                uint32_t key;
                int64_t index;
                entry(i, key, index);
                ties += key == tau ? 1u : 0u;
            }
            tie_before = block_excl_scan(ties, S.warp_tmp, nullptr);
        }
        const bool all_ties = need == eq;
        uint32_t take_n = 0;
        {
            uint32_t tb = tie_before;
            for (int64_t i = r0; i < r1; ++i) {
                uint32_t key;
                int64_t index;
                entry(i, key, index);
                const bool is_tie = key == tau;
                take_n += key > tau || (is_tie && (all_ties || tb < need)) ? 1u : 0u;
                tb += is_tie ? 1u : 0u;
            }
        }
        uint32_t taken = 0;
        // no barrier since the tie scan: the other buffer
        uint32_t pos = block_excl_scan(take_n, S.warp_tmp + 32, &taken);
        {
            uint32_t tb = tie_before;
            for (int64_t i = r0; i < r1; ++i) {
                uint32_t key;
                int64_t index;
                entry(i, key, index);
                const bool is_tie = key == tau;
                if (key > tau || (is_tie && (all_ties || tb < need))) {
                    if (pos < kk) out[pos] = static_cast<int32_t>(index);
                    ++pos;
                }
                tb += is_tie ? 1u : 0u;
            }
        }
        for (int i = kk + tid; i < P.top_k; i += blockDim.x) out[i] = -1;
        if (taken != kk && tid == 0) raise_status(P.status, CSA_DEV_BAD_INDEX);
    }
    if (tid == 0) P.nsel_out[t] = static_cast<int32_t>(kk);
    // ---- leave the per-token state zeroed for the next call (in one-CTA mode
    // the histograms were built in shared memory, but the state is cleared all
    // the same: it keeps the contract simple)
    for (int i = tid; i < kD1Bins + kD2Bins; i += blockDim.x) gh[i] = 0;
    if (tid == 0) cnt->ticket = 0;
}

void topk_grid(int64_t T, int64_t max_comp_rows, int32_t *chunk_out, int32_t *per_tok_out) {
    const int64_t maxn = max_comp_rows > 0 ? max_comp_rows : 1;
    // CTAs per token: about kTargetCtas in total, each with 1024 .. 4096 scores
    const int64_t Tp = T > 0 ? T : 1;
    const int64_t want = (kTargetCtas + Tp - 1) / Tp;
    int64_t chunk = (maxn + want - 1) / want;
    chunk = ((chunk + 1023) / 1024) * 1024;
    if (chunk < 1024) chunk = 1024;
    int64_t per_tok = (maxn + chunk - 1) / chunk;
    if (chunk > kMaxFilterChunk || per_tok > kMaxPerTok) per_tok = 1;  // one CTA per token
    if (per_tok == 1) chunk = maxn;
    *chunk_out = static_cast<int32_t>(chunk);
    *per_tok_out = static_cast<int32_t>(per_tok);
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
    P.slots = ws.slots;
    P.slot_cnt = ws.slot_cnt;
    P.idx_out = idx;
    P.nsel_out = n_sel;
    P.status = status;
    topk_grid(T, L.max_comp_rows, &P.chunk, &P.per_tok);
    if (!P.slots || !P.slot_cnt) {  // no filter slots: one CTA owns each row
        P.per_tok = 1;
        P.chunk = static_cast<int32_t>(L.max_comp_rows > 0 ? L.max_comp_rows : 1);
    }
    P.local_hist = P.per_tok == 1 ? 1 : 0;
    cudaError_t e;
    if (!hist_ready && !P.local_hist) {
        e = set_kernel_smem(score_hist_kernel, 0);
        if (e != cudaSuccess) return e;
        e = launch_pdl(score_hist_kernel, dim3(static_cast<unsigned>(P.per_tok), T), dim3(256), 0,
                       lc.stream, P);
        if (e != cudaSuccess) return e;
    }
    const size_t smem = sizeof(SelectSmem) + 16;
    e = set_kernel_smem(select_kernel, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(select_kernel, dim3(static_cast<unsigned>(P.per_tok), T), dim3(kSelThreads),
                      smem, lc.stream, P);
}

}  // namespace csa
