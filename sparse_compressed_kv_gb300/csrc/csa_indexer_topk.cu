// csa_indexer_topk.cu -- the decode indexer (one query token per key tile),
// optionally with the top-k selection folded in.
//
//   score[t, s] = sum_h w[t,h] * ReLU(q^I[t,h,:] . K^I[s,:])      (indexer)
//   top_k blocks by (score descending, block index ascending)     (selection)
//
// ("ARCHITECTURE & MEMORY AUDIT -- Post-probe rewrite", F1 and F3: one
// 128-wide key per compressed block shared by the 64 indexer heads; the
// top_k best blocks, tk = min(top_k, n_comp).)
//
// Work split.  Every token's visible blocks are cut into units of kBoxRows
// keys; the units of all tokens, token after token, are divided into one
// contiguous range per CTA (equal to within one unit).  A CTA walks its range
// in key tiles of up to 128 keys, each tile loaded by TMA as 32-row boxes, and
// runs the contraction swap-AB on the tensor cores as the prefill indexer
// does: A = keys (M = 128), B = the token's 64 query heads (N = 64), f32 in
// TMEM, ReLU . w . sum_h in the epilogue, one key per TMEM lane.
//
// Folded selection.  The part of a token's range one CTA owns is a segment.
// The epilogue keeps the segment's order-preserving score keys in shared
// memory and histograms their top 11 bits.  When the segment ends it finds the
// digit d where the count from the top reaches k' (the segment's share of
// top_k plus 16), writes every entry whose digit is >= d, in
// block order, to the segment's candidate slot with the bound B = d << 21 (the
// entries it left out all have keys below B), and adds those entries' digits
// to the token's digit-1 histogram.  The last CTA to finish a segment of the
// token (atomic ticket) resolves it: with M the largest bound of the token's
// segments, every key >= M of the token is among the candidates and counted
// by the histogram, so when at least k of them are >= M, the k best
// candidates are the k best blocks, exactly.  Otherwise (or when a slot
// overflowed) that CTA selects from the token's whole score row instead,
// which the epilogue wrote to global memory.  Either way the result is a pure
// function of the score bits, equal to csa_topk's on the same scores.
//
// Warp roles: 0 TMA producer, 1 TMEM allocator + tcgen05.mma issuer, 2..5
// epilogue (one TMEM lane quarter each), 6..7 the candidate-slot table while
// the first tiles stream in; all eight finish the CTA's last segment and run
// the resolve.  No CTA waits for another: the hand-off is the ticket.  With
// FP4 keys the block has two more warps: 8, 9 and 6, 7 expand the key tiles
// into tensor memory (lane quarters 0..3), 6..7 also convert the queries to
// f16, and 8..9 leave when the keys are done.
//
// The selection code runs once per launch, in one CTA: it is written as
// short dependency chains (thread-contiguous runs of independent loads, one
// block scan per ordered output), since each step's latency is exposed.
#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {
namespace {

constexpr int kWarps = 8;                      // the warps that select (0..7)
constexpr int kThreads = 32 * kWarps;
constexpr int kThreadsFp4 = kThreads + 64;     // FP4: warps 8, 9 expand key quarters 0, 1
constexpr int kEpiThreads = 128;               // warps 2..5
constexpr int kBarEpi = 1;                     // named barrier of the epilogue warps
constexpr int kBarSlots = 2;                   // epilogue + warps 6..7: slot table ready
constexpr int kBarAux = 3;                     // warps 6..7
constexpr int kBarMain = 5;                    // warps 0..7 (the selection's CTA-wide barrier)
constexpr int kStages = 4;
constexpr int kAcc = 4;
constexpr int kN = 64;                         // MMA N: one token's indexer heads
constexpr int kTileUnits = kTileKeys / kBoxRows;   // 4 units per 128-key tile
constexpr int kHalfBytes = kTileKeys * 128;    // 16 KiB: 64 columns of a 128-key tile
constexpr int kABytes = 2 * kHalfBytes;        // 32 KiB per stage
constexpr int kBoxBytes = kBoxRows * 128;      // 4 KiB: one 32-row box of one half
constexpr int kBBytes = 2 * kN * 128;          // 16 KiB: one token's queries
constexpr int kStageEntries = kStages * kABytes / 8;  // resolver staging in the ring
static_assert(kStageEntries < 65536, "the resolve packs two entry counts in one word");
// FP4 keys (80-byte MXFP4 rows): a ring of raw code tiles in shared memory.
// Four warps, one per TMEM lane quarter (8, 9, 6, 7), expand each tile into
// f16 keys in tensor memory, where the MMA reads its A operand; no f16 tile
// passes through shared memory.  The raw
// ring and a second query buffer (the next token's, loaded ahead) fit in the
// bf16 ring's 128 KiB, which the resolver stages in afterwards.
constexpr int kFRow = 80;
constexpr int kFBytes = kTileKeys * kFRow;     // 10 KiB: one raw tile
constexpr int kFStages = 8;
constexpr int kATm = 4;                        // f16 key tiles in tensor memory
constexpr int kAColsF = kIHD / 2;              // 64 columns: one f16 key per lane
constexpr int kScaleStages = kATm + kAcc;      // per-key scales, read by the epilogue
constexpr int kConvThreads = 64;               // warps 6, 7: the queries' conversion
constexpr int kExpThreads = 128;               // warps 8, 9, 6, 7: the keys' expansion
constexpr int kBarConv = 4;                    // named barrier of the converter warps
constexpr uint32_t kTmemColsF = 512;           // accumulators + f16 key tiles
static_assert(kAcc * kN + kATm * kAColsF <= static_cast<int>(kTmemColsF), "FP4 tensor memory");
static_assert(kFStages * kFBytes + kBBytes <= kStages * kABytes, "FP4 rings");
static_assert(kFStages * kFBytes % 1024 == 0, "second query buffer: 1024-byte aligned");
constexpr int kWarmKeys = 4 * kTileKeys;       // keys a CTA warms L2 with before its layout

struct DecParams {
    csa_layout_t L;
    int32_t ratio;
    int32_t top_k;
    const float *w_idx;
    const uint8_t *k_idx;  // the key rows (for the L2 warm-up)
    float *scores;
    int64_t ld;
    int32_t *status;
    FusedTopk f;           // fused selection (f.idx == nullptr: scores only)
};

struct DecSmem {
    uint32_t keys[kSegKeysMax];        // this CTA's score keys; the resolver's histograms
    uint32_t hist[kD1Bins];            // digit-1 histogram of the current segment
    int64_t U[kDecMaxTokens + 1];      // first unit of each token (prefix over tokens)
    int64_t off[kDecMaxTokens];        // first cache row of each token's sequence
    int32_t nvis[kDecMaxTokens];
    int32_t sb[kDecMaxTokens + 1];     // first candidate slot of each token
    int32_t resolve[kDecMaxTokens];    // tokens whose last segment this CTA finished
    int32_t nresolve;
    uint32_t gbuf[8], gbuf2[8];        // group scans
    uint32_t bscan[8], bt[8];          // block scans of the resolve
    uint32_t red_or, red_max;
    int32_t fd;                        // digit found by the current search
    uint32_t fgt;                      // count above it
    uint64_t bars[40];                 // pipeline barriers (layout per key format)
    uint64_t sfull[kScaleStages];      // FP4: a tile's key scales are written
    float fscale[kScaleStages][kTileKeys];   // FP4: 2^(E_max - 127 + s_q) per key
    float qmax[2];                     // FP4: the converter warps' max |q|
    int32_t qsi[2];                    // FP4: s_q of the token in each query buffer
    alignas(16) float wc[4][kNIH];     // each epilogue warp's copy of its token's weights
    uint64_t rbar;                     // the resolver's staging copies
    uint32_t rphase;
    uint32_t tmem_holder;
};

__device__ __forceinline__ uint32_t lt_mask() { return (1u << lane_id()) - 1u; }

// Shared-memory histogram increment, aggregated over the lanes of a warp that
// hit the same bin (for rows where many scores tie).  Every lane must call it.
__device__ __forceinline__ void hist_add(uint32_t *h, uint32_t bin, bool active) {
    const unsigned act = __ballot_sync(0xffffffffu, active);
    if (!active) return;
    const unsigned peers = __match_any_sync(act, bin);
    if (static_cast<int>(lane_id()) == __ffs(peers) - 1) atomicAdd(&h[bin], __popc(peers));
}

// Barrier of warps 0..7 (with FP4 keys the block has two more warps, which
// leave after the key loop).
__device__ __forceinline__ void main_sync() { named_bar_sync(kBarMain, kThreads); }

__device__ __forceinline__ void group_sync(int bar, int nthreads) {
    if (bar == 0) main_sync();
    else named_bar_sync(bar, nthreads);
}

// Exclusive scan of one value per thread over a group of NW warps (group
// warp gw) meeting at barrier `bar`; *total gets the group's sum.  Ends with
// the reads of buf: a second scan must use another buffer or follow a barrier.
template <int NW>
__device__ __forceinline__ uint32_t group_scan(uint32_t v, uint32_t *buf, int gw, int bar,
                                               uint32_t *total) {
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (static_cast<int>(lane_id()) >= o) incl += y;
    }
    if (lane_id() == 31) buf[gw] = incl;
    group_sync(bar, NW * 32);
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const uint32_t x = buf[w];
        before += w < gw ? x : 0u;
        all += x;
    }
    if (total) *total = all;
    return before + incl - v;
}

// Thread i of a group of NW warps holds the PER bins just below NB - i * PER
// of a histogram (thread 0 the top ones) in v, starting at bin hb, and the
// group finds the digit d with count(> d) < k <= count(>= d): into S.fd and
// S.fgt; S.fd = -1 when the histogram holds fewer than k.  Ends with a barrier.
template <int NW, int PER>
__device__ __forceinline__ void group_find_digit(const uint32_t (&v)[PER], int hb, uint32_t k,
                                                 uint32_t *buf, int gw, int bar, DecSmem &S) {
    uint32_t local = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) local += v[j];
    if (gw == 0 && lane_id() == 0) S.fd = -1;
    uint32_t run = group_scan<NW>(local, buf, gw, bar, nullptr);   // count in bins above
#pragma unroll
    for (int j = PER - 1; j >= 0; --j) {
        if (run < k && run + v[j] >= k) {
            S.fd = hb + j;
            S.fgt = run;
        }
        run += v[j];
    }
    group_sync(bar, NW * 32);
}

template <int PER>
__device__ __forceinline__ void load_bins(const uint32_t *h, int hb, uint32_t (&v)[PER]) {
#pragma unroll
    for (int j = 0; j < PER; j += 4) {
        const uint4 q = *reinterpret_cast<const uint4 *>(h + hb + j);
        v[j] = q.x;
        v[j + 1] = q.y;
        v[j + 2] = q.z;
        v[j + 3] = q.w;
    }
}

// Unit u's CTA under the partition A_c = floor(K32 * c / G) (0 <= u < K32).
__device__ __forceinline__ int cta_of(int64_t u, int64_t K32, int G) {
    return static_cast<int>(((u + 1) * G - 1) / K32);
}

// One key tile of a CTA's range: token t, blocks s0 .. s0 + 32 * nunits - 1
// of it (some past n_vis at the token's end), `last`: the tile ends the
// CTA's part of the token (a segment).
struct Tile {
    int t;
    int nunits;
    bool last;
    int64_t u;    // first unit of the tile
    int64_t s0;   // first block of the tile
};

__device__ __forceinline__ bool next_tile(const int64_t *U, int64_t ub, int &t, int64_t &u,
                                          Tile &tl) {
    if (u >= ub) return false;
    while (U[t + 1] <= u) ++t;   // tokens that end at or before u (empty ones included)
    const int64_t tend = U[t + 1];
    int64_t e = u + kTileUnits;
    e = e < tend ? e : tend;
    e = e < ub ? e : ub;
    tl.t = t;
    tl.u = u;
    tl.s0 = (u - U[t]) * kBoxRows;
    tl.nunits = static_cast<int>(e - u);
    tl.last = e == tend || e == ub;
    u = e;
    return true;
}

// The token whose units contain u (U[t] <= u < U[t+1]).
__device__ __forceinline__ int token_of(const int64_t *U, int T, int64_t u) {
    int lo = 0, hi = T;   // U[lo] <= u < U[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (U[mid] <= u) lo = mid;
        else hi = mid;
    }
    return lo;
}

// Exclusive prefix over x[1..n] in place, x[0] = 0 (one warp).
template <typename V>
__device__ __forceinline__ void warp_prefix(V *x, int n) {
    const int lane = static_cast<int>(lane_id());
    const int seg = (n + 31) >> 5;
    const int beg = min(n, lane * seg), end = min(n, beg + seg);
    V sum = 0;
    for (int i = beg; i < end; ++i) {
        sum += x[i + 1];
        x[i + 1] = sum;
    }
    V incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const V y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const V excl = incl - sum;
    for (int i = beg; i < end; ++i) x[i + 1] += excl;
    if (lane == 0) x[0] = 0;
}

// n items split into thread-contiguous runs, the run length made odd so that
// lanes reading their runs in step hit distinct banks.
__device__ __forceinline__ int odd_run(int n, int nthreads) {
    return ((n + nthreads - 1) / nthreads) | 1;
}

// The end of the segment [seg_u0, su1) (units) of token tk in the CTA that
// owns units [ua, ...): pick the threshold digit, hand the candidates on,
// take the ticket.  A group of NW warps (thread gt of it) meeting at `bar`.
template <int NW>
__device__ __forceinline__ void finalize_segment(const DecParams &P, DecSmem &S, int tk,
                                                 int64_t seg_u0, int64_t su1, int64_t ua,
                                                 int64_t K32, int Ge, int c, int gt, int bar) {
    constexpr int NT = NW * 32;
    constexpr int PER = kD1Bins / NT;
    const int gw = gt >> 5;
    group_sync(bar, NT);   // every key of the segment is in S.keys and S.hist
    const int64_t nv = S.nvis[tk];
    const int64_t s_begin = (seg_u0 - S.U[tk]) * kBoxRows;
    int64_t s_end = (su1 - S.U[tk]) * kBoxRows;
    s_end = s_end < nv ? s_end : nv;
    const int64_t lo0 = (seg_u0 - ua) * kBoxRows;
    int64_t len = s_end - s_begin;
    const bool lost = lo0 + len > kSegKeysMax;   // keys beyond the buffer (the host plan excludes it)
    if (lost) len = kSegKeysMax - lo0 > 0 ? kSegKeysMax - lo0 : 0;
    // k': the segment's share of top_k plus a margin of 16 (the digit's
    // granularity, about a fifth of the score's magnitude, gives the proof
    // its slack: with 1.25 x the share the largest bound was the same)
    int64_t kq = (static_cast<int64_t>(P.top_k) * len + nv - 1) / nv + 16;
    kq = kq < P.top_k ? kq : P.top_k;
    kq = kq < len ? kq : len;
    const int hb = kD1Bins - PER * (gt + 1);
    uint32_t hv[PER];
    load_bins<PER>(S.hist, hb, hv);
    uint32_t d1 = 0;
    if (kq < len) {
        group_find_digit<NW, PER>(hv, hb, static_cast<uint32_t>(kq), S.gbuf, gw, bar, S);
        d1 = static_cast<uint32_t>(S.fd);
    }
    // the digits of the entries handed on, into the token's digit-1
    // histogram: at and above the largest bound of the token's segments it
    // counts every key of the token
    uint32_t *gh = P.f.state + static_cast<int64_t>(tk) * kStateWords;
#pragma unroll
    for (int j = 0; j < PER; ++j)
        if (hv[j] && static_cast<uint32_t>(hb + j) >= d1) atomicAdd(gh + hb + j, hv[j]);
    // every entry with digit >= d1, in block order, to the slot
    int slot = S.sb[tk] + (c - cta_of(S.U[tk], K32, Ge));
    if (!CSA_CHECK(slot >= 0 && slot < P.f.slots, P.status)) slot = 0;   // (checked builds only)
    uint64_t *dst = P.f.cand + static_cast<int64_t>(slot) * P.f.cap;
    const int R = odd_run(static_cast<int>(len), NT);
    const int r0 = min(static_cast<int>(len), gt * R);
    const int r1 = min(static_cast<int>(len), r0 + R);
    const uint32_t *kr = S.keys + lo0;
    uint32_t cnt = 0;
#pragma unroll 4
    for (int i = r0; i < r1; ++i) cnt += (kr[i] >> kD1Shift) >= d1 ? 1u : 0u;
    uint32_t total = 0;
    uint32_t pos = group_scan<NW>(cnt, S.gbuf2, gw, bar, &total);
#pragma unroll 4
    for (int i = r0; i < r1; ++i) {
        const uint32_t k2 = kr[i];
        if ((k2 >> kD1Shift) >= d1) {
            if (pos < static_cast<uint32_t>(P.f.cap))
                dst[pos] = (static_cast<uint64_t>(k2) << 32) | static_cast<uint32_t>(s_begin + i);
            ++pos;
        }
    }
    if (gt == 0) {
        const bool ovf = lost || total > static_cast<uint32_t>(P.f.cap);
        P.f.meta[slot] = make_uint4(ovf ? 0u : total, kq < len ? d1 << kD1Shift : 0u, ovf ? 1u : 0u,
                                    static_cast<uint32_t>(len));
    }
#pragma unroll
    for (int j = 0; j < PER; j += 4)
        *reinterpret_cast<uint4 *>(S.hist + hb + j) = make_uint4(0, 0, 0, 0);
    // the barrier orders every thread's slot, header, score and histogram
    // writes before the ticket's release
    group_sync(bar, NT);
    if (gt == 0) {
        // release: this segment's data; acquire (for the last): every other's
        uint32_t prev;
        uint32_t *tkt = &reinterpret_cast<TokCounters *>(P.f.state + static_cast<int64_t>(tk) * kStateWords +
                                                         kD1Bins + kD2Bins)->ticket;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(tkt) : "memory");
        if (prev + 1 == static_cast<uint32_t>(S.sb[tk + 1] - S.sb[tk]) &&
            CSA_CHECK(S.nresolve < kDecMaxTokens, P.status))
            S.resolve[S.nresolve++] = tk;
    }
}

// An entry of the resolver's staging area that holds no candidate (the pad
// that keeps each slot's copy 16-byte aligned); it reads as key 0, below the
// key of every finite score, so it is never selected.
constexpr uint64_t kNoEntry = 0xffffffffull;

// f(e) for each staged entry of a thread's run [r0, r1), the entries loaded
// eight at a time ahead of the work on them: shared-memory atomics in that
// work would otherwise hold each following load behind them.
template <typename F>
__device__ __forceinline__ void for_run(const uint64_t *stage, int r0, int r1, F &&f) {
#pragma unroll 1
    for (int b = r0; b < r1; b += 8) {
        uint64_t e[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) e[k] = b + k < r1 ? stage[b + k] : 0ull;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (b + k < r1) f(e[k]);
    }
}

// The exact top-k of token t, from the candidates of its segments or, when
// they do not prove the result, from its whole score row.  Whole CTA.
__device__ __forceinline__ void resolve_token(const DecParams &P, DecSmem &S, uint64_t *stage,
                                              int t) {
    const int tid = threadIdx.x;
    const int lane = static_cast<int>(lane_id()), warp = tid >> 5;
    const uint32_t lt = lt_mask();
    const int64_t nv = S.nvis[t];
    const uint32_t kk = static_cast<uint32_t>(min(static_cast<int64_t>(P.top_k), nv));
    const int base = S.sb[t], nseg = S.sb[t + 1] - base;
    uint32_t *h = S.keys;             // histograms of the digits
    uint32_t *gh = P.f.state + static_cast<int64_t>(t) * kStateWords;   // digit 1, global
    if (tid == 0) {
        S.red_or = 0;
        S.red_max = 0;
    }
    // one round trip: the slot headers and the token's digit-1 histogram
    // (thread i: bins 2048 - 8(i+1) .. 2048 - 8i - 1, zeroed behind it)
    uint4 m = make_uint4(0, 0, 0, 0);
    if (tid < nseg) m = __ldcg(P.f.meta + base + tid);
    const int hb = kD1Bins - 8 * (tid + 1);
    const uint4 ga = __ldcg(reinterpret_cast<const uint4 *>(gh + hb));
    const uint4 gb = __ldcg(reinterpret_cast<const uint4 *>(gh + hb + 4));
    *reinterpret_cast<uint4 *>(gh + hb) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4 *>(gh + hb + 4) = make_uint4(0, 0, 0, 0);
#pragma unroll 1
    for (int i = tid; i < kD2Bins + kD3Bins; i += kThreads) h[i] = 0;
    main_sync();
    if (tid < nseg) {
        if (m.z) atomicOr(&S.red_or, 1u);
        atomicMax(&S.red_max, m.y);
    }
    // slot regions in the staging area start at even entries (16-byte copies)
    uint32_t M = 0;
    const uint32_t soff = group_scan<kWarps>((m.x + 1u) & ~1u, S.bscan, warp, 0, &M);
    main_sync();
    const uint32_t maxD = S.red_max >> kD1Shift;   // every key of the token in bins >= maxD is here
    bool from_row = S.red_or != 0 || M > static_cast<uint32_t>(kStageEntries);
    int32_t *out = P.f.idx + static_cast<int64_t>(t) * P.top_k;
    uint32_t total = kk;
    if (!from_row) {
        // stage the candidates: one bulk copy per slot, all in flight at once
        const uint32_t ph = S.rphase;
        if (tid == 0) mbar_arrive_expect_tx(&S.rbar, M * 8u);
        if (tid < nseg && m.x > 0) {
            const uint64_t *src = P.f.cand + static_cast<int64_t>(base + tid) * P.f.cap;
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_addr(stage + soff)),
                "l"(src), "r"(((m.x + 1u) & ~1u) * 8u), "r"(smem_addr(&S.rbar))
                : "memory");
        }
        // digit 1 from the token's histogram, counting the bins >= maxD only
        uint32_t v[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (static_cast<uint32_t>(hb + j) < maxD) v[j] = 0;
        group_find_digit<kWarps, 8>(v, hb, kk, S.bt, warp, 0, S);
        mbar_wait(&S.rbar, ph, P.status);
        // an odd slot's copy brought one stale entry past its end
        if (tid < nseg && (m.x & 1u) && CSA_CHECK(soff + m.x < kStageEntries, P.status))
            stage[soff + m.x] = kNoEntry;
        if (tid == 0) S.rphase = ph ^ 1u;
        main_sync();
        from_row = S.fd < 0;   // fewer than k keys >= the bound: it proves nothing
    }
    if (!from_row) {
        // thread tid owns the run [tid R, tid R + R) of the staged entries
        // (block order): independent loads, plain shared atomics (the digit-2
        // bins of one digit-1 bin are spread), one block scan per output
        uint32_t *h2 = h, *h3 = h + kD2Bins;
        const uint32_t d1 = static_cast<uint32_t>(S.fd);
        uint32_t need = kk - S.fgt;
        const int R = odd_run(static_cast<int>(M), kThreads);
        const int r0 = min(static_cast<int>(M), tid * R), r1 = min(static_cast<int>(M), r0 + R);
        for_run(stage, r0, r1, [&](uint64_t e) {
            const uint32_t key = static_cast<uint32_t>(e >> 32);
            if ((key >> kD1Shift) == d1) atomicAdd(&h2[(key >> kD2Shift) & (kD2Bins - 1)], 1u);
        });
        main_sync();
        {
            uint32_t v[8];
            load_bins<8>(h2, kD2Bins - 8 * (tid + 1), v);
            group_find_digit<kWarps, 8>(v, kD2Bins - 8 * (tid + 1), need, S.bt, warp, 0, S);
        }
        const uint32_t pre = (d1 << kD2Bits) | static_cast<uint32_t>(S.fd);
        need -= S.fgt;
        for_run(stage, r0, r1, [&](uint64_t e) {
            const uint32_t key = static_cast<uint32_t>(e >> 32);
            if ((key >> kD2Shift) == pre) atomicAdd(&h3[key & (kD3Bins - 1)], 1u);
        });
        main_sync();
        {
            uint32_t v[4];
            load_bins<4>(h3, kD3Bins - 4 * (tid + 1), v);
            group_find_digit<kWarps, 4>(v, kD3Bins - 4 * (tid + 1), need, S.bt, warp, 0, S);
        }
        const uint32_t tau = (pre << kD2Shift) | static_cast<uint32_t>(S.fd);
        need -= S.fgt;
        const bool all_ties = need == h3[S.fd];
        // one pass and one block scan: the entries above tau and the ties at
        // tau before this thread's run (packed, each count below 2^16); the
        // ties are taken in block order, the first `need` of them
        uint32_t ties = 0, gt = 0;
#pragma unroll 4
        for (int i = r0; i < r1; ++i) {
            const uint32_t key = static_cast<uint32_t>(stage[i] >> 32);
            ties += key == tau ? 1u : 0u;
            gt += key > tau ? 1u : 0u;
        }
        uint32_t both = 0;
        const uint32_t before = group_scan<kWarps>(gt | (ties << 16), S.bt, warp, 0, &both);
        const uint32_t tb = before >> 16;
        uint32_t pos = (before & 0xffffu) + (all_ties ? tb : min(tb, need));
        total = (both & 0xffffu) + (all_ties ? (both >> 16) : min(both >> 16, need));
        uint32_t r = tb;
#pragma unroll 4
        for (int i = r0; i < r1; ++i) {
            const uint64_t e = stage[i];
            const uint32_t key = static_cast<uint32_t>(e >> 32);
            const bool tie = key == tau;
            if (key > tau || (tie && (all_ties || r < need))) {
                if (pos < kk) out[pos] = static_cast<int32_t>(e & 0xffffffffu);
                ++pos;
            }
            r += tie ? 1u : 0u;
        }
    } else {
        // ---- the whole score row (every visible score of the token was
        // written by the epilogues before their tickets): the digits by
        // warp-strided passes, then an ordered emit by warp spans
        const float *sc = P.scores + static_cast<int64_t>(t) * P.ld;
        uint32_t need = kk, prefix = 0, eq = 0;
#pragma unroll 1
        for (int lvl = 0; lvl < 3; ++lvl) {
            const int nb = lvl == 2 ? kD3Bins : kD1Bins;
            const int shift = lvl == 0 ? kD1Shift : (lvl == 1 ? kD2Shift : 0);
            main_sync();
#pragma unroll 1
            for (int i = tid; i < kD1Bins; i += kThreads) h[i] = 0;
            main_sync();
#pragma unroll 1
            for (int64_t b = 0; b < nv; b += kThreads) {
                const int64_t i = b + tid;
                const uint32_t key = i < nv ? score_key(__ldcg(sc + i)) : 0u;
                const bool in = lvl == 0 || (key >> (lvl == 1 ? kD1Shift : kD2Shift)) == prefix;
                hist_add(h, (key >> shift) & static_cast<uint32_t>(nb - 1), i < nv && in);
            }
            main_sync();
            if (lvl == 2) {
                uint32_t v[4];
                load_bins<4>(h, kD3Bins - 4 * (tid + 1), v);
                group_find_digit<kWarps, 4>(v, kD3Bins - 4 * (tid + 1), need, S.bt, warp, 0, S);
            } else {
                uint32_t v[8];
                load_bins<8>(h, kD1Bins - 8 * (tid + 1), v);
                group_find_digit<kWarps, 8>(v, kD1Bins - 8 * (tid + 1), need, S.bt, warp, 0, S);
            }
            prefix = (prefix << (lvl == 2 ? 10 : 11)) | static_cast<uint32_t>(S.fd);
            need -= S.fgt;
            if (lvl == 2) eq = h[S.fd];
        }
        const uint32_t tau = prefix;
        const bool all_ties = need == eq;
        const int64_t W = ((nv + kWarps * 32 - 1) / (kWarps * 32)) * 32;
        const int64_t w0 = min(nv, warp * W), w1 = min(nv, w0 + W);
        uint32_t tb = 0, before = 0;
#pragma unroll 1
        for (int pass = all_ties ? 1 : 0; pass < 3; ++pass) {
            uint32_t rt = tb, cnt = 0;
#pragma unroll 1
            for (int64_t b = w0; b < w1; b += 32) {
                const int64_t i = b + lane;
                const uint32_t key = i < w1 ? score_key(__ldcg(sc + i)) : 0u;
                const bool tie = i < w1 && key == tau;
                const uint32_t tm = __ballot_sync(0xffffffffu, tie);
                const bool selb = i < w1 && (key > tau || (tie && (all_ties || rt + __popc(tm & lt) < need)));
                const uint32_t sm = __ballot_sync(0xffffffffu, pass == 0 ? tie : selb);
                if (pass == 2 && selb) {
                    const uint32_t p = before + cnt + __popc(sm & lt);
                    if (p < kk) out[p] = static_cast<int32_t>(i);
                }
                cnt += __popc(sm);
                rt += __popc(tm);
            }
            if (pass < 2) {
                if (lane == 0) S.bscan[warp] = cnt;
                main_sync();
                uint32_t x = 0, all = 0;
#pragma unroll 1
                for (int w = 0; w < kWarps; ++w) {
                    const uint32_t y = S.bscan[w];
                    x += w < warp ? y : 0u;
                    all += y;
                }
                if (pass == 0) tb = x;
                else {
                    before = x;
                    total = all;
                }
                main_sync();
            }
        }
    }
#pragma unroll 1
    for (int i = static_cast<int>(kk) + tid; i < P.top_k; i += kThreads) out[i] = -1;
    if (tid == 0) {
        P.f.n_sel[t] = static_cast<int32_t>(kk);
        if (total != kk) raise_status(P.status, CSA_DEV_BAD_INDEX);
        // the token's ticket back to zero for the next call
        reinterpret_cast<TokCounters *>(P.f.state + static_cast<int64_t>(t) * kStateWords + kD1Bins +
                                        kD2Bins)->ticket = 0;
    }
    main_sync();
}

// f16 x2 from two e2m1 codes (the low nibble in the low half), exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte_in_low_bits) {
    uint32_t d;
    asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }"
        : "=r"(d)
        : "r"(byte_in_low_bits));
    return d;
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Instruction descriptor: kind::f16 with f16 A/B (formats 0), f32 accumulator,
// both operands K-major, shape M x N.
template <int M, int N>
__device__ __forceinline__ constexpr uint32_t idesc_f16_f32() {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// One MXFP4 key row -> TMEM lane `taddr` of an f16 key tile: elements 2j and
// 2j + 1 in column j, the e2m1 codes of block b times 2^(E_b - E_max), exact
// (an e2m1 value times a power of two >= 2^-24 is an f16 value; blocks more
// than 24 binades below the key's largest are dropped: below f16's range, and
// below 2^-24 of the key's largest term).  Returns E_max.  Warp-collective:
// a lane with no key (valid false) stores zeros.
__device__ __forceinline__ int fp4_expand_row_tmem(const uint8_t *row, bool valid, uint32_t taddr) {
    uint32_t cw32[16];
    uint32_t ev = 0;
    if (valid) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            const uint4 v = *reinterpret_cast<const uint4 *>(row + 16 * q4);
            cw32[4 * q4 + 0] = v.x;
            cw32[4 * q4 + 1] = v.y;
            cw32[4 * q4 + 2] = v.z;
            cw32[4 * q4 + 3] = v.w;
        }
        ev = *reinterpret_cast<const uint32_t *>(row + 64);
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) cw32[j] = 0u;
    }
    int eb[4];
    int emax = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        eb[b] = static_cast<int>((ev >> (8 * b)) & 0xFFu);
        emax = eb[b] > emax ? eb[b] : emax;
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        // block b = words 4b .. 4b + 3 = columns 16b .. 16b + 15; 2^-dlt as an
        // f16 pair: normal down to 2^-14, subnormal to 2^-24
        const int dlt = emax - eb[b];
        const uint32_t hb = dlt <= 14 ? static_cast<uint32_t>(15 - dlt) << 10
                                      : (dlt <= 24 ? 1u << (24 - dlt) : 0u);
        const uint32_t sc = hb | (hb << 16);
        uint32_t o[16];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const uint32_t wd = cw32[4 * b + jj];   // elements 8j .. 8j + 7, j = 4b + jj
            o[4 * jj + 0] = hmul2_bits(e2m1x2_to_f16x2(wd), sc);
            o[4 * jj + 1] = hmul2_bits(e2m1x2_to_f16x2(wd >> 8), sc);
            o[4 * jj + 2] = hmul2_bits(e2m1x2_to_f16x2(wd >> 16), sc);
            o[4 * jj + 3] = hmul2_bits(e2m1x2_to_f16x2(wd >> 24), sc);
        }
        tmem_st16(taddr + 16u * b, o);
    }
    return emax;
}

// 2^(emax - 127 + qs) as an f32, built from its bits: normal, subnormal,
// zero below f32's range, infinity above it (where the product overflows)
__device__ __forceinline__ float fp4_key_scale(int emax, int qs) {
    const int e = emax - 127 + qs;
    if (e > 127) return __int_as_float(0x7F800000);
    if (e >= -126) return __int_as_float((e + 127) << 23);
    if (e >= -149) return __int_as_float(1 << (e + 149));
    return 0.f;
}

// The barriers of the FP4 key pipeline.
struct Fp4Bars {
    uint64_t *f_full, *f_empty;    // raw tile landed / read by the four expander warps
    uint64_t *a_full, *a_empty;    // f16 tile in TMEM / the MMA is done with it
    uint64_t *sfull;               // the tile's key scales are written
};

// One expander warp's part of FP4 key tile `it`: lane l expands key
// r = 32 * (warp's quarter) + l into TMEM lane r of key stage it % kATm and
// writes the key's scale 2^(E_max - 127 + s_q) for the epilogue.
__device__ __forceinline__ void fp4_expand_quarter(DecSmem &S, const uint8_t *sF, const Fp4Bars &B,
                                                   uint32_t tmem_base, int quarter, const Tile &tl,
                                                   int64_t row0, int64_t total_rows, int it, int qs,
                                                   bool &dead, int32_t *status) {
    const int lane = static_cast<int>(lane_id());
    const int fs = it % kFStages, as = it % kATm, ss = it % kScaleStages;
    bool ok = dead || mbar_wait(&B.f_full[fs], static_cast<uint32_t>(it / kFStages) & 1u, status);
    ok = ok && (dead || mbar_wait(&B.a_empty[as], (static_cast<uint32_t>(it / kATm) & 1u) ^ 1u, status));
    if (!__all_sync(0xffffffffu, ok)) dead = true;
    tc_fence_after();
    // the rows the producer copied: the tile's, clamped at the cache's end
    int64_t nload = static_cast<int64_t>(tl.nunits) * kBoxRows;
    if (row0 + nload > total_rows) nload = total_rows - row0;
    const int r = quarter * 32 + lane;
    const bool valid = r < nload;
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                           static_cast<uint32_t>(kAcc * kN + as * kAColsF);
    const int emax = fp4_expand_row_tmem(sF + fs * kFBytes + r * kFRow, valid, taddr);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&B.a_full[as]);
    mbar_arrive(&B.f_empty[fs]);
    S.fscale[ss][r] = valid ? fp4_key_scale(emax, qs) : 0.f;   // others: never scored
    mbar_arrive(&B.sfull[ss]);
}

template <bool kFused, bool kFp4>
__global__ void __launch_bounds__(kFp4 ? kThreadsFp4 : kThreads, 1)
    dec_indexer_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_q, const DecParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_smem<1024>(smem_raw);
    constexpr int kAst = kFp4 ? kATm : kStages;        // stages of the MMA's A operand
    constexpr int kQb = kFp4 ? 2 : 1;                  // query buffers
    uint8_t *sA = smem;
    uint8_t *sF = smem;                                // FP4: raw code ring
    uint8_t *sB = smem + kStages * kABytes;
    uint8_t *sB1 = smem + kFStages * kFBytes;          // FP4: the second query buffer
    DecSmem &S = *reinterpret_cast<DecSmem *>(sB + kBBytes);
    uint64_t *a_full = S.bars;
    uint64_t *a_empty = a_full + kAst;
    uint64_t *b_full = a_empty + kAst;                 // [kQb]
    uint64_t *b_empty = b_full + kQb;                  // [kQb]
    uint64_t *acc_full = b_empty + kQb;
    uint64_t *acc_empty = acc_full + kAcc;
    uint64_t *b_conv = acc_empty + kAcc;               // FP4 [2]: q converted to f16
    uint64_t *f_full = b_conv + 2;                     // FP4: raw tile landed
    uint64_t *f_empty = f_full + kFStages;             // FP4: raw tile expanded
    static_assert(2 * kATm + 4 + 2 * kAcc + 2 + 2 * kFStages <= 40 && 2 * kStages + 2 + 2 * kAcc <= 40,
                  "pipeline barriers");
    const Fp4Bars fb{f_full, f_empty, a_full, a_empty, S.sfull};

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int T = P.L.num_tokens;
    const int G = gridDim.x;
    const int c = blockIdx.x;

    if (tid == 0) {
        for (int s = 0; s < kAst; ++s) {
            mbar_init(&a_full[s], kFp4 ? kExpThreads : 1);
            mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < kQb; ++s) {
            mbar_init(&b_full[s], 1);
            mbar_init(&b_empty[s], 1);
        }
        for (int a = 0; a < kAcc; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], kEpiThreads);
        }
        if (kFp4) {
            for (int s = 0; s < 2; ++s) mbar_init(&b_conv[s], kConvThreads);
            for (int s = 0; s < kFStages; ++s) {
                mbar_init(&f_full[s], 1);
                mbar_init(&f_empty[s], kExpThreads);
            }
            for (int s = 0; s < kScaleStages; ++s) mbar_init(&S.sfull[s], kExpThreads);
        }
        mbar_init(&S.rbar, 1);
        mbar_fence_init();
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_q);
        S.nresolve = 0;
        S.rphase = 0;
    }
    if (warp == 1) {
        tmem_alloc(&S.tmem_holder, kFp4 ? kTmemColsF : static_cast<uint32_t>(kAcc * kN));
        tmem_relinquish();
    }
    constexpr int kCta = kFp4 ? kThreadsFp4 : kThreads;
    if (kFused)
        for (int i = tid; i < kD1Bins; i += kCta) S.hist[i] = 0;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = S.tmem_holder;

    // ---- every token's visible blocks and units (the same in every CTA).
    // The layout is read before the wait for the preceding grid: no kernel
    // of this library writes a layout while letting its dependents start
    // early, and any other kernel has finished before this one starts.
    for (int t = tid; t < T; t += kCta) {
        const TokenView v = token_view(P.L, P.ratio, t);
        if (v.bad && c == 0) raise_status(P.status, v.bad);
        const int64_t nv = v.bad & CSA_DEV_BAD_LAYOUT ? 0 : v.n_vis;
        S.nvis[t] = static_cast<int32_t>(nv);
        S.off[t] = v.off;
        // a token with no more visible blocks than top_k selects all of them
        S.U[t + 1] = (kFused && nv <= P.top_k) ? 0 : (nv + kBoxRows - 1) / kBoxRows;
    }
    __syncthreads();
    if (warp == 0) warp_prefix(S.U, T);
    __syncthreads();
    const int64_t K32 = S.U[T];
    const int Ge = static_cast<int>(K32 < G ? K32 : G);   // CTAs with work: one unit at least
    const int64_t ua = c < Ge ? K32 * c / Ge : K32;
    const int64_t ub = c < Ge ? K32 * (c + 1) / Ge : K32;
    // The queries, weights and keys may come from the preceding grid.
    pdl_wait();
    // Warm L2 with the first keys of this CTA's range (one bulk prefetch, from
    // a warp that is idle until later).
    if (warp == 6 && lane == 0 && ua < ub) {
        const int t0 = token_of(S.U, T, ua);
        int64_t u1 = S.U[t0 + 1] < ub ? S.U[t0 + 1] : ub;
        int64_t n = (u1 - ua) * kBoxRows;
        n = n < kWarmKeys ? n : kWarmKeys;
        const int64_t r0 = S.off[t0] + (ua - S.U[t0]) * kBoxRows;
        if (r0 + n > P.L.total_comp_rows) n = P.L.total_comp_rows - r0;
        constexpr int64_t kRowB = kFp4 ? kFRow : 256;
        if (n > 0)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(P.k_idx + r0 * kRowB),
                         "r"(static_cast<uint32_t>(n * kRowB))
                         : "memory");
    }
    // The next kernel may start its prologue; it waits for this grid to finish.
    pdl_launch_dependents();

    if (warp == 0) {
      if constexpr (kFp4) {
        // ------------------------------------------------ FP4: TMA / bulk producer
        // Each token's queries go to buffer g & 1 (g counts the CTA's
        // tokens) once the MMA is done with token g - 2's; the raw key tiles
        // fill the ring behind them.
        if (lane == 0 && ua < ub) {
            const uint64_t pol_k = policy_evict_first();
            const uint64_t pol_q = policy_evict_last();
            int t = token_of(S.U, T, ua), cur = -1, g = -1;
            int64_t u = ua;
            int it = 0;
            bool dead = false;
            Tile tl;
            while (next_tile(S.U, ub, t, u, tl)) {
                if (tl.t != cur) {
                    ++g;
                    const int slot = g & 1;
                    const uint32_t ph = static_cast<uint32_t>(g >> 1) & 1u;
                    if (!dead && !mbar_wait(&b_empty[slot], ph ^ 1u, P.status)) dead = true;
                    uint8_t *dst = slot ? sB1 : sB;
                    mbar_arrive_expect_tx(&b_full[slot], kBBytes);
                    tma_load_2d(dst, &tm_q, 0, tl.t * kN, &b_full[slot], pol_q);
                    tma_load_2d(dst + kBBytes / 2, &tm_q, 64, tl.t * kN, &b_full[slot], pol_q);
                    cur = tl.t;
                }
                // the tile's rows are contiguous: one bulk copy (clamped at the
                // cache's end; rows past it are never scored)
                const int fs = it % kFStages;
                const uint32_t ph = static_cast<uint32_t>(it / kFStages) & 1u;
                if (!dead && !mbar_wait(&f_empty[fs], ph ^ 1u, P.status)) dead = true;
                const int64_t r0 = S.off[tl.t] + tl.s0;
                int64_t nr = static_cast<int64_t>(tl.nunits) * kBoxRows;
                if (r0 + nr > P.L.total_comp_rows) nr = P.L.total_comp_rows - r0;
                const uint32_t bytes = static_cast<uint32_t>(nr * kFRow);
                mbar_arrive_expect_tx(&f_full[fs], bytes);
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
                    "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(sF + fs * kFBytes)),
                    "l"(P.k_idx + r0 * kFRow), "r"(bytes), "r"(smem_addr(&f_full[fs])), "l"(pol_k)
                    : "memory");
                ++it;
            }
        }
      } else {
        // ------------------------------------------------ TMA producer
        if (lane == 0 && ua < ub) {
            const uint64_t pol_k = policy_evict_first();
            const uint64_t pol_q = policy_evict_last();
            int t = token_of(S.U, T, ua), cur = -1;
            int64_t u = ua, row_base = 0;
            uint32_t gsw = 0;
            int it = 0;
            bool dead = false;
            Tile tl;
            while (next_tile(S.U, ub, t, u, tl)) {
                if (tl.t != cur) {
                    if (!dead && !mbar_wait(b_empty, (gsw & 1u) ^ 1u, P.status)) dead = true;
                    mbar_arrive_expect_tx(b_full, kBBytes);
                    const int y = tl.t * kN;
                    tma_load_2d(sB, &tm_q, 0, y, b_full, pol_q);
                    tma_load_2d(sB + kBBytes / 2, &tm_q, 64, y, b_full, pol_q);
                    row_base = S.off[tl.t];
                    cur = tl.t;
                    ++gsw;
                }
                const int stage = it % kStages;
                const uint32_t ph = static_cast<uint32_t>(it / kStages) & 1u;
                if (!dead && !mbar_wait(&a_empty[stage], ph ^ 1u, P.status)) dead = true;
                mbar_arrive_expect_tx(&a_full[stage], static_cast<uint32_t>(tl.nunits) * 2u * kBoxBytes);
                uint8_t *dst = sA + stage * kABytes;
                const int32_t row0 = static_cast<int32_t>(row_base + tl.s0);
                for (int bx = 0; bx < tl.nunits; ++bx) {
                    tma_load_2d(dst + bx * kBoxBytes, &tm_k, 0, row0 + bx * kBoxRows, &a_full[stage], pol_k);
                    tma_load_2d(dst + kHalfBytes + bx * kBoxBytes, &tm_k, 64, row0 + bx * kBoxRows,
                                &a_full[stage], pol_k);
                }
                ++it;
            }
        }
      }
    } else if (warp == 1) {
      if constexpr (kFp4) {
        // ------------------------------------------------ FP4: MMA issuer (A from tensor memory)
        if (lane == 0 && ua < ub) {
            constexpr uint32_t idesc = idesc_f16_f32<kTileKeys, kN>();
            int t = token_of(S.U, T, ua), cur = -1, g = -1;
            int64_t u = ua;
            int it = 0;
            bool dead = false;
            Tile tl;
            while (next_tile(S.U, ub, t, u, tl)) {
                if (tl.t != cur) {
                    ++g;   // the token's queries, converted to f16
                    if (!dead && !mbar_wait(&b_conv[g & 1], static_cast<uint32_t>(g >> 1) & 1u, P.status))
                        dead = true;
                    cur = tl.t;
                }
                const int acc = it % kAcc;
                if (!dead && !mbar_wait(&acc_empty[acc], (static_cast<uint32_t>(it / kAcc) & 1u) ^ 1u,
                                        P.status))
                    dead = true;
                const int stage = it % kATm;
                if (!dead && !mbar_wait(&a_full[stage], static_cast<uint32_t>(it / kATm) & 1u, P.status))
                    dead = true;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kN);
                const uint32_t a_tm = tmem_base + static_cast<uint32_t>(kAcc * kN + stage * kAColsF);
                const uint32_t b_base = smem_addr((g & 1) ? sB1 : sB);
#pragma unroll
                for (int kk = 0; kk < kIHD / 16; ++kk) {
                    const uint32_t b_addr = b_base + (kk >> 2) * (kBBytes / 2) + (kk & 3) * 32;
                    umma_f16_ts(d_tmem, a_tm + static_cast<uint32_t>(kk * 8), sw128_kmajor_desc(b_addr), idesc,
                                kk > 0 ? 1u : 0u);
                }
                umma_commit(&a_empty[stage]);
                umma_commit(&acc_full[acc]);
                if (tl.last) umma_commit(&b_empty[g & 1]);
                ++it;
            }
        }
      } else {
        // ------------------------------------------------ MMA issuer
        if (lane == 0 && ua < ub) {
            constexpr uint32_t idesc = idesc_bf16_f32<kTileKeys, kN>();
            int t = token_of(S.U, T, ua), cur = -1;
            int64_t u = ua;
            uint32_t gsw = 0;
            int it = 0;
            bool dead = false;
            const uint32_t a_base = smem_addr(sA);
            const uint32_t b_base = smem_addr(sB);
            Tile tl;
            while (next_tile(S.U, ub, t, u, tl)) {
                if (tl.t != cur) {
                    if (!dead && !mbar_wait(b_full, gsw & 1u, P.status)) dead = true;
                    cur = tl.t;
                    ++gsw;
                }
                const int acc = it % kAcc;
                if (!dead && !mbar_wait(&acc_empty[acc], (static_cast<uint32_t>(it / kAcc) & 1u) ^ 1u,
                                        P.status))
                    dead = true;
                const int stage = it % kStages;
                const uint32_t ph = static_cast<uint32_t>(it / kStages) & 1u;
                if (!dead && !mbar_wait(&a_full[stage], ph, P.status)) dead = true;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kN);
                const uint32_t a_st = a_base + stage * kABytes;
#pragma unroll
                for (int kk = 0; kk < kIHD / 16; ++kk) {
                    const uint32_t a_addr = a_st + (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                    const uint32_t b_addr = b_base + (kk >> 2) * (kBBytes / 2) + (kk & 3) * 32;
                    umma_bf16(d_tmem, sw128_kmajor_desc(a_addr), sw128_kmajor_desc(b_addr), idesc,
                              kk > 0 ? 1u : 0u);
                }
                umma_commit(&a_empty[stage]);
                umma_commit(&acc_full[acc]);
                if (tl.last) umma_commit(b_empty);
                ++it;
            }
        }
      }
    } else if (warp < 6) {
        // ------------------------------------------------ epilogue
        // No early exit from this loop: segment ends meet at named barriers,
        // so a warp that gave up on a wait still walks every tile.
        const int gt = tid - 64;
        const int quarter = warp & 3;   // the TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        int t = ua < ub ? token_of(S.U, T, ua) : 0;
        int64_t u = ua, seg_u0 = ua;
        int it = 0;
        bool dead = false, slots_ready = false;
        int wcur = -1;
        float *wc = S.wc[warp - 2];
        Tile tl;
        while (next_tile(S.U, ub, t, u, tl)) {
            if (tl.t != wcur) {
                // the token's 64 weights, once per token, for broadcast reads
                const float *wt = P.w_idx + static_cast<int64_t>(tl.t) * kNIH;
                __syncwarp();
                wc[lane] = __ldg(wt + lane);
                wc[lane + 32] = __ldg(wt + lane + 32);
                __syncwarp();
                wcur = tl.t;
            }
            const int acc = it % kAcc;
            bool ok = dead || mbar_wait(&acc_full[acc], static_cast<uint32_t>(it / kAcc) & 1u, P.status);
            if (!__all_sync(0xffffffffu, ok)) dead = true;
            tc_fence_after();
            float v[4][16];
            const uint32_t col = tmem_base + lane_addr + static_cast<uint32_t>(acc * kN);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) tmem_ld16(col + c4 * 16, v[c4]);
            tmem_wait_ld();
            // FP4: the key's scale 2^(E_max - 127 + s_q), read before the
            // accumulator goes back (the converters reuse the slot after that)
            float ksc = 1.f;
            if constexpr (kFp4) {
                const int ss = it % kScaleStages;
                const bool ok2 =
                    dead || mbar_wait(&S.sfull[ss], static_cast<uint32_t>(it / kScaleStages) & 1u, P.status);
                if (!__all_sync(0xffffffffu, ok2)) dead = true;
                ksc = S.fscale[ss][row];
            }
            // the accumulator is in registers: hand it back before the math
            tc_fence_before();
            mbar_arrive(&acc_empty[acc]);
            const int tk = tl.t;
            const int64_t nv = S.nvis[tk];
            const int64_t s = tl.s0 + row;
            const bool valid = row < tl.nunits * kBoxRows && s < nv;
            float part[4] = {0.f, 0.f, 0.f, 0.f};  // four short chains, summed in order
            const float4 *wc4 = reinterpret_cast<const float4 *>(wc);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    const float4 w4 = wc4[(c4 * 16 + i) / 4];
                    part[c4] = fmaf(w4.x, fmaxf(v[c4][i + 0], 0.f), part[c4]);
                    part[c4] = fmaf(w4.y, fmaxf(v[c4][i + 1], 0.f), part[c4]);
                    part[c4] = fmaf(w4.z, fmaxf(v[c4][i + 2], 0.f), part[c4]);
                    part[c4] = fmaf(w4.w, fmaxf(v[c4][i + 3], 0.f), part[c4]);
                }
            // (FP4: relu(c x) = c relu(x) for the positive key scale c)
            const float score = ((part[0] + part[1]) + (part[2] + part[3])) * ksc;
            if (valid && CSA_CHECK(s < P.ld, P.status)) P.scores[static_cast<int64_t>(tk) * P.ld + s] = score;
            if (kFused) {
                const uint32_t key = score_key(score);
                const int64_t lo = (tl.u - ua) * kBoxRows + row;
                if (valid && lo < kSegKeysMax) {
                    S.keys[lo] = key;
                    atomicAdd(&S.hist[key >> kD1Shift], 1u);   // 32 neighbours rarely share a bin
                }
                // a segment that ends before the CTA's range does is closed
                // here; the range's last one by the whole CTA after the loop
                if (tl.last && tl.u + tl.nunits < ub) {
                    if (!slots_ready) {
                        named_bar_sync(kBarSlots, kEpiThreads + 64);
                        slots_ready = true;
                    }
                    finalize_segment<4>(P, S, tk, seg_u0, tl.u + tl.nunits, ua, K32, Ge, c, gt, kBarEpi);
                }
            }
            if (tl.last) seg_u0 = tl.u + tl.nunits;
            ++it;
        }
        if (kFused && !slots_ready) named_bar_sync(kBarSlots, kEpiThreads + 64);
    } else if (warp < kWarps) {
      if constexpr (kFused) {
        // ------------------------------------------------ slot table (warps 6, 7)
        // candidate slots: one per (token, CTA that owns part of it)
        const int at = tid - 192;
        for (int t = at; t < T; t += 64) {
            const int64_t u0 = S.U[t], u1 = S.U[t + 1];
            S.sb[t + 1] = u1 > u0 ? cta_of(u1 - 1, K32, Ge) - cta_of(u0, K32, Ge) + 1 : 0;
        }
        named_bar_sync(kBarAux, 64);
        if (warp == 6) warp_prefix(S.sb, T);
        named_bar_sync(kBarAux, 64);
        // tokens that select every visible block: written right away
        for (int t = c; t < T; t += G) {
            if (S.U[t + 1] != S.U[t]) continue;
            const int nv = S.nvis[t];
            int32_t *out = P.f.idx + static_cast<int64_t>(t) * P.top_k;
            for (int i = at; i < P.top_k; i += 64) out[i] = i < nv ? i : -1;
            if (at == 0) P.f.n_sel[t] = nv;
        }
        if (at == 0 && (S.sb[T] > P.f.slots || (ub - ua) * kBoxRows > kSegKeysMax))
            raise_status(P.status, CSA_DEV_CAPACITY);   // the host plan rules this out
        // the epilogue waits for the table; these warps go on (FP4: to convert)
        named_bar_arrive(kBarSlots, kEpiThreads + 64);
      }
      if constexpr (kFp4) {
        // ------------------------------------------------ FP4: queries + expansion of TMEM lanes 64..127
        // Each token's q: bf16 -> f16 in place, scaled by 2^-s_q so that its
        // largest magnitude lands in [2^14, 2^15): below f16's largest value
        // and clear of its subnormals (s_q goes to the other expanders).
        // Then these warps expand their quarters of each key tile, as warps
        // 0 and 1 do theirs.
        const int ct = tid - 192;
        const int cw = warp - 6;
        int t = ua < ub ? token_of(S.U, T, ua) : 0, cur = -1, g = -1;
        int64_t u = ua;
        int it = 0;
        bool dead = false;
        int qs = 0;
        Tile tl;
        while (next_tile(S.U, ub, t, u, tl)) {
            if (tl.t != cur) {
                ++g;
                uint8_t *qb = (g & 1) ? sB1 : sB;
                const bool ok = dead || mbar_wait(&b_full[g & 1], static_cast<uint32_t>(g >> 1) & 1u, P.status);
                if (!__all_sync(0xffffffffu, ok)) dead = true;
                constexpr int kQv = kBBytes / 16 / kConvThreads;   // 16 x 16 bytes per thread
                uint4 *qv = reinterpret_cast<uint4 *>(qb) + ct * kQv;
                uint4 w[kQv];
                float mx = 0.f;
#pragma unroll
                for (int j = 0; j < kQv; ++j) {
                    w[j] = qv[j];
                    const uint32_t ww[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        mx = fmaxf(mx, fabsf(__uint_as_float(ww[e] << 16)));
                        mx = fmaxf(mx, fabsf(__uint_as_float(ww[e] & 0xFFFF0000u)));
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                if (lane == 0) S.qmax[cw] = mx;
                named_bar_sync(kBarConv, kConvThreads);
                mx = fmaxf(S.qmax[0], S.qmax[1]);
                // (|s_q| <= 126 keeps 2^-s_q a finite f32; all-zero q: s_q = 0)
                qs = mx > 0.f ? min(max(ilogbf(mx) - 14, -126), 126) : 0;
                const float f = ldexpf(1.f, -qs);
#pragma unroll
                for (int j = 0; j < kQv; ++j) {
                    const uint32_t ww[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __half2 h2 = __floats2half2_rn(__uint_as_float(ww[e] << 16) * f,
                                                             __uint_as_float(ww[e] & 0xFFFF0000u) * f);
                        o[e] = *reinterpret_cast<const uint32_t *>(&h2);
                    }
                    qv[j] = make_uint4(o[0], o[1], o[2], o[3]);
                }
                if (ct == 0) S.qsi[g & 1] = qs;
                named_bar_sync(kBarConv, kConvThreads);   // S.qmax is read by both warps first
                fence_proxy_async_smem();
                mbar_arrive(&b_conv[g & 1]);
                cur = tl.t;
            }
            fp4_expand_quarter(S, sF, fb, tmem_base, warp & 3, tl, S.off[tl.t] + tl.s0, P.L.total_comp_rows, it,
                               qs, dead, P.status);
            ++it;
        }
      }
    }
    if constexpr (kFp4) {
        if (warp >= kWarps) {
            // ------------------------------------------------ FP4: expansion of TMEM lanes 0..63 (warps 8, 9)
            int t = ua < ub ? token_of(S.U, T, ua) : 0, cur = -1, g = -1;
            int64_t u = ua;
            int it = 0;
            bool dead = false;
            int qs = 0;
            Tile tl;
            while (next_tile(S.U, ub, t, u, tl)) {
                if (tl.t != cur) {
                    ++g;   // the token's s_q, from the converter warps
                    const bool okq = dead || mbar_wait(&b_conv[g & 1], static_cast<uint32_t>(g >> 1) & 1u,
                                                       P.status);
                    if (!__all_sync(0xffffffffu, okq)) dead = true;
                    qs = S.qsi[g & 1];
                    cur = tl.t;
                }
                fp4_expand_quarter(S, sF, fb, tmem_base, warp & 3, tl, S.off[tl.t] + tl.s0,
                                   P.L.total_comp_rows, it, qs, dead, P.status);
                ++it;
            }
            // done: every TMEM store of these warps completed before the
            // MMAs that read it, and the rest of the kernel is warps 0..7's
            return;
        }
    }

    if (kFused && ua < ub) {
        // the CTA's last segment, by all eight warps
        const int tk = token_of(S.U, T, ub - 1);
        const int64_t su0 = S.U[tk] > ua ? S.U[tk] : ua;
        finalize_segment<kWarps>(P, S, tk, su0, ub, ua, K32, Ge, c, tid, 0);
    }
    tc_fence_before();
    main_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kFp4 ? kTmemColsF : static_cast<uint32_t>(kAcc * kN));
    }
    if (kFused) {
        const int nr = S.nresolve;
        for (int r = 0; r < nr; ++r)
            resolve_token(P, S, reinterpret_cast<uint64_t *>(sA), S.resolve[r]);
    }
}

constexpr size_t kDecSmemBytes = 1024 + kStages * kABytes + kBBytes + sizeof(DecSmem);
static_assert(kDecSmemBytes <= 227 * 1024, "decode indexer shared memory");

size_t dec_smem_bytes() { return kDecSmemBytes; }

int dec_grid(const csa_layout_t &L, int sm_count) {
    const int64_t units = static_cast<int64_t>(L.num_tokens) *
                          ((L.max_comp_rows + kBoxRows - 1) / kBoxRows);
    int64_t g = (units + kTileUnits - 1) / kTileUnits;   // about one key tile per CTA at least
    if (g > sm_count) g = sm_count;
    if (g > kMaxIdxCtas) g = kMaxIdxCtas;
    return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

bool decode_indexer_fits(const csa_layout_t &L, int sm_count, bool fused) {
    if (L.num_tokens < 1 || L.num_tokens > (fused ? kFusedMaxTokens : kDecMaxTokens)) return false;
    if (!fused) return true;
    const int64_t units = static_cast<int64_t>(L.num_tokens) *
                          ((L.max_comp_rows + kBoxRows - 1) / kBoxRows);
    const int64_t G = dec_grid(L, sm_count);
    return ((units + G - 1) / G) * kBoxRows <= kSegKeysMax;
}

cudaError_t launch_decode_indexer(const Launch &lc, const csa_layout_t &L, const csa_params_t &p,
                                  const void *q_idx, const float *w_idx, const void *k_idx,
                                  float *scores, int64_t ld, int32_t *status,
                                  const FusedTopk *fused, bool fp4) {
    const int T = L.num_tokens;
    if (T <= 0) return cudaSuccess;
    CUtensorMap tk, tq;
    if (L.total_comp_rows > 0 && !fp4) {
        if (encode_tensor_map_2d_bf16(&tk, k_idx, kIHD, static_cast<uint64_t>(L.total_comp_rows),
                                      kIHD * 2, 64, kBoxRows) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else {
        // FP4 keys come by bulk copies, and with no cache rows at all no key
        // tile is ever loaded: a map over the queries keeps the argument valid
        if (encode_tensor_map_2d_bf16(&tk, q_idx, kIHD, static_cast<uint64_t>(T) * kNIH, kIHD * 2,
                                      64, kBoxRows) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    if (encode_tensor_map_2d_bf16(&tq, q_idx, kIHD, static_cast<uint64_t>(T) * kNIH, kIHD * 2, 64,
                                  kN) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    DecParams P;
    P.L = L;
    P.ratio = p.ratio;
    P.top_k = p.top_k;
    P.w_idx = w_idx;
    P.k_idx = static_cast<const uint8_t *>(k_idx);
    P.scores = scores;
    P.ld = ld;
    P.status = status;
    P.f = fused ? *fused : FusedTopk{};
    const size_t smem = dec_smem_bytes();
    const int grid = dec_grid(L, lc.sm_count);
    auto kern = fused ? (fp4 ? dec_indexer_kernel<true, true> : dec_indexer_kernel<true, false>)
                      : (fp4 ? dec_indexer_kernel<false, true> : dec_indexer_kernel<false, false>);
    cudaError_t e = set_kernel_smem(kern, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(fp4 ? kThreadsFp4 : kThreads), smem, lc.stream, tk, tq, P);
}

}  // namespace csa
