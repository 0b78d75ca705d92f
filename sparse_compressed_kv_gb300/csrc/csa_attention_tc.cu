// csa_attention_tc.cu -- shared-KV multi-query attention on the 5th-generation
// tensor cores, all of a token's query heads (up to 64) in one CTA.
//
//   l_j = scale * q_h . row_j,   out_h = sum_j softmax_j(l) row_j
//
// ("ARCHITECTURE & MEMORY AUDIT -- 1M-context viability", D5 and D6: every
// 512-wide row is the key and the value of all query heads; M5: the selected
// compressed rows are read by index, the window rows from the ring, with no
// gather buffer.  "PART A -- Next Session Clues", section 3: both kept where
// they overlap.)
//
// A CTA owns one token, up to 64 heads, a contiguous range of the token's
// row slots, which it walks in chunks of 64 rows, and 1, 2 or all 4 of the
// output's 128-column tiles (with few CTAs in the grid, 2 or 4 CTAs share a
// row range: each computes its logits and weights in full and accumulates
// only its own columns).  Each row is read from DRAM once for all heads:
//   warp 1      TMEM allocator + tcgen05.mma issuer:
//                 S  = Q . rows^T       M = 64 heads, N = 64 rows, K = 512
//                 O^T += rows^T . P^T   M = 128 of the 512 columns per owned
//                                       tile (the row tile read MN-major),
//                                       N = 64 heads, K = 64 rows; P as two
//                                       bf16 terms
//   warps 0, 6+ fetch a chunk's rows by index into a two-stage ring (16-byte
//               cp.async, 512 contiguous bytes per warp instruction, placed
//               in the 128-byte-swizzled layout the MMA reads); a chunk is
//               handed to the MMA as soon as it has landed
//   warps 2..5  online softmax: two lanes per head (the M = 64 accumulator's
//               row h sits in lane h % 16 of lane quarter h / 16; one
//               two-access tensor-memory load gives its lower 32 columns to
//               that thread and its upper 32 to the thread 16 above), then
//               the epilogue (one
//               output column per lane).
// S is double-buffered in TMEM and the MMA warp issues QK^T of chunk i+1
// before PV of chunk i, so it runs during the softmax of chunk i; O^T
// accumulates in TMEM across chunks.  Exponentials use the
// running maximum of each head; when a chunk raises it by more than 8 (log2
// units) the accumulated O^T and l are rescaled first, so a weight never
// exceeds 2^8 and the two bf16 terms of P keep ~14 bits of it or more.
//
// Row slots of a token: its selected compressed rows (or, HCA, every visible
// block) first, then its window rows starting at the next multiple of 4,
// padding masked.  With several splits per token each CTA writes its
// partial (O, m, l) of its columns and a combine kernel merges them.
#include <math.h>

#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {
namespace {

#ifndef CSA_TC_LOAD_WARPS
#define CSA_TC_LOAD_WARPS 4
#endif
constexpr int kLdWarps = CSA_TC_LOAD_WARPS;    // row-fetch warps: warp 0 and warps 6 ..
constexpr int kLdRows = 64 / kLdWarps;         // rows of a chunk per fetch warp
constexpr int kTcWarps = 5 + kLdWarps;
constexpr int kTcThreads = 32 * kTcWarps;
constexpr int kSmThreads = 128;                // warps 2..5
constexpr int kBarSm = 1;                      // named barrier of the softmax warps
constexpr int kLdThreads = 32 * kLdWarps;
constexpr int kHG = 64;                        // heads per CTA (MMA M of QK^T)
constexpr int kChunk = kTcChunk;               // rows per chunk (QK^T N, PV K): 64
static_assert(kChunk == 64, "the softmax gives each lane 32 rows of a chunk");
constexpr int kQBytes = 8 * kHG * 128;         // 64 KiB: Q, eight 64-column boxes
constexpr int kRowBox = kChunk * 128;          // 8 KiB: 64 columns of a chunk's rows
constexpr int kRowsBytes = 8 * kRowBox;        // 64 KiB per stage
constexpr int kPBytes = kHG * kChunk * 2;      // 8 KiB: one bf16 term of P
constexpr int kTmemCols = 512;
constexpr int kSCol = 0;                       // S buffers: columns 0 .. 127
constexpr int kOCol = 128;                     // O^T: up to 4 tiles x 64 heads
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleAbove = 8.f;           // log2 units

struct TcParams {
    RowSource R;
    int32_t H;
    int32_t splits;
    int32_t rows_split;      // slots per split, a multiple of kChunk
    float scale_log2;
    const float *sinks;      // [H] or null
    float *out;              // [T][H][512]
    float *part_o;           // [T][splits][H][512]
    float *part_ml;          // [T][splits][H][2]  (m in log2 units, l)
    int32_t *status;
    int32_t early_q;
    int32_t raw;             // one split: write the unnormalised partial to part_o / part_ml
    // the combine: where split s of token t, head h starts, in floats
    // (part_o + t * po_t + s * po_s + h * 512, part_ml + t * ml_t + s * ml_s + h * 2)
    int64_t po_t, po_s, ml_t, ml_s;
    float *raw_ml;           // the combine: write the merged partial (out = O, raw_ml = (m, l))
};

struct TcTok;

struct TcSmem {
    uint32_t maskw[2][kLdWarps];   // valid rows of the chunk in each stage, per fetch warp
    uint64_t q_full;
    uint64_t full[2], empty[2];
    uint64_t sfull[2], sfree[2];
    uint64_t pfull[2], pfree[2];
    uint64_t odone;
    float alpha[kHG];        // rescale factors of the current chunk
    float fin[kHG];          // output scale per head
    float mh[kHG], lh[kHG];
    uint32_t flag[2][4];     // per chunk parity: heads of each warp that rescale
    uint32_t tmem_holder;
    int32_t nslots;          // the token's row slots
};

// Row slots of token t: selected (or every visible) compressed rows first, then
// the window rows from the next multiple of 4.  Fills the counts; returns the
// slot count.
struct TcTok {
    int32_t nsel;      // compressed rows
    int32_t nswa;      // window rows
    int32_t wslot;     // first window slot
    int64_t first;     // first window position
    int64_t off;       // the sequence's first cache row
    int64_t n_vis;
    int64_t first_res;  // oldest position the ring holds
    int b;
    int bad;
    int32_t gathered_len;
};

// The layout half of token t's record (read before the kernel waits for the
// preceding grid: no kernel of this library writes a layout while letting
// its dependents start early).
__device__ __forceinline__ TcTok tc_token_layout(const RowSource &R, int t) {
    TcTok k{};
    if (R.fused == kRowsGathered) return k;
    const TokenView v = token_view(R.L, R.ratio, t);
    k.bad = v.bad;
    if (v.bad & CSA_DEV_BAD_LAYOUT) return k;
    k.first = window_first(v.pos, R.window);
    k.nswa = R.no_window ? 0 : static_cast<int32_t>(v.pos - k.first + 1);
    k.off = v.off;
    k.n_vis = v.n_vis;
    k.b = v.b;
    k.first_res = R.L.swa_first_pos[v.b];
    return k;
}

// The rest, after the wait: the selection count (or the gathered length)
// the preceding kernels produced, and the slots that follow from it.
__device__ __forceinline__ void tc_token_finish(const RowSource &R, int t, TcTok &k) {
    if (R.fused == kRowsGathered) {
        int32_t len = R.kv_len[t];
        if (len < 0 || len > R.rows_per_token) {
            k.bad = CSA_DEV_BAD_LENGTH;
            len = len < 0 ? 0 : R.rows_per_token;
        }
        k.gathered_len = len;
        k.nsel = len;
        k.wslot = len;
        return;
    }
    if (k.bad & CSA_DEV_BAD_LAYOUT) return;
    // (the window's partial has no selection to read)
    int32_t ns;
    if (R.fused == kRowsAllVisible) {
        ns = static_cast<int32_t>(k.n_vis);
    } else {
        ns = (R.fused == kRowsSelected && !R.no_selected) ? R.n_sel[t] : 0;
        if (ns < 0 || ns > R.top_k) {
            k.bad |= CSA_DEV_BAD_LENGTH;
            ns = ns < 0 ? 0 : R.top_k;
        }
    }
    if (R.no_selected) ns = 0;
    k.nsel = ns;
    k.wslot = (ns + 3) & ~3;
}

__device__ __forceinline__ void tmem_ld16_raw(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// 16 lanes x 16 columns twice: threads 0..15 read lanes 0..15 of the quarter
// at columns c..c+15, threads 16..31 the same lanes at columns c+32..c+47
__device__ __forceinline__ void tmem_ld16x2_raw(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16], 32;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// 2^x with the hardware's approximate exponential (relative error about
// 2^-22, far below the bf16 terms P is stored in); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}


// Shared-memory descriptor with explicit leading / stride byte offsets
// (128-byte swizzle).  K-major: the stride is the step between 8-row groups.
// MN-major: the leading offset is the step between 64-element column boxes,
// the stride the step between 8-row groups of the K dimension.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// kind::f16, bf16 x bf16 -> f32, M x N, A transposed (MN-major) or not.
template <int M, int N, bool kTransA>
__device__ __forceinline__ constexpr uint32_t idesc_bf16() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((kTransA ? 1u : 0u) << 15) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// kDT: 128-column tiles of the output this CTA owns (4: all 512 columns;
// 2 or 1 when 2 or 4 CTAs share a row split, each computing the split's
// logits and weights in full and accumulating only its own columns).
template <int kDT>
__global__ void __launch_bounds__(kTcThreads, 1)
    attention_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const TcParams A) {
    static_assert(kDT == 1 || kDT == 2 || kDT == 4, "1, 2 or 4 column tiles");
    constexpr int kParts = 4 / kDT;
    constexpr uint32_t kCols = kDT == 4 ? kTmemCols : kTmemCols / 2;   // S + O^T columns, a power of 2
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_smem<1024>(smem_raw);
    uint8_t *sQ = smem;
    uint8_t *sRows = smem + kQBytes;                       // [2][8 boxes][64 rows][128 B]
    uint8_t *sP = sRows + 2 * kRowsBytes;                  // [2 buffers][hi, lo][64 heads][128 B]
    TcSmem &S = *reinterpret_cast<TcSmem *>(sP + 4 * kPBytes);

    const int split = blockIdx.x, t = blockIdx.z;
    const int hg = static_cast<int>(blockIdx.y) / kParts;
    const int dt0 = (static_cast<int>(blockIdx.y) % kParts) * kDT;   // first owned column tile
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h0 = hg * kHG;
    const int H = A.H;

    if (tid == 0) {
        mbar_init(&S.q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&S.full[i], kLdThreads);
            mbar_init(&S.empty[i], 1);
            mbar_init(&S.sfull[i], 1);
            mbar_init(&S.sfree[i], kSmThreads);
            mbar_init(&S.pfull[i], kSmThreads);
            mbar_init(&S.pfree[i], 1);
        }
        mbar_init(&S.odone, 1);
        mbar_fence_init();
        tma_prefetch_desc(&tm_q);
    }
    if (warp == 1) {
        tmem_alloc(&S.tmem_holder, kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_holder;

    // Q of this token's head group: eight 64 x 64 boxes (heads past H read the
    // next token's rows or the tensor's zero fill; their outputs are dropped)
    auto load_q = [&]() {
        mbar_arrive_expect_tx(&S.q_full, kQBytes);
        const int y = t * H + h0;
        for (int bx = 0; bx < 8; ++bx)
            tma_load_2d(sQ + bx * (kHG * 128), &tm_q, bx * 64, y, &S.q_full, policy_evict_normal());
    };
    // the token's row slots (one reader, shared): the layout half now
    __shared__ TcTok tok_s;
    if (tid == 0) tok_s = tc_token_layout(A.R, t);
    if (A.early_q && tid == 0) load_q();
    pdl_wait();
    pdl_launch_dependents();
    if (!A.early_q && tid == 0) load_q();

    // The fetch warps load the selection entries of their first chunk's rows
    // now, in the same round trip as the token record (entries past the
    // token's selection count are read but not used).
    const bool fetch_warp = warp == 0 || warp >= 6;
    int32_t pre_sidx = -1;
    if (fetch_warp && A.R.fused == kRowsSelected && !A.R.no_selected) {
        const int li = warp == 0 ? 0 : warp - 5;
        const int j = split * A.rows_split + kLdRows * li + lane;
        if (lane < kLdRows && j < A.R.top_k) pre_sidx = A.R.idx[static_cast<int64_t>(t) * A.R.top_k + j];
    }
    // ... and the selection half after the wait
    if (tid == 0) {
        TcTok kk = tok_s;
        tc_token_finish(A.R, t, kk);
        tok_s = kk;
        S.nslots = A.R.fused == kRowsGathered ? kk.gathered_len : kk.wslot + kk.nswa;
        if (split == 0 && blockIdx.y == 0) raise_status(A.status, kk.bad);
    }
    __syncthreads();
    const int nslots = S.nslots;
    const int s_begin = split * A.rows_split;
    const int s_end = min(nslots, s_begin + A.rows_split);
    const int nch = s_end > s_begin ? (s_end - s_begin + kChunk - 1) / kChunk : 0;

    if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0 && nch > 0) {
            mbar_wait(&S.q_full, 0, A.status);
            constexpr uint32_t id_qk = idesc_bf16<kHG, kChunk, false>();
            constexpr uint32_t id_pv = idesc_bf16<128, kHG, true>();
            // Descriptors are built once and stepped by adding an operand's
            // byte offset / 16 to the start-address field (every shared
            // address is below 256 KiB, so the 14-bit field never carries):
            // building one per instruction made the issuing thread, not the
            // tensor pipe, set the pace of these small MMAs.
            const uint64_t q_desc = sw128_desc(smem_addr(sQ), 16, 1024);
            const uint64_t r_desc = sw128_desc(smem_addr(sRows), 16, 1024);
            const uint64_t a_desc = sw128_desc(smem_addr(sRows) + (2 * dt0) * kRowBox, kRowBox, 1024);
            const uint64_t p_desc = sw128_desc(smem_addr(sP), 16, 1024);
            auto off = [](uint32_t bytes) { return static_cast<uint64_t>(bytes >> 4); };
            // S = Q . rows^T of chunk i, into S buffer i % 2 (rows landed,
            // the S buffer read by the softmax)
            auto qk = [&](int i) {
                const int st = i & 1;
                const uint64_t rd = r_desc + off(st * kRowsBytes);
                const uint32_t d = tmem + kSCol + st * kChunk;
#pragma unroll
                for (int kk = 0; kk < 32; ++kk) {
                    const uint32_t bx = kk >> 2, ko = (kk & 3) * 32;
                    umma_bf16(d, q_desc + off(bx * (kHG * 128) + ko), rd + off(bx * kRowBox + ko), id_qk,
                              kk > 0 ? 1u : 0u);
                }
                umma_commit(&S.sfull[st]);
            };
            // O^T[d][h] += sum_j rows[j][d] P[h][j] of chunk i (P written),
            // per owned 128-column tile of d
            auto pv = [&](int i) {
                const int st = i & 1;
                const uint64_t ad = a_desc + off(st * kRowsBytes);
                const uint64_t pd = p_desc + off(st * 2 * kPBytes);
#pragma unroll
                for (int dd = 0; dd < kDT; ++dd)
#pragma unroll
                    for (int ks = 0; ks < kChunk / 16; ++ks) {
                        const uint64_t adesc = ad + off((2 * dd) * kRowBox + ks * 16 * 128);
                        const uint32_t acc0 = (i > 0 || ks > 0) ? 1u : 0u;
                        umma_bf16(tmem + kOCol + dd * kHG, adesc, pd + off(ks * 32), id_pv, acc0);
                        umma_bf16(tmem + kOCol + dd * kHG, adesc, pd + off(kPBytes + ks * 32), id_pv, 1u);
                    }
                umma_commit(&S.empty[st]);
                umma_commit(&S.pfree[st]);
            };
            // Issue whichever is ready: QK^T of chunk nq (at most one chunk
            // ahead of PV, so it runs during the softmax of chunk nq - 1) or
            // PV of chunk np.  PV does not wait behind a QK^T whose rows are
            // still in flight (those rows wait for the PV two chunks back).
            // Every poll is bounded: after the wait limit the status word gets
            // CSA_DEV_TIMEOUT and the rest is issued without waiting.
            int nq = 0, np = 0;
            bool dead = false;
            uint32_t polls = 0;
            uint64_t t_start = 0;
            while (np < nch) {
                bool did = false;
                if (nq < nch && nq <= np + 1) {
                    const int st = nq & 1;
                    const uint32_t ph = static_cast<uint32_t>(nq >> 1) & 1u;
                    if (dead || (mbar_try_wait(&S.full[st], ph) && mbar_try_wait(&S.sfree[st], ph ^ 1u))) {
                        tc_fence_after();
                        qk(nq++);
                        did = true;
                    }
                }
                if (!did && np < nq) {
                    const int st = np & 1;
                    const uint32_t ph = static_cast<uint32_t>(np >> 1) & 1u;
                    if (dead || mbar_try_wait(&S.pfull[st], ph)) {
                        tc_fence_after();
                        pv(np++);
                        did = true;
                    }
                }
                if (did) {
                    polls = 0;
                } else if (++polls == 1) {
                    t_start = global_timer_ns();
                } else if ((polls & 1023u) == 0 && global_timer_ns() - t_start > kWaitNs) {
                    raise_status(A.status, CSA_DEV_TIMEOUT);
                    dead = true;
                }
            }
            umma_commit(&S.odone);
        }
    } else if (fetch_warp) {
        // ------------------------------------------------ row fetch
        const TcTok k = tok_s;
        const int li = warp == 0 ? 0 : warp - 5;   // rows kLdRows li .. of each chunk
        const void *dummy = A.R.fused == kRowsGathered ? A.R.kv_buf : A.R.L.swa_kv;
        int bad = 0;
        // lane r < kLdRows resolves row r of the warp's share, then the warp
        // copies row after row, 512 contiguous bytes per instruction
        auto issue = [&](int i) {
            const int st = i & 1;
            const int j = s_begin + i * kChunk + kLdRows * li + lane;
            const __nv_bfloat16 *src = nullptr;
            if (lane < kLdRows && j < s_end) {
                if (A.R.fused == kRowsGathered) {
                    src = static_cast<const __nv_bfloat16 *>(A.R.kv_buf) +
                          (static_cast<int64_t>(t) * A.R.rows_per_token + j) * kHD;
                } else if (j < k.nsel) {
                    const int32_t sidx = A.R.fused == kRowsAllVisible
                                             ? j
                                             : (i == 0 ? pre_sidx
                                                       : A.R.idx[static_cast<int64_t>(t) * A.R.top_k + j]);
                    if (sidx < 0 || sidx >= k.n_vis) bad |= CSA_DEV_BAD_INDEX;
                    else if (CSA_CHECK(k.off + sidx < A.R.L.total_comp_rows, A.status))
                        src = static_cast<const __nv_bfloat16 *>(A.R.comp_kv) + (k.off + sidx) * kHD;
                } else if (j >= k.wslot) {
                    const int64_t x = k.first + (j - k.wslot);
                    if (x < k.first_res) bad |= CSA_DEV_MISSING_SWA;
                    else
                        src = static_cast<const __nv_bfloat16 *>(A.R.L.swa_kv) +
                              (static_cast<int64_t>(k.b) * A.R.L.swa_cap + x % A.R.L.swa_cap) * kHD;
                }
            }
            const uint32_t okm = __ballot_sync(0xffffffffu, src != nullptr);
            if (lane == 0) S.maskw[st][li] = okm;
            uint8_t *rows = sRows + st * kRowsBytes;
#pragma unroll 4
            for (int rr = 0; rr < kLdRows; ++rr) {
                const __nv_bfloat16 *p = reinterpret_cast<const __nv_bfloat16 *>(__shfl_sync(
                    0xffffffffu, reinterpret_cast<unsigned long long>(src), rr));
                const int row = kLdRows * li + rr;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int c = lane + 32 * u;   // 16-byte piece of the row
                    uint8_t *dst = rows + (c >> 3) * kRowBox + row * 128 + (((c & 7) ^ (row & 7)) << 4);
                    cp_async16(dst, p ? static_cast<const void *>(p + c * 8) : dummy, p != nullptr);
                }
            }
            cp_async_commit();
        };
        // chunk i + 1 is handed over as soon as it has landed; chunk i + 2
        // goes into the stage of chunk i once PV of chunk i is done with it
        if (nch > 0) issue(0);
        if (nch > 1) {
            issue(1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        if (nch > 0) {
            fence_proxy_async_smem();
            mbar_arrive(&S.full[0]);
        }
        for (int i = 0; i < nch; ++i) {
            if (i + 1 < nch) {
                cp_async_wait<0>();
                fence_proxy_async_smem();
                mbar_arrive(&S.full[(i + 1) & 1]);
            }
            if (i + 2 < nch) {
                mbar_wait(&S.empty[i & 1], static_cast<uint32_t>(i >> 1) & 1u, A.status);
                issue(i + 2);
            }
        }
        bad = static_cast<int>(__reduce_or_sync(0xffffffffu, static_cast<unsigned>(bad)));
        if (lane == 0) raise_status(A.status, bad);
    } else if (warp >= 2) {
        // ------------------------------------------------ softmax, epilogue
        const int q = warp & 3;                  // TMEM lane quarter
        const int hl = q * 16 + (lane & 15);     // head of this lane (two lanes per head)
        const bool upper = lane >= 16;           // rows 32..63 of the chunk
        const bool hv = h0 + hl < H;
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        float m_ref = -INFINITY, l = 0.f;
        const int st_t = tid - 64;
        for (int i = 0; i < nch; ++i) {
            const int st = i & 1;
            const uint32_t ph = static_cast<uint32_t>(i >> 1) & 1u;
            mbar_wait(&S.sfull[st], ph, A.status);
            tc_fence_after();
            // S of the M = 64 product sits in lanes 0..15 of the quarter: the
            // two-access load gives lanes 0..15 columns c.. to threads 0..15
            // and columns c + 32.. to threads 16..31
            uint32_t sr[2][16];
            tmem_ld16x2_raw(tmem + lane_off + kSCol + st * kChunk, sr[0]);
            tmem_ld16x2_raw(tmem + lane_off + kSCol + st * kChunk + 16, sr[1]);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&S.sfree[st]);
            mbar_wait(&S.full[st], ph, A.status);   // orders the fetch warps' mask writes
            uint64_t msk = 0;
#pragma unroll
            for (int w = 0; w < kLdWarps; ++w) msk |= static_cast<uint64_t>(S.maskw[st][w]) << (kLdRows * w);
            // lane l < 16 takes rows 0..31 of head hl, lane l + 16 rows 32..63
            // Every row valid and a scale >= 0: x keeps the raw logits, the
            // maximum is taken on them (scaling by a constant >= 0 keeps the
            // maximum, rounding included) and the scale enters the exponent
            // pass as one fma.  Otherwise x holds the scaled logits (masked
            // rows -inf) and the exponent pass multiplies by 1.
            float x[32];
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // four short max chains
            float xs = 1.f;
            if (msk == ~0ull && A.scale_log2 >= 0.f) {
                xs = A.scale_log2;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    x[j] = __uint_as_float(sr[j >> 4][j & 15]);
                    mq[j & 3] = fmaxf(mq[j & 3], x[j]);
                }
            } else {
                const uint32_t mh = static_cast<uint32_t>(msk >> (upper ? 32 : 0));
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const uint32_t v = sr[j >> 4][j & 15];
                    x[j] = ((mh >> j) & 1u) ? __uint_as_float(v) * A.scale_log2 : -INFINITY;
                    mq[j & 3] = fmaxf(mq[j & 3], x[j]);
                }
            }
            float mc = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
            mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, 16)) * xs;
            // a head whose maximum rises by more than kRescaleAbove rescales
            // what it has accumulated (every lane of the four warps takes part)
            const bool need = hv && m_ref != -INFINITY && mc > m_ref + kRescaleAbove;
            const uint32_t wneed = __ballot_sync(0xffffffffu, need);
            if (lane == 0) S.flag[st][q] = wneed;
            float alpha = 1.f;
            if (need) {
                alpha = exp2f(m_ref - mc);
                m_ref = mc;
                l *= alpha;
            } else if (m_ref == -INFINITY) {
                m_ref = mc;
            }
            named_bar_sync(kBarSm, kSmThreads);
            const bool any = (S.flag[st][0] | S.flag[st][1] | S.flag[st][2] | S.flag[st][3]) != 0;
            if (any) {
                if (!upper) S.alpha[hl] = alpha;
                // PV of the previous chunk must have landed in O^T
                mbar_wait(&S.pfree[st ^ 1], static_cast<uint32_t>((i - 1) >> 1) & 1u, A.status);
                named_bar_sync(kBarSm, kSmThreads);
                tc_fence_after();
#pragma unroll 1
                for (int dd = 0; dd < kDT; ++dd)
#pragma unroll 1
                    for (int hb = 0; hb < 4; ++hb) {
                        uint32_t r[16];
                        const uint32_t ta = tmem + lane_off + kOCol + dd * kHG + hb * 16;
                        tmem_ld16_raw(ta, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            r[c] = __float_as_uint(__uint_as_float(r[c]) * S.alpha[hb * 16 + c]);
                        tmem_st16(ta, r);
                    }
                tmem_wait_st();
                tc_fence_before();
                named_bar_sync(kBarSm, kSmThreads);
            }
            // P = 2^(x - m_ref) as hi + lo bf16 terms, this lane's half of row hl
            // (a head with no valid row yet keeps m_ref = -inf; its masked
            // logits must give 0, not 2^(-inf + inf)).  Both terms are the
            // truncated upper halves of f32 values, so they cost integer
            // operations only: hi = p with its low 16 bits cleared, lo = the
            // same of p - hi; hi + lo is within 2^-14 of p (relative).
            const float mr = m_ref == -INFINITY ? 0.f : m_ref;
            float sq[2] = {0.f, 0.f};
            uint32_t phi[16], plo[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float p0 = fast_exp2(fmaf(x[j], xs, -mr));
                const float p1 = fast_exp2(fmaf(x[j + 1], xs, -mr));
                sq[(j >> 1) & 1] += p0 + p1;
                const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
                const float r0 = p0 - __uint_as_float(b0 & 0xFFFF0000u);
                const float r1 = p1 - __uint_as_float(b1 & 0xFFFF0000u);
                phi[j >> 1] = __byte_perm(b0, b1, 0x7632);
                plo[j >> 1] = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
            }
            const float sum = sq[0] + sq[1];
            l += sum + __shfl_xor_sync(0xffffffffu, sum, 16);
            mbar_wait(&S.pfree[st], ph ^ 1u, A.status);   // PV of chunk i-2 is done with the buffer
            {
                uint8_t *pr = sP + st * 2 * kPBytes + hl * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int cch = (upper ? 4 : 0) + c;
                    const uint32_t sw = static_cast<uint32_t>((cch ^ (hl & 7)) << 4);
                    *reinterpret_cast<uint4 *>(pr + sw) =
                        make_uint4(phi[4 * c], phi[4 * c + 1], phi[4 * c + 2], phi[4 * c + 3]);
                    *reinterpret_cast<uint4 *>(pr + kPBytes + sw) =
                        make_uint4(plo[4 * c], plo[4 * c + 1], plo[4 * c + 2], plo[4 * c + 3]);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&S.pfull[st]);
        }
        // ---- epilogue: O^T column h / l_h (one split) or the raw partial
        if (!upper) {
            S.mh[hl] = m_ref;
            S.lh[hl] = l;
            float f = 1.f;
            if (A.splits == 1 && !A.raw) {
                float z = l;
                if (A.sinks && hv && m_ref != -INFINITY) z += exp2f(A.sinks[h0 + hl] * kLog2e - m_ref);
                f = (z > 0.f && l > 0.f) ? 1.f / z : 0.f;
            }
            S.fin[hl] = f;
        }
        if (nch > 0) mbar_wait(&S.odone, 0, A.status);
        named_bar_sync(kBarSm, kSmThreads);
        tc_fence_after();
        const bool part = A.splits > 1 || A.raw;
        const int64_t obase = part ? ((static_cast<int64_t>(t) * A.splits + split) * H + h0) * kHD
                                   : (static_cast<int64_t>(t) * H + h0) * kHD;
        float *dst = part ? A.part_o : A.out;
        const int hmax = min(kHG, H - h0);
        // one output column per lane: every warp store is 128 contiguous bytes
        if (nch == 0) {
            for (int e = st_t; e < hmax * 128 * kDT; e += kSmThreads)
                dst[obase + (e / (128 * kDT)) * kHD + dt0 * 128 + e % (128 * kDT)] = 0.f;
        } else {
#pragma unroll 1
            for (int dd = 0; dd < kDT; ++dd) {
                const int d = (dt0 + dd) * 128 + q * 32 + lane;
                uint32_t r[4][16];
#pragma unroll
                for (int hb = 0; hb < 4; ++hb) tmem_ld16_raw(tmem + lane_off + kOCol + dd * kHG + hb * 16, r[hb]);
                tmem_wait_ld();
                float *od = dst + obase + d;
                if (part && hmax == kHG) {
                    // a raw partial of a full head group: no scale, no head bound
#pragma unroll
                    for (int hb = 0; hb < 4; ++hb)
#pragma unroll
                        for (int c = 0; c < 16; ++c) od[(hb * 16 + c) * kHD] = __uint_as_float(r[hb][c]);
                } else {
#pragma unroll
                    for (int hb = 0; hb < 4; ++hb)
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const int h = hb * 16 + c;
                            if (h < hmax) od[h * kHD] = __uint_as_float(r[hb][c]) * S.fin[h];
                        }
                }
            }
        }
        if (part && !upper && hv && dt0 == 0) {
            const int64_t mb = ((static_cast<int64_t>(t) * A.splits + split) * H + h0 + hl) * 2;
            A.part_ml[mb + 0] = nch > 0 ? m_ref : -INFINITY;
            A.part_ml[mb + 1] = nch > 0 ? l : 0.f;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kCols);
    }
}

// out[t,h,:] = sum_s 2^(m_s - M) O_s / (sum_s 2^(m_s - M) l_s [+ 2^(sink log2e - M)]),
// splits without rows (m = -inf) skipped.  CTA = (head, token, column part)
// of cw nsub threads and one more warp, cw = 128 / parts: thread (sub, c4)
// holds columns 4 c4 .. 4 c4 + 3 of the part for splits sub, sub + nsub,
// ..., loaded kPer at a time (all of them in flight), the last warp reads
// every split's (m, l) meanwhile, and the nsub partial sums meet in shared
// memory in a fixed order.  Many splits: 4 parts of 128 columns (each CTA
// reads a quarter of the partials); few: one part, fewer and larger CTAs.
constexpr int kMaxSplits = 256;
constexpr int kMlPer = kMaxSplits / 32;    // (m, l) pairs per lane of the last warp
constexpr int kCombWideSub = 7;            // one part: at most 7 x 128 column threads
constexpr int kCombMaxSub = 31;            // four parts: at most 31 x 32
constexpr int kCombMaxThreads = 32 * kCombMaxSub + 32;
constexpr int kCombRed = 960;              // partial sums of subs 1..: 30 x 32 or 6 x 128
static_assert((kCombMaxSub - 1) * 32 <= kCombRed && (kCombWideSub - 1) * 128 <= kCombRed, "combine sums");

// kCw: column threads per sub, 128 (one part) or 32 (four parts); kPer:
// splits a thread loads per round, 8 or 4 (fewer registers: more CTAs per SM
// when the grid is large, more subs in flight when splits are many).
template <int kCw, int kPer>
__global__ void __launch_bounds__(kCombMaxThreads) combine_tc_kernel(const TcParams A) {
    pdl_wait();
    pdl_launch_dependents();
    const int h = blockIdx.x, t = blockIdx.y;
    if (!CSA_CHECK(A.splits <= kMaxSplits, A.status)) return;
    constexpr int cw = kCw;
    const int nsub = (static_cast<int>(blockDim.x) - 32) / cw;
    const bool ml_warp = static_cast<int>(threadIdx.x) >= cw * nsub;
    const int c4 = static_cast<int>(threadIdx.x) % cw, sub = static_cast<int>(threadIdx.x) / cw;
    const int col = static_cast<int>(blockIdx.z) * 4 * cw + 4 * c4;
    __shared__ float wgt[kMaxSplits];
    __shared__ float inv_z;
    __shared__ float4 red[kCombRed];
    const int ns = A.splits;
    const float *mlb = A.part_ml + t * A.ml_t + h * 2;
    const int64_t mstride = A.ml_s;
    // the first kPer of a thread's partial columns are in flight while
    // the last warp reads (m, l) (every split writes its partial, zeros when
    // it has no rows, so the loads need not wait for the weights)
    const float *pb = A.part_o + t * A.po_t + h * kHD + col;
    const int64_t pstride = A.po_s;
    float4 v[kPer];
    if (!ml_warp) {
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int sp = sub + k * nsub;
            if (sp < ns) v[k] = __ldcg(reinterpret_cast<const float4 *>(pb + sp * pstride));
        }
    } else {
        const int lane = threadIdx.x & 31;
        float m[kMlPer], lv[kMlPer];
#pragma unroll
        for (int k = 0; k < kMlPer; ++k) {
            m[k] = -INFINITY;
            lv[k] = 0.f;
            if (lane + 32 * k < ns) {
                const float2 x = __ldcg(reinterpret_cast<const float2 *>(mlb + (lane + 32 * k) * mstride));
                m[k] = x.x;
                lv[k] = x.y;
            }
        }
        float M = m[0];
#pragma unroll
        for (int k = 1; k < kMlPer; ++k) M = fmaxf(M, m[k]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float sink = (A.sinks && !A.raw_ml) ? A.sinks[h] * kLog2e : -INFINITY;
        const float Mall = fmaxf(M, sink);
        float z = 0.f;
#pragma unroll
        for (int k = 0; k < kMlPer; ++k) {
            const float w = m[k] == -INFINITY ? 0.f : exp2f(m[k] - Mall);
            if (lane + 32 * k < ns) wgt[lane + 32 * k] = w;
            z += w * lv[k];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        if (lane == 0) {
            const bool any = M != -INFINITY;
            if (A.raw_ml) {
                // the merged partial: O scaled to M, l = sum_s 2^(m_s - M) l_s
                if (blockIdx.z == 0) {
                    A.raw_ml[(static_cast<int64_t>(t) * A.H + h) * 2 + 0] = M;
                    A.raw_ml[(static_cast<int64_t>(t) * A.H + h) * 2 + 1] = any ? z : 0.f;
                }
                inv_z = 1.f;
            } else {
                if (A.sinks && any) z += exp2f(sink - Mall);
                inv_z = (any && z > 0.f) ? 1.f / z : 0.f;
            }
        }
    }
    __syncthreads();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = sub; !ml_warp && base < ns; base += kPer * nsub) {
        if (base != sub) {
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const int sp = base + k * nsub;
                if (sp < ns && wgt[sp] != 0.f) v[k] = __ldcg(reinterpret_cast<const float4 *>(pb + sp * pstride));
            }
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int sp = base + k * nsub;
            if (sp < ns && wgt[sp] != 0.f) {
                const float w = wgt[sp];
                acc.x += w * v[k].x;
                acc.y += w * v[k].y;
                acc.z += w * v[k].z;
                acc.w += w * v[k].w;
            }
        }
    }
    if (sub > 0 && !ml_warp) red[(sub - 1) * cw + c4] = acc;
    __syncthreads();
    if (sub == 0) {
        for (int j = 0; j + 1 < nsub; ++j) {
            const float4 r = red[j * cw + c4];
            acc.x += r.x;
            acc.y += r.y;
            acc.z += r.z;
            acc.w += r.w;
        }
        const float iz = inv_z;
        float *o = A.out + (static_cast<int64_t>(t) * A.H + h) * kHD + col;
        *reinterpret_cast<float4 *>(o) = make_float4(acc.x * iz, acc.y * iz, acc.z * iz, acc.w * iz);
    }
}

// The combine's launch shape for ns splits of `heads` (head, token) pairs:
// rounds of 4 loads when the grid is large or the splits many, else 8; one
// part while 7 subs of 128 column threads hold every split in one round,
// else four parts.
struct CombShape {
    int parts, threads;
    void (*kernel)(const TcParams);
};
CombShape comb_shape(int ns, int64_t heads, int sm_count) {
    const int nsub8 = (ns + 7) / 8, nsub4 = (ns + 3) / 4;
    if (nsub8 > kCombWideSub)
        return {4, 32 * (nsub4 < kCombMaxSub ? nsub4 : kCombMaxSub) + 32, combine_tc_kernel<32, 4>};
    if (heads > 2 * static_cast<int64_t>(sm_count) && nsub4 <= kCombWideSub)
        return {1, 128 * nsub4 + 32, combine_tc_kernel<128, 4>};
    return {1, 128 * nsub8 + 32, combine_tc_kernel<128, 8>};
}

}  // namespace

size_t attention_tc_smem_bytes() { return 1024 + kQBytes + 2 * kRowsBytes + 4 * kPBytes + sizeof(TcSmem); }

cudaError_t launch_attention_tc(const Launch &lc, const RowSource &src, int32_t T,
                                const csa_params_t &p, const WsPlan &plan, const void *q,
                                const float *sinks, float *out, float *part_o, float *part_ml,
                                int32_t *status, bool early_q, float *raw_ml) {
    if (T <= 0) return cudaSuccess;
    CUtensorMap tq;
    const int H = p.n_heads;
    if (encode_tensor_map_2d_bf16(&tq, q, kHD, static_cast<uint64_t>(T) * H, kHD * 2, 64, kHG) !=
        CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    TcParams A{};
    A.R = src;
    A.H = H;
    A.splits = plan.splits;
    A.rows_split = plan.rows_split;
    A.scale_log2 = p.scale * kLog2e;
    A.sinks = sinks;
    A.out = out;
    A.part_o = part_o;
    A.part_ml = part_ml;
    A.status = status;
    A.early_q = early_q ? 1 : 0;
    if (raw_ml && plan.splits == 1) {
        // one split: the kernel writes the partial straight to the caller's buffers
        A.raw = 1;
        A.part_o = out;
        A.part_ml = raw_ml;
    }
    const size_t smem = attention_tc_smem_bytes();
    // dparts CTAs per (row split, head group), each owning 4 / dparts of the
    // output's 128-column tiles
    void (*kern)(const CUtensorMap, const TcParams) =
        plan.dparts == 4 ? attention_tc_kernel<1> : plan.dparts == 2 ? attention_tc_kernel<2> : attention_tc_kernel<4>;
    cudaError_t e = set_kernel_smem(kern, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(plan.splits, ((H + kHG - 1) / kHG) * plan.dparts, T);
    e = launch_pdl(kern, grid, dim3(kTcThreads), smem, lc.stream, tq, A);
    if (e != cudaSuccess || plan.splits == 1) return e;
    if (plan.splits > kMaxSplits) return cudaErrorInvalidValue;
    A.po_t = static_cast<int64_t>(plan.splits) * H * kHD;
    A.po_s = static_cast<int64_t>(H) * kHD;
    A.ml_t = static_cast<int64_t>(plan.splits) * H * 2;
    A.ml_s = static_cast<int64_t>(H) * 2;
    A.raw_ml = raw_ml;
    const CombShape cs = comb_shape(plan.splits, static_cast<int64_t>(H) * T, lc.sm_count);
    e = set_kernel_smem(cs.kernel, 0);
    if (e != cudaSuccess) return e;
    return launch_pdl(cs.kernel, dim3(H, T, cs.parts), dim3(cs.threads), 0, lc.stream, A);
}

cudaError_t launch_partials_combine(const Launch &lc, int32_t P, int32_t T, int32_t H,
                                    const float *part_o, const float *part_ml, const float *sinks,
                                    float *out, int32_t *status) {
    if (T <= 0) return cudaSuccess;
    if (P < 1 || P > kMaxSplits) return cudaErrorInvalidValue;
    TcParams A{};
    A.H = H;
    A.splits = P;
    A.sinks = sinks;
    A.out = out;
    A.part_o = const_cast<float *>(part_o);
    A.part_ml = const_cast<float *>(part_ml);
    A.status = status;
    A.po_t = static_cast<int64_t>(H) * kHD;
    A.po_s = static_cast<int64_t>(T) * H * kHD;
    A.ml_t = static_cast<int64_t>(H) * 2;
    A.ml_s = static_cast<int64_t>(T) * H * 2;
    const CombShape cs = comb_shape(P, static_cast<int64_t>(H) * T, lc.sm_count);
    cudaError_t e = set_kernel_smem(cs.kernel, 0);
    if (e != cudaSuccess) return e;
    return launch_pdl(cs.kernel, dim3(H, T, cs.parts), dim3(cs.threads), 0, lc.stream, A);
}

}  // namespace csa
