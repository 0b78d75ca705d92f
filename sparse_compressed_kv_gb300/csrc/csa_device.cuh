// csa_device.cuh -- device-side building blocks of the CSA decode kernels
// (sm_103a): inline-PTX wrappers for mbarrier, TMA, tcgen05/TMEM, cp.async
// and mma.sync, plus the per-token layout rule shared by every kernel.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa.h"

namespace csa {

// Problem constants the library supports.
constexpr int kNIH = 64;        // indexer heads
constexpr int kIHD = 128;       // indexer key width
constexpr int kHD = 512;        // main row width (shared key/value)
constexpr int kTileKeys = 128;  // compressed blocks per indexer tile (MMA M)
constexpr int kMaxTopK = 2048;

// Radix digits of the top-k: 11 + 11 + 10 bits of the order-preserving key.
constexpr int kD1Bits = 11;
constexpr int kD1Bins = 1 << kD1Bits;
constexpr int kD1Shift = 32 - kD1Bits;      // 21
constexpr int kD2Bits = 11;
constexpr int kD2Bins = 1 << kD2Bits;
constexpr int kD2Shift = kD1Shift - kD2Bits;  // 10
constexpr int kD3Bins = 1 << kD2Shift;        // 1024

// Per-token top-k state at the front of the workspace: the digit-1 and
// digit-2 histograms followed by the counters, kStateWords 32-bit words per
// token.  It must be zero when a call starts; the kernel that consumes it
// zeroes it again.
constexpr int kStateWords = kD1Bins + kD2Bins + 64;  // 16640 bytes, a multiple of 256

struct TokCounters {
    uint32_t sel;     // entries appended to the "certainly selected" list
    uint32_t cand;    // entries appended to the candidate list (may exceed cap)
    uint32_t ticket;  // CTAs of this token that finished the filter pass
    uint32_t pad;
};

// ---------------------------------------------------------------- layout rule

// Token t of sequence b at position p sees blocks 0 .. n_vis-1, the blocks
// strictly preceding the block that holds p ("PART A -- Next Session Clues",
// section 3), capped by what the cache holds.
struct TokenView {
    int b;
    int64_t pos;
    int64_t off;    // first row of the sequence in k_idx / comp_kv
    int64_t n_vis;
    int bad;        // CSA_DEV_* bits (0 = consistent)
};

__device__ __forceinline__ TokenView token_view(const csa_layout_t &L, int ratio, int t) {
    TokenView v;
    v.b = 0;
    v.pos = 0;
    v.off = 0;
    v.n_vis = 0;
    v.bad = 0;
    // The sequence's offsets depend on its id.  Token t usually belongs to
    // sequence min(t, num_seqs - 1) (one token per sequence in a decode
    // batch, one sequence in a prefill chunk): its offsets are loaded in the
    // same round trip as the id and reloaded only when the guess is wrong.
    const int g = t < L.num_seqs ? t : L.num_seqs - 1;
    const int gs = g > 0 ? g : 0;
    int b = L.tok_seq[t];
    int64_t p = L.tok_pos[t];
    int64_t o0 = L.comp_off[gs], o1 = L.comp_off[gs + 1];
    if (b < 0 || b >= L.num_seqs || p < 0) {
        v.bad = CSA_DEV_BAD_LAYOUT;
        return v;
    }
    if (b != gs) {
        o0 = L.comp_off[b];
        o1 = L.comp_off[b + 1];
    }
    if (o0 < 0 || o1 < o0 || o1 > L.total_comp_rows) {
        v.bad = CSA_DEV_BAD_LAYOUT;
        return v;
    }
    int64_t n_comp = o1 - o0;
    if (n_comp > L.max_comp_rows) {
        v.bad = CSA_DEV_CAPACITY;
        n_comp = L.max_comp_rows;
    }
    int64_t pre = p / ratio;
    v.b = b;
    v.pos = p;
    v.off = o0;
    v.n_vis = pre < n_comp ? pre : n_comp;
    return v;
}

// Window of a query at position p: positions max(0, p-window+1) .. p.
__device__ __forceinline__ int64_t window_first(int64_t p, int window) {
    int64_t f = p - window + 1;
    return f < 0 ? 0 : f;
}

__device__ __forceinline__ void raise_status(int32_t *st, int bits) {
    if (bits && st) atomicOr(st, bits);
}

// Bounds checks of the build with CSA_CHECKS defined (libcsa_checks.so): an
// index inside the library that leaves its array sets CSA_DEV_CHECK in the
// status word and the access is skipped, never trapped.  In the default build
// the condition is not evaluated: every such index is in range by
// construction (the layout and argument checks come first).
#ifdef CSA_CHECKS
__device__ __forceinline__ bool csa_check(bool ok, int32_t *st) {
    if (!ok) raise_status(st, CSA_DEV_CHECK);
    return ok;
}
#define CSA_CHECK(cond, st) ::csa::csa_check((cond), (st))
#else
#define CSA_CHECK(cond, st) true
#endif

// Order-preserving map of an f32 score to u32 (larger score -> larger key);
// -0.0 is folded onto +0.0 so the two tie.
__device__ __forceinline__ uint32_t score_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------- PTX: misc

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The dynamic shared-memory array rounded up to an A-byte boundary.  The
// padding is added to the array's own pointer (not through an integer), so
// the compiler still sees a shared-memory address and emits shared loads and
// stores for what is reached through it.
template <uint32_t A>
__device__ __forceinline__ uint8_t *align_smem(uint8_t *base) {
    const uint32_t s = smem_addr(base);
    return base + (((s + (A - 1u)) & ~(A - 1u)) - s);
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.b32 %0, 1, 0, P;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// Programmatic dependent launch: wait for the preceding grid's results /
// allow the next grid to start its prologue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Arrive at a named barrier without waiting (the producer side of a
// hand-off: writes before it are visible to the threads that bar.sync on it).
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, P;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: gives up after kWaitNs of wall time (or kWaitPolls polls,
// whichever comes first), raises CSA_DEV_TIMEOUT and returns false.  No wait
// in this library depends on another grid or another GPU, so a timeout only
// fires if the hardware or a launch-shape bug stalls a pipeline.
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kWaitPolls = 1u << 28;

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int32_t *status) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1; i < kWaitPolls; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 1023u) == 0 && global_timer_ns() - t0 > kWaitNs) break;
    }
    raise_status(status, CSA_DEV_TIMEOUT);
    return false;
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled load of one box into shared memory, completing on `bar`.
// x (innermost coordinate, elements) must keep x * elem_size a multiple of 16.
// Warm L2 with one box of a tensor: nothing lands in shared memory and
// nothing waits for it.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap *m, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *m, int32_t x, int32_t y,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Orders this thread's earlier generic-proxy writes of shared memory before
// later async-proxy reads of it (TMA stores, tcgen05.mma operands).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// Global f32 store carrying an L2 eviction policy.
__device__ __forceinline__ void st_global_hint(float *ptr, float v, uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(ptr), "f"(v), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t *holder, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(holder)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand stored in the
// 128-byte swizzled layout TMA writes (8-row x 128-byte atoms, atoms of
// consecutive rows 1024 bytes apart).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);          // start address
    d |= static_cast<uint64_t>(1u) << 16;                          // leading offset (unused)
    d |= static_cast<uint64_t>((1024u >> 4) & 0x3FFFu) << 32;      // stride: 8 rows x 128 B
    d |= static_cast<uint64_t>(1u) << 46;                          // descriptor version
    d |= static_cast<uint64_t>(2u) << 61;                          // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::f16 with bf16 A/B, f32 accumulator, both
// operands K-major, shape M x N.
template <int M, int N>
__device__ __forceinline__ constexpr uint32_t idesc_bf16_f32() {
    return (1u << 4)                               // D: f32
           | (1u << 7)                             // A: bf16
           | (1u << 10)                            // B: bf16
           | (static_cast<uint32_t>(N >> 3) << 17)  // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24); // M / 16
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same with A read from tensor memory: a_tmem addresses an M x 16 slice
// of 16-bit elements, row m in TMEM lane m, elements 2j and 2j + 1 of the
// slice in column j (low half first).
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread i of the warp gets lane
// (lane base + i), columns col .. col+15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 16 consecutive 32-bit columns from registers (the inverse of
// tmem_ld16).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- cp.async / mma.sync

__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid) {
    uint32_t n = valid ? 16u : 0u;  // 0 source bytes: the 16 destination bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)),
                 "l"(src), "r"(n)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                              uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D; bf16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace csa
