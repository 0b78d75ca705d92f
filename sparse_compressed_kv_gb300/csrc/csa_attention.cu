// csa_attention.cu -- mixed gather and shared-KV multi-query attention.
//
// Rows attended by token t ("ARCHITECTURE & MEMORY AUDIT -- 1M-context
// viability", D3 and D5; "PART A -- Next Session Clues", section 3): the
// selected compressed rows in index order, then the sliding-window rows
// oldest first, both kept where they overlap.  Each 512-wide row is the key
// and the value of every query head (shared-KV MQA).
//
// Attention is a split-KV flash decode.  A CTA owns one token, 16 query heads
// and a contiguous range of rows, which it walks in chunks of 32 rows: the
// rows are fetched with 16-byte cp.async (straight from the compressed cache
// by index and from the window ring in fused mode, "1M-context viability",
// M5), QK^T and PV run on mma.sync bf16 tensor-core tiles with f32
// accumulation, and the softmax is online across chunks with warp-shuffle
// reductions.  Each row is read once for all 16 heads of the CTA.  With 2 to
// 8 splits per token, the splits run as one thread-block cluster that merges
// their partial (m, l, O) through distributed shared memory with log-sum-exp
// weights and writes the output.  With more, each split writes its partial
// to the workspace and a combine kernel merges them the same way.  (The merge
// also handles clusters that cover part of a token, one partial per cluster;
// the plan does not use that, as an on-chip merge of partials is no faster
// than a pass through L2.)
#include <math.h>

#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

constexpr int kAttnThreads = 256;  // 8 warps
constexpr int kRowBytes = kHD * 2;  // 1 KiB
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSplits = 64;   // attention splits per token (the plan never exceeds it)
constexpr int kCombineParts = 4;  // combine CTAs per (token, head): 128 columns each
constexpr int kMaxCluster = 8;    // attention CTAs per cluster (portable limit)

// Row count of token t and the address of its row j (nullptr: skipped row).
struct TokRows {
    int32_t len;
    int32_t n_sel;
    int64_t first;  // first window position (fused)
    int64_t n_vis;
    int64_t off;
    int b;
    int bad;
};

__device__ __forceinline__ TokRows token_rows(const RowSource &R, int t) {
    TokRows r;
    r.n_sel = 0;
    r.first = 0;
    r.n_vis = 0;
    r.off = 0;
    r.b = 0;
    r.bad = 0;
    if (R.fused == kRowsGathered) {
        int32_t len = R.kv_len[t];
        if (len < 0 || len > R.rows_per_token) {
            r.bad = CSA_DEV_BAD_LENGTH;
            len = len < 0 ? 0 : R.rows_per_token;
        }
        r.len = len;
        return r;
    }
    // the selection count does not depend on the layout: load it alongside
    const int32_t ns_sel = R.fused == kRowsSelected ? R.n_sel[t] : 0;
    TokenView v = token_view(R.L, R.ratio, t);
    r.bad = v.bad;
    if (v.bad & CSA_DEV_BAD_LAYOUT) {
        r.len = 0;
        return r;
    }
    int32_t ns;
    if (R.fused == kRowsAllVisible) {
        ns = static_cast<int32_t>(v.n_vis);   // every visible block, in index order
    } else {
        ns = ns_sel;
        if (ns < 0 || ns > R.top_k) {
            r.bad |= CSA_DEV_BAD_LENGTH;
            ns = ns < 0 ? 0 : R.top_k;
        }
    }
    r.n_sel = ns;
    r.first = window_first(v.pos, R.window);
    r.n_vis = v.n_vis;
    r.off = v.off;
    r.b = v.b;
    r.len = ns + static_cast<int32_t>(v.pos - r.first + 1);
    return r;
}

// Compressed-cache index of selected row j (j < top_k; padding entries past
// the token's selection count hold -1 and are never used).  It needs no
// token record, so a caller may load it before the record arrives.
__device__ __forceinline__ int32_t sel_index(const RowSource &R, int t, int j) {
    if (R.fused == kRowsAllVisible) return j;
    if (R.fused == kRowsSelected && j < R.top_k) return R.idx[static_cast<int64_t>(t) * R.top_k + j];
    return 0;
}

// Address of row j given its preloaded selection index s (used when j < n_sel).
__device__ __forceinline__ const __nv_bfloat16 *row_ptr_at(const RowSource &R, const TokRows &tr,
                                                            int t, int j, int32_t s, int *bad) {
    if (R.fused == kRowsGathered)
        return static_cast<const __nv_bfloat16 *>(R.kv_buf) +
               (static_cast<int64_t>(t) * R.rows_per_token + j) * kHD;
    if (j < tr.n_sel) {
        if (s < 0 || s >= tr.n_vis) {
            *bad |= CSA_DEV_BAD_INDEX;
            return nullptr;
        }
        return static_cast<const __nv_bfloat16 *>(R.comp_kv) + (tr.off + s) * kHD;
    }
    const int64_t x = tr.first + (j - tr.n_sel);
    if (x < R.L.swa_first_pos[tr.b]) {
        *bad |= CSA_DEV_MISSING_SWA;
        return nullptr;
    }
    const int64_t slot = x % R.L.swa_cap;
    return static_cast<const __nv_bfloat16 *>(R.L.swa_kv) +
           (static_cast<int64_t>(tr.b) * R.L.swa_cap + slot) * kHD;
}

__device__ __forceinline__ const __nv_bfloat16 *row_ptr(const RowSource &R, const TokRows &tr,
                                                         int t, int j, int *bad) {
    const int32_t s = (R.fused != kRowsGathered && j < tr.n_sel) ? sel_index(R, t, j) : 0;
    return row_ptr_at(R, tr, t, j, s, bad);
}

// ---------------------------------------------------------------- gather

__global__ void __launch_bounds__(256) gather_kernel(const RowSource R, __nv_bfloat16 *kv_buf,
                                                     int32_t *kv_len, int32_t *status) {
    pdl_wait();
    pdl_launch_dependents();
    const int t = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = blockIdx.x * 8 + warp;
    const TokRows tr = token_rows(R, t);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        kv_len[t] = tr.len;
        raise_status(status, tr.bad);
    }
    if (j < tr.len) {
        int bad = 0;
        const __nv_bfloat16 *src = row_ptr(R, tr, t, j, &bad);
        uint4 *dst = reinterpret_cast<uint4 *>(kv_buf + (static_cast<int64_t>(t) * R.rows_per_token + j) * kHD);
        if (src) {
            const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
            const uint4 a = __ldg(s4 + lane), b = __ldg(s4 + lane + 32);
            dst[lane] = a;
            dst[lane + 32] = b;
        } else {
            const uint4 z = make_uint4(0, 0, 0, 0);
            dst[lane] = z;
            dst[lane + 32] = z;
            if (lane == 0) raise_status(status, bad);
        }
    }
}

// ---------------------------------------------------------------- attention

struct AttnParams {
    RowSource R;
    int32_t H;
    int32_t splits;
    int32_t rows_split;
    int32_t cluster;         // CTAs per cluster along the splits (divides splits)
    float scale_log2;        // scale * log2(e)
    const __nv_bfloat16 *q;  // [T][H][512]
    const float *sinks;      // [H] or null
    float *out;              // [T][H][512]
    float *part_o;           // [T][splits][H][512]
    float *part_ml;          // [T][splits][H][2]  (m in log2 units, l)
    int32_t *status;
    int32_t early_q;         // q may be read before the grid-dependency wait: the
                             // launching chain's first kernel already waited on
                             // whatever produced the caller's inputs
};

struct AttnSmem {
    __nv_bfloat16 q[kHeadGroup * kHD];              // 16 KiB, 16-byte chunks xor-swizzled by row
    __nv_bfloat16 rows[2][kAttnChunk * kHD];        // 2 x 32 KiB, same swizzle; rows[0]
                                                    // stages the f32 output at the end
    const __nv_bfloat16 *ptr[2][kAttnChunk];
    float s[2][kHeadGroup][kAttnChunk];             // QK^T of the chunk, one per half of hd
    // probabilities as two bf16 terms, p = hi + lo (padded rows): the PV product
    // keeps ~16 bits of each weight instead of bf16's 8
    __nv_bfloat16 p[2][kHeadGroup][kAttnChunk + 8];
    float m[kHeadGroup], l[kHeadGroup], alpha[kHeadGroup];
    float wc[8][kHeadGroup];    // cluster merge: weight of each rank's partial per head
    float fin[kHeadGroup];      // cluster merge: output scale per head
    float mc[kHeadGroup], lc[kHeadGroup];
    TokRows tr;
};

// 16-byte chunk c of row r lives at chunk (c ^ (r & 7)): ldmatrix of 8 rows at
// one column then touches 8 distinct bank groups.
__device__ __forceinline__ uint32_t swz(int r, int chunk) {
    return static_cast<uint32_t>(r * kRowBytes + ((chunk ^ (r & 7)) << 4));
}

// 32 x 64 sixteen-byte copies of the chunk whose row addresses are in S.ptr[buf]
// (null rows are zero-filled and masked later).
__device__ __forceinline__ void issue_chunk_copies(AttnSmem &S, const RowSource &R, int buf) {
    uint8_t *base = reinterpret_cast<uint8_t *>(S.rows[buf]);
    const void *dummy = R.comp_kv ? R.comp_kv : R.kv_buf;
    for (int i = threadIdx.x; i < kAttnChunk * 64; i += kAttnThreads) {
        const int r = i >> 6, c = i & 63;
        const __nv_bfloat16 *src = S.ptr[buf][r];
        cp_async16(base + swz(r, c), src ? static_cast<const void *>(src + c * 8) : dummy,
                   src != nullptr);
    }
    cp_async_commit();
}

// Row addresses of the chunk starting at r0 (warp 0), then its copies.
__device__ __forceinline__ void issue_chunk(AttnSmem &S, const RowSource &R, int t, int buf,
                                            int r0, int r_end, int *bad) {
    if (threadIdx.x < kAttnChunk) {
        const int j = r0 + threadIdx.x;
        S.ptr[buf][threadIdx.x] = j < r_end ? row_ptr(R, S.tr, t, j, bad) : nullptr;
    }
    __syncthreads();
    issue_chunk_copies(S, R, buf);
}

// Merge of the cluster's partials (every CTA has staged its unnormalised O in
// rows[0], f32 [16][512] with 16-byte chunks xor-swizzled by head, and its m,
// l per head).  Rank r combines chunk range r/C of the 16 x 128 chunks from
// every rank's staging area; the result is the cluster's partial in slot
// split / C, or, when one cluster covers all of the token's splits (the
// plan's choice), the normalised output (with the sink in the denominator).
__device__ __forceinline__ void cluster_merge(const AttnParams &A, AttnSmem &S, int t, int split,
                                           int h0, int bad) {
    const int C = A.cluster;
    const uint32_t rank = cluster_ctarank();
    const bool final = C == A.splits;
    cluster_sync_all();   // every rank's staging, m and l are written
    if (threadIdx.x < kHeadGroup) {
        const int h = threadIdx.x;
        // every remote load is issued before any is used: the loads are
        // ordered, so a use between them would serialise the round trips
        float mr[kMaxCluster], lr[kMaxCluster];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
            mr[r] = -INFINITY;
            lr[r] = 0.f;
            if (r < C) {
                mr[r] = ld_cluster_f32(cluster_map(&S.m[h], r));
                lr[r] = ld_cluster_f32(cluster_map(&S.l[h], r));
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) M = fmaxf(M, mr[r]);
        float L = 0.f;
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
            const float w = mr[r] == -INFINITY ? 0.f : exp2f(mr[r] - M);
            if (r < C) S.wc[r][h] = w;
            L += w * lr[r];
        }
        S.mc[h] = M;
        S.lc[h] = L;
        if (final) {
            // out = O / (L + 2^(sink - M)), scaled against max(M, sink)
            const float sk = A.sinks ? A.sinks[h0 + h] * kLog2e : -INFINITY;
            const float Mall = fmaxf(M, sk);
            const float sM = M == -INFINITY ? 0.f : exp2f(M - Mall);
            const float z = L * sM + (A.sinks ? exp2f(sk - Mall) : 0.f);
            S.fin[h] = z > 0.f ? sM / z : 0.f;
        } else {
            S.fin[h] = 1.f;
        }
    }
    __syncthreads();
    const float *stg = reinterpret_cast<const float *>(S.rows[0]);
    constexpr int kChunks = kHeadGroup * (kHD / 4);
    const int e0 = static_cast<int>((static_cast<int64_t>(kChunks) * rank) / C);
    const int e1 = static_cast<int>((static_cast<int64_t>(kChunks) * (rank + 1)) / C);
    const int64_t slot = split / C;
    const int64_t pbase = (static_cast<int64_t>(t) * A.splits + slot) * A.H + h0;
    float *dst = final ? A.out + (static_cast<int64_t>(t) * A.H + h0) * kHD : A.part_o + pbase * kHD;
    const bool vec = (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
    for (int e = e0 + threadIdx.x; e < e1; e += kAttnThreads) {
        const int h = e / (kHD / 4), ch = e % (kHD / 4);
        const float *src = stg + h * kHD + ((ch ^ (h & 7)) << 2);
        float4 v[kMaxCluster];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r)
            if (r < C) v[r] = ld_cluster_v4f32(cluster_map(src, r));
        // a rank without rows (weight 0) staged nothing: its values are skipped
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) {
            if (r < C) {
                const float w = S.wc[r][h];
                if (w != 0.f) {
                    acc.x += w * v[r].x;
                    acc.y += w * v[r].y;
                    acc.z += w * v[r].z;
                    acc.w += w * v[r].w;
                }
            }
        }
        const float f = S.fin[h];
        acc.x *= f;
        acc.y *= f;
        acc.z *= f;
        acc.w *= f;
        float *d = dst + h * kHD + ch * 4;
        if (vec) {
            *reinterpret_cast<float4 *>(d) = acc;
        } else {
            d[0] = acc.x;
            d[1] = acc.y;
            d[2] = acc.z;
            d[3] = acc.w;
        }
    }
    if (!final && rank == 0 && threadIdx.x < kHeadGroup) {
        A.part_ml[(pbase + threadIdx.x) * 2 + 0] = S.mc[threadIdx.x];
        A.part_ml[(pbase + threadIdx.x) * 2 + 1] = S.lc[threadIdx.x];
    }
    cluster_sync_all();   // no CTA leaves while another still reads its shared memory
    raise_status(A.status, bad);
}

__global__ void __launch_bounds__(kAttnThreads) attention_kernel(const AttnParams A) {
    extern __shared__ uint8_t smem_raw[];
    AttnSmem &S = *reinterpret_cast<AttnSmem *>(align_smem<128>(smem_raw));
    const int split = blockIdx.x, hg = blockIdx.y, t = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;

    const int h0 = hg * kHeadGroup;
    auto load_q = [&]() {
        const __nv_bfloat16 *qg = A.q + (static_cast<int64_t>(t) * A.H + h0) * kHD;
        uint8_t *qs = reinterpret_cast<uint8_t *>(S.q);
        for (int i = threadIdx.x; i < kHeadGroup * 64; i += kAttnThreads) {
            const int r = i >> 6, ch = i & 63;
            cp_async16(qs + swz(r, ch), qg + r * kHD + ch * 8, true);
        }
        cp_async_commit();
    };
    if (A.early_q) load_q();
    pdl_wait();
    pdl_launch_dependents();

    // Warp 0 resolves the token's rows and the first chunk's row addresses.
    // The chunk's selection indices, the selection count and the layout
    // record are independent loads, issued together; only the sequence's
    // offsets wait for the record.
    const int r_begin = split * A.rows_split;
    int bad = 0;
    if (warp == 0) {
        const int j = r_begin + lane;
        const int32_t s_pre = sel_index(A.R, t, j);
        const TokRows tr = token_rows(A.R, t);
        if (lane == 0) S.tr = tr;
        const int re = min(tr.len, r_begin + A.rows_split);
        S.ptr[0][lane] = j < re ? row_ptr_at(A.R, tr, t, j, s_pre, &bad) : nullptr;
        if (lane == 0 && split == 0 && hg == 0) bad |= tr.bad;
    }
    __syncthreads();
    const int len = S.tr.len;
    const int r_end = min(len, r_begin + A.rows_split);

    const bool empty = r_begin >= r_end;
    if (empty) {
        if (A.early_q) cp_async_wait<0>();
        if (A.cluster == 1) {
            // nothing here; with one split this CTA still owns the output (zeros)
            if (A.splits == 1) {
                float *o = A.out + (static_cast<int64_t>(t) * A.H + h0) * kHD;
                for (int i = threadIdx.x; i < kHeadGroup * kHD; i += kAttnThreads) o[i] = 0.f;
            }
            raise_status(A.status, bad);
            return;
        }
        // in a cluster the CTA still takes part in the merge, with no rows
        if (threadIdx.x < kHeadGroup) {
            S.m[threadIdx.x] = -INFINITY;
            S.l[threadIdx.x] = 0.f;
        }
        __syncthreads();
        cluster_merge(A, S, t, split, h0, bad);
        return;
    }
    if (!A.early_q) load_q();
    if (threadIdx.x < kHeadGroup) {
        S.m[threadIdx.x] = -INFINITY;
        S.l[threadIdx.x] = 0.f;
    }
    const int nchunks = (r_end - r_begin + kAttnChunk - 1) / kAttnChunk;
    issue_chunk_copies(S, A.R, 0);

    // Output columns 64w .. 64w+63 of all 16 heads: 8 n8 tiles.
    float o[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    const uint32_t q_base = smem_addr(S.q);
    const uint32_t p_base = smem_addr(&S.p[0][0][0]);
    constexpr uint32_t kPLoOffset = kHeadGroup * (kAttnChunk + 8) * 2;   // bytes from hi to lo

    for (int ci = 0; ci < nchunks; ++ci) {
        const int buf = ci & 1;
        const int r0 = r_begin + ci * kAttnChunk;
        if (ci + 1 < nchunks) {
            issue_chunk(S, A.R, t, buf ^ 1, r0 + kAttnChunk, r_end, &bad);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint32_t rows_base = smem_addr(S.rows[buf]);

        // ---- QK^T: warp w owns rows 8(w%4) .. +7 of the chunk, all 16 heads,
        // and half w/4 of the 512 dimensions; the halves add in the softmax
        {
            float sacc[4] = {0.f, 0.f, 0.f, 0.f};
            float sacc2[4] = {0.f, 0.f, 0.f, 0.f};
            const int rr = (warp & 3) * 8 + (lane & 7);
            const int qr = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int kb = (warp >> 2) * (kHD / 32);
#pragma unroll 4
            for (int kk = 0; kk < kHD / 32; kk += 2) {
                const int k = kb + kk;
                uint32_t a0, a1, a2, a3, e0, e1, e2, e3, b0, b1, b2, b3;
                ldsm_x4(q_base + swz(qr, k * 2 + (lane >> 4)), a0, a1, a2, a3);
                ldsm_x4(q_base + swz(qr, (k + 1) * 2 + (lane >> 4)), e0, e1, e2, e3);
                ldsm_x4(rows_base + swz(rr, k * 2 + (lane >> 3)), b0, b1, b2, b3);
                mma_bf16_16816(sacc, a0, a1, a2, a3, b0, b1);
                mma_bf16_16816(sacc2, e0, e1, e2, e3, b2, b3);
            }
            // c-fragment: heads g, g+8; rows 2c, 2c+1 of this warp's 8
            float(&sp)[kHeadGroup][kAttnChunk] = S.s[warp >> 2];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sp[g + (e >> 1) * 8][(warp & 3) * 8 + 2 * c + (e & 1)] = sacc[e] + sacc2[e];
        }
        __syncthreads();

        // ---- online softmax: warp w owns heads 2w, 2w+1, lane = row
        {
            const bool valid = r0 + lane < r_end && S.ptr[buf][lane] != nullptr;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int h = warp * 2 + hh;
                const float x = valid ? (S.s[0][h][lane] + S.s[1][h][lane]) * A.scale_log2 : -INFINITY;
                float mx = x;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const float m_old = S.m[h];
                const float m_new = fmaxf(m_old, mx);
                const float p = (x == -INFINITY) ? 0.f : exp2f(x - m_new);
                float sum = p;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
                const float alpha = (m_old == -INFINITY) ? 0.f : exp2f(m_old - m_new);
                const __nv_bfloat16 p_hi = __float2bfloat16_rn(p);
                S.p[0][h][lane] = p_hi;
                S.p[1][h][lane] = __float2bfloat16_rn(p - __bfloat162float(p_hi));
                __syncwarp();
                if (lane == 0) {
                    S.l[h] = S.l[h] * alpha + sum;
                    S.m[h] = m_new;
                    S.alpha[h] = alpha;
                }
            }
        }
        __syncthreads();

        // ---- O = alpha O + P V: warp w owns columns 64w .. 64w+63
        {
            const float al0 = S.alpha[g], al1 = S.alpha[g + 8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                o[i][0] *= al0;
                o[i][1] *= al0;
                o[i][2] *= al1;
                o[i][3] *= al1;
            }
#pragma unroll
            for (int ks = 0; ks < kAttnChunk / 16; ++ks) {
                uint32_t a0, a1, a2, a3, l0, l1, l2, l3;
                const int pr = (lane & 7) + ((lane >> 3) & 1) * 8;
                const int pc = ks * 16 + (lane >> 4) * 8;
                const uint32_t pa = p_base + static_cast<uint32_t>((pr * (kAttnChunk + 8) + pc) * 2);
                ldsm_x4(pa, a0, a1, a2, a3);
                ldsm_x4(pa + kPLoOffset, l0, l1, l2, l3);
                const int vr = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    const int chunk = (warp * 64 + np * 16) / 8 + (lane >> 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_trans(rows_base + swz(vr, chunk), b0, b1, b2, b3);
                    mma_bf16_16816(o[2 * np], a0, a1, a2, a3, b0, b1);
                    mma_bf16_16816(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
                    mma_bf16_16816(o[2 * np], l0, l1, l2, l3, b0, b1);
                    mma_bf16_16816(o[2 * np + 1], l0, l1, l2, l3, b2, b3);
                }
            }
        }
        __syncthreads();
    }

    // ---- write: the fragments go through shared memory (rows[0], free now:
    // the last chunk's copies were waited for and its PV is done), 16-byte
    // chunks of each head's 512 floats xor-swizzled by head, and leave as
    // contiguous 16-byte stores (one head row of 2 KiB per 4 warp stores)
    float sc0 = 1.f, sc1 = 1.f;
    if (A.splits == 1 && A.cluster == 1) {
        float z0 = S.l[g], z1 = S.l[g + 8];
        if (A.sinks) {
            z0 += exp2f(A.sinks[h0 + g] * kLog2e - S.m[g]);
            z1 += exp2f(A.sinks[h0 + g + 8] * kLog2e - S.m[g + 8]);
        }
        sc0 = z0 > 0.f ? 1.f / z0 : 0.f;
        sc1 = z1 > 0.f ? 1.f / z1 : 0.f;
    }
    float *stg = reinterpret_cast<float *>(S.rows[0]);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int col = warp * 64 + i * 8 + 2 * c;
        const int ch = col >> 2, wi = col & 3;
        *reinterpret_cast<float2 *>(stg + g * kHD + ((ch ^ (g & 7)) << 2) + wi) =
            make_float2(o[i][0] * sc0, o[i][1] * sc0);
        *reinterpret_cast<float2 *>(stg + (g + 8) * kHD + ((ch ^ (g & 7)) << 2) + wi) =
            make_float2(o[i][2] * sc1, o[i][3] * sc1);
    }
    if (A.cluster > 1) {
        __syncthreads();
        cluster_merge(A, S, t, split, h0, bad);
        return;
    }
    const int64_t pbase = (static_cast<int64_t>(t) * A.splits + split) * A.H + h0;
    if (A.splits > 1 && threadIdx.x < kHeadGroup) {
        A.part_ml[(pbase + threadIdx.x) * 2 + 0] = S.m[threadIdx.x];
        A.part_ml[(pbase + threadIdx.x) * 2 + 1] = S.l[threadIdx.x];
    }
    __syncthreads();
    float *dst = A.splits == 1 ? A.out + (static_cast<int64_t>(t) * A.H + h0) * kHD
                               : A.part_o + pbase * kHD;
    const bool vec = (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
    for (int e = threadIdx.x; e < kHeadGroup * (kHD / 4); e += kAttnThreads) {
        const int h = e / (kHD / 4), ch = e % (kHD / 4);
        const float4 v = *reinterpret_cast<const float4 *>(stg + h * kHD + ((ch ^ (h & 7)) << 2));
        float *d = dst + h * kHD + ch * 4;
        if (vec) {
            *reinterpret_cast<float4 *>(d) = v;
        } else {
            d[0] = v.x;
            d[1] = v.y;
            d[2] = v.z;
            d[3] = v.w;
        }
    }
    raise_status(A.status, bad);
}

// out[t,h,:] = sum_s 2^(m_s - M) O_s / (sum_s 2^(m_s - M) l_s [+ 2^(sink*log2e - M)])
// Runs only when a token's splits span more than one cluster, and then the
// plan makes every cluster a single CTA: one partial per split.
__global__ void __launch_bounds__(64) combine_kernel(const AttnParams A) {
    pdl_wait();
    pdl_launch_dependents();
    const int h = blockIdx.x, t = blockIdx.y;
    const int c0 = blockIdx.z * (kHD / kCombineParts);   // this CTA's 128 columns
    __shared__ float wgt[64];
    __shared__ float inv_z;
    __shared__ int nsp_s;
    // one thread reads the token's record (every thread of every CTA
    // reading the same lines would queue their requests) and shares it
    if (threadIdx.x == 0) {
        const TokRows tr = token_rows(A.R, t);
        nsp_s = min(A.splits, (tr.len + A.rows_split - 1) / A.rows_split);
    }
    __syncthreads();
    const int nsp = nsp_s;
    float *o = A.out + (static_cast<int64_t>(t) * A.H + h) * kHD;
    if (nsp <= 0) {
        for (int i = threadIdx.x; i < kHD / kCombineParts; i += blockDim.x) o[c0 + i] = 0.f;
        return;
    }
    // Issue every partial load first (they do not depend on the weights),
    // then the (m, l) of each split, then combine: one round trip.
    const int d = c0 + threadIdx.x * 2;   // 64 threads x 2 columns
    const float *pb = A.part_o + (static_cast<int64_t>(t) * A.splits * A.H + h) * kHD + d;
    const int64_t pstride = static_cast<int64_t>(A.H) * kHD;
    float2 v[kMaxSplits];
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s)
        if (s < nsp) v[s] = __ldcg(reinterpret_cast<const float2 *>(pb + s * pstride));
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        // each lane holds (m, l) of splits lane and lane + 32 (at most 64 splits)
        float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
        const float *mlb = A.part_ml + (static_cast<int64_t>(t) * A.splits * A.H + h) * 2;
        const int64_t stride = static_cast<int64_t>(A.H) * 2;
        if (lane < nsp) {
            const float2 x = __ldcg(reinterpret_cast<const float2 *>(mlb + lane * stride));
            m0 = x.x;
            l0 = x.y;
        }
        if (lane + 32 < nsp) {
            const float2 x = __ldcg(reinterpret_cast<const float2 *>(mlb + (lane + 32) * stride));
            m1 = x.x;
            l1 = x.y;
        }
        float M = fmaxf(m0, m1);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float sink = A.sinks ? A.sinks[h] * kLog2e : -INFINITY;
        const float Mall = fmaxf(M, sink);
        const float w0 = m0 == -INFINITY ? 0.f : exp2f(m0 - Mall);
        const float w1 = m1 == -INFINITY ? 0.f : exp2f(m1 - Mall);
        if (lane < nsp) wgt[lane] = w0;
        if (lane + 32 < nsp) wgt[lane + 32] = w1;
        float z = w0 * l0 + w1 * l1;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        if (lane == 0) {
            if (A.sinks) z += exp2f(sink - Mall);
            inv_z = z > 0.f ? 1.f / z : 0.f;
        }
    }
    __syncthreads();
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s) {
        if (s < nsp) {
            const float w = wgt[s];
            acc.x += w * v[s].x;
            acc.y += w * v[s].y;
        }
    }
    const float iz = inv_z;
    *reinterpret_cast<float2 *>(o + d) = make_float2(acc.x * iz, acc.y * iz);
}

cudaError_t launch_gather(const Launch &lc, const RowSource &src, int32_t T, void *kv_buf,
                          int32_t *kv_len, int32_t *status) {
    if (T <= 0) return cudaSuccess;
    const int rows = src.rows_per_token;
    dim3 grid((rows + 7) / 8, T);
    cudaError_t e = set_kernel_smem(gather_kernel, 0);
    if (e != cudaSuccess) return e;
    return launch_pdl(gather_kernel, grid, dim3(256), 0, lc.stream, src,
                      static_cast<__nv_bfloat16 *>(kv_buf), kv_len, status);
}

cudaError_t launch_attention(const Launch &lc, const RowSource &src, int32_t T,
                             const csa_params_t &p, const WsPlan &plan, const void *q,
                             const float *sinks, float *out, float *part_o, float *part_ml,
                             int32_t *status, bool early_q) {
    if (T <= 0) return cudaSuccess;
    AttnParams A;
    A.R = src;
    A.H = p.n_heads;
    A.splits = plan.splits;
    A.rows_split = plan.rows_split;
    A.cluster = plan.attn_cluster;
    A.scale_log2 = p.scale * kLog2e;
    A.q = static_cast<const __nv_bfloat16 *>(q);
    A.sinks = sinks;
    A.out = out;
    A.part_o = part_o;
    A.part_ml = part_ml;
    A.status = status;
    A.early_q = early_q ? 1 : 0;
    const size_t smem = sizeof(AttnSmem) + 128;
    cudaError_t e = set_kernel_smem(attention_kernel, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(plan.splits, p.n_heads / kHeadGroup, T);
    e = launch_pdl_cluster(attention_kernel, grid, dim3(kAttnThreads), smem, lc.stream,
                           plan.attn_cluster, A);
    if (e != cudaSuccess || plan.splits == plan.attn_cluster) return e;
    e = set_kernel_smem(combine_kernel, 0);
    if (e != cudaSuccess) return e;
    return launch_pdl(combine_kernel, dim3(p.n_heads, T, kCombineParts), dim3(64), 0, lc.stream,
                      A);
}

}  // namespace csa
