// csa_attention.cu -- the rows a token attends, gathered into one buffer.
//
// Rows attended by token t ("ARCHITECTURE & MEMORY AUDIT -- 1M-context
// viability", D3 and D5; "PART A -- Next Session Clues", section 3): the
// selected compressed rows in index order, then the sliding-window rows
// oldest first, both kept where they overlap.  The gathered layout feeds
// csa_sparse_mqa_decode; the attention kernels themselves (which also read
// the rows in place by index) are in csa_attention_tc.cu.
#include <math.h>

#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

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

}  // namespace csa
