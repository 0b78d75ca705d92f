// csa_noalloc.cu -- csa_topk_noalloc: the top-k with its scratch in a
// file-scope device array instead of a caller-provided workspace.
//
// For callers that cannot allocate device memory at all (an engine whose
// memory planner owns the whole device, firmware-style hosts with a fixed
// memory map, plug-ins that may not touch the allocator).  The scratch lives
// in g_topk_scratch below: every GPU that loads this library holds it until
// the process exits, whether or not the entry point is ever called.
#include <mutex>

#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

// Limits of the no-allocation top-k (the scratch is sized for them): the
// top-k runs one CTA per token here, which needs only each token's state
// (histogram and counters), kStateWords words per token.
constexpr int kNoAllocMaxTokens = 16;
constexpr size_t kNoAllocBytes = size_t(kNoAllocMaxTokens) * kStateWords * 4;

// 16 x 16640 bytes = 260 KiB per device.
static __device__ __align__(256) uint8_t g_topk_scratch[kNoAllocBytes];

// Device address of g_topk_scratch, looked up once per device.  In host code
// the name g_topk_scratch is only a host-side stand-in, never a device address.
static void *g_scratch_ptr[64];
static std::mutex g_scratch_mu;

static cudaError_t scratch_address(int dev, void **out) {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_topk_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace csa

using namespace csa;

extern "C" csa_status_t csa_topk_noalloc(const csa_layout_t *layout, const csa_params_t *params,
                                         const float *scores, int64_t ld_scores, int32_t *idx,
                                         int32_t *n_sel, int32_t *dev_status, void *stream) {
    // the same checks, in the same order, as csa_topk; only the token limit
    // of the fixed scratch is this entry point's own
    csa_status_t st = check_params(params);
    if (st != CSA_OK) return st;
    st = check_layout(layout, params, false);
    if (st != CSA_OK) return st;
    if (layout->num_tokens == 0) return CSA_OK;
    if (!scores || !idx || !n_sel || !dev_status) return CSA_ERR_INVALID_ARGUMENT;
    if (ld_scores < layout->max_comp_rows || ld_scores < 1) return CSA_ERR_CAPACITY;
    // beyond the static scratch: refuse instead of overrunning it
    if (layout->num_tokens > kNoAllocMaxTokens) return CSA_ERR_CAPACITY;

    int sms = 0, dev = 0;
    st = current_device(&sms);
    if (st != CSA_OK) return st;
    if (cudaGetDevice(&dev) != cudaSuccess) return CSA_ERR_CUDA;
    void *base = nullptr;
    if (scratch_address(dev, &base) != cudaSuccess) return CSA_ERR_CUDA;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *b = static_cast<uint8_t *>(base);
    // The per-token histogram and counters must start at zero; the array keeps
    // whatever the previous call (or an interrupted one) left, so clear them.
    const size_t state = size_t(layout->num_tokens) * kStateWords * 4;
    if (cudaMemsetAsync(b, 0, state, s) != cudaSuccess) return CSA_ERR_CUDA;
    TopkWs tw{reinterpret_cast<uint32_t *>(b), nullptr, nullptr};
    Launch lc{s, sms};
    return launch_topk(lc, *layout, *params, scores, ld_scores, tw, false, idx, n_sel,
                       dev_status) == cudaSuccess
               ? CSA_OK
               : CSA_ERR_CUDA;
}
