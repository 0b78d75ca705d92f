// csa_fp4.cu -- the FP4 indexer key cache: bf16 keys -> MXFP4 rows.
//
// ("ARCHITECTURE & MEMORY AUDIT -- Post-probe rewrite", C4, and
// "ARCHITECTURE & MEMORY AUDIT -- 1M-context viability", M1: the indexer keys
// are cached in FP4.)  The pages fix no format; this library reads it as OCP
// MXFP4: e2m1 elements, one e8m0 scale 2^(E-127) per 32 elements with
// E = floor(log2(block amax)) - 2 + 127 (clamped to 0..254, 0 for an all-zero
// block), elements rounded to the nearest e2m1 value, ties to the even code,
// saturating at 6, a zero magnitude stored as code 0.
//
// Row of one 128-wide key (80 bytes, so rows stay 16-byte aligned for TMA):
// bytes 0..63 the codes (element 2i in the low nibble of byte i, 2i+1 in the
// high nibble), bytes 64..67 the four block scales, bytes 68..79 zero.
#include "csa_device.cuh"
#include "csa_internal.h"

namespace csa {

// One warp per key row; lane l holds elements 4l .. 4l+3, so the 8 lanes of
// a quarter-warp own one 32-element block.
__global__ void __launch_bounds__(256) fp4_quantize_kernel(int64_t R, const uint16_t *k,
                                                           uint8_t *rows) {
    const int lane = threadIdx.x & 31;
    const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t r = w0; r < R; r += nw) {
        const uint2 raw = *reinterpret_cast<const uint2 *>(k + r * kIHD + lane * 4);
        float x[4];
        x[0] = __uint_as_float(raw.x << 16);
        x[1] = __uint_as_float(raw.x & 0xFFFF0000u);
        x[2] = __uint_as_float(raw.y << 16);
        x[3] = __uint_as_float(raw.y & 0xFFFF0000u);
        float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
        int E = 0;
        if (a > 0.f) E = min(254, max(0, ilogbf(a) - 2 + 127));
        uint32_t packed = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            // |x| / 2^(E-127): a power-of-two scaling, exact in f32 (a result
            // too small for f32 is below the first rounding point anyway)
            const float v = ldexpf(fabsf(x[j]), 127 - E);
            // nearest of 0, .5, 1, 1.5, 2, 3, 4, 6: at a midpoint the even
            // code wins (">" above an even code, ">=" above an odd one)
            const uint32_t mag = (v > 0.25f) + (v >= 0.75f) + (v > 1.25f) + (v >= 1.75f) +
                                 (v > 2.5f) + (v >= 3.5f) + (v > 5.0f);
            const uint32_t code = mag ? (mag | (signbit(x[j]) ? 8u : 0u)) : 0u;
            packed |= code << (4 * j);
        }
        uint8_t *row = rows + r * 80;
        reinterpret_cast<uint16_t *>(row)[lane] = static_cast<uint16_t>(packed);
        if ((lane & 7) == 0) row[64 + (lane >> 3)] = static_cast<uint8_t>(E);
        if (lane < 3) reinterpret_cast<uint32_t *>(row + 68)[lane] = 0u;
    }
}

cudaError_t launch_fp4_quantize(const Launch &lc, int64_t rows, const void *k_idx, void *k_fp4) {
    if (rows <= 0) return cudaSuccess;
    const int64_t blocks = (rows + 7) / 8;  // eight rows (warps) per block
    const int64_t cap = static_cast<int64_t>(lc.sm_count) * 8;
    const unsigned grid = static_cast<unsigned>(blocks < cap ? blocks : cap);
    fp4_quantize_kernel<<<grid, 256, 0, lc.stream>>>(rows, static_cast<const uint16_t *>(k_idx),
                                                     static_cast<uint8_t *>(k_fp4));
    return cudaGetLastError();
}

}  // namespace csa
