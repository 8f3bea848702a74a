// q2_0_quantize_ref: the reference quantizer on the GPU, bit-exact.
//
// Source: "Llama.cpp umí dvoubitový Q2_0 i na kartách NVIDIA" (aisvetem.cz),
// section "Na běžný model to není": the scale is the block's largest |w| and
// every weight is rounded to the nearest of the four levels (q - 1) * scale.
// With |w| <= amax only -amax, 0, +amax can be nearest; the midpoints are
// +-amax/2. 2*w is exact in f32 (or overflows to +-inf, which keeps the
// order), so "2w >= amax" and "2w <= -amax" decide exactly; equality (a tie)
// goes away from zero. The stored scale is fp16(amax), round to nearest even.
// amax == 0 stores d = 0 and code 1 everywhere. Code 3 is never produced.
//
// One warp per 64-weight block: lane l owns elements 2l and 2l+1; the packed
// word w (elements 16w..16w+15, code of element 16w+i at bits 2i) is OR-reduced
// over the 8 lanes that own it; lanes 0..17 then write the block's 18 bytes
// (little-endian), so the destination may have any alignment.
#include "q2_0_device.cuh"
#include "q2_0_internal.h"

namespace q2 {

namespace {

__device__ __forceinline__ uint32_t quant_code(float w, float amax) {
    if (amax == 0.0f) return 1u;
    const float w2 = 2.0f * w;
    if (w2 >= amax) return 2u;
    if (w2 <= -amax) return 0u;
    return 1u;
}

__global__ void __launch_bounds__(256) quantize_kernel(const float *__restrict__ src,
                                                       uint8_t *__restrict__ dst, int64_t n_blocks) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5;
    const int64_t n_warps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    for (int64_t b = warp; b < n_blocks; b += n_warps) {
        const float *x = src + b * 64;
        const float w0 = x[2 * lane];
        const float w1 = x[2 * lane + 1];
        float a = fmaxf(fabsf(w0), fabsf(w1));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const uint32_t c0 = quant_code(w0, a);
        const uint32_t c1 = quant_code(w1, a);
        // elements 2l, 2l+1 sit in word l/8 at bits 4*(l%8) and 4*(l%8)+2
        uint32_t part = (c0 | (c1 << 2)) << (4 * (lane & 7));
        part |= __shfl_xor_sync(0xffffffffu, part, 1);
        part |= __shfl_xor_sync(0xffffffffu, part, 2);
        part |= __shfl_xor_sync(0xffffffffu, part, 4);
        // gather the four words, then lanes 0..17 write the block's 18 bytes
        const uint32_t word0 = __shfl_sync(0xffffffffu, part, 0);
        const uint32_t word1 = __shfl_sync(0xffffffffu, part, 8);
        const uint32_t word2 = __shfl_sync(0xffffffffu, part, 16);
        const uint32_t word3 = __shfl_sync(0xffffffffu, part, 24);
        const uint32_t dbits = __half_as_ushort(__float2half_rn(a));
        if (lane < 18) {
            uint32_t v;
            if (lane < 2) {
                v = dbits >> (8 * lane);
            } else {
                const int j = lane - 2;  // code byte j = byte j%4 of word j/4
                const uint32_t wsel = j < 4 ? word0 : (j < 8 ? word1 : (j < 12 ? word2 : word3));
                v = wsel >> (8 * (j & 3));
            }
            dst[b * 18 + lane] = static_cast<uint8_t>(v & 0xFFu);
        }
    }
}

}  // namespace

cudaError_t launch_quantize(const float *src, uint8_t *dst, int64_t nrows, int64_t K,
                            cudaStream_t s) {
    const int64_t n_blocks = nrows * (K / 64);
    int64_t grid = (n_blocks + 7) / 8;  // 8 warps per CTA
    const int64_t cap = int64_t(sm_count()) * 32;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    quantize_kernel<<<unsigned(grid), 256, 0, s>>>(src, dst, n_blocks);
    return cudaGetLastError();
}

}  // namespace q2
