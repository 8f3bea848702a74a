// Split (structure-of-arrays) layout of a Q2_0 matrix.
//
// Source: "kopitiam_runtime::gpu_offload" (docs.rs), section "Why the weight
// has to stay quantized": a block format's scales are split from its quants
// into separate arrays when the weights are loaded. For an N x K Q2_0 matrix
// with nb = K/64 blocks per row:
//   qs[n][b][16]  the 16 code bytes of block (n, b), row-major;
//   d[n][b]       its fp16 scale, row-major, starting round_up(N*nb*16, 256)
//                 bytes after qs.
// The split is a byte move; the code and scale rules are those of the 18-byte
// block ("WebGPU: add Q2_0 support", format paragraph).
//
// On GB300 the split gives 128-byte code rows per 8 blocks, a width the TMA
// engine can swizzle, so the fp4 mat-vec reads them with
// conflict-free 16-byte shared-memory loads and no byte shuffles
// (mv_t4_kernel<kLaySplit>). This file holds the layout kernels and the CUDA-core
// mat-vec used off that fast path.
#include "q2_0_device.cuh"
#include "q2_0_internal.h"

namespace q2 {
namespace {

// One thread per block: 18 bytes in, 16 + 2 bytes out (or back).
template <bool kToSoa>
__global__ void __launch_bounds__(256) soa_move_kernel(const uint8_t *__restrict__ src,
                                                       uint8_t *__restrict__ dst,
                                                       int64_t n_blocks, int64_t d_offset) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n_blocks;
         i += int64_t(gridDim.x) * blockDim.x) {
        if (kToSoa) {
            const uint8_t *b = src + i * 18;
            uint8_t *qs = dst + i * 16;
            uint8_t *d = dst + d_offset + i * 2;
            d[0] = __ldg(b);
            d[1] = __ldg(b + 1);
#pragma unroll
            for (int j = 0; j < 16; ++j) qs[j] = __ldg(b + 2 + j);
        } else {
            const uint8_t *qs = src + i * 16;
            const uint8_t *d = src + d_offset + i * 2;
            uint8_t *b = dst + i * 18;
            b[0] = __ldg(d);
            b[1] = __ldg(d + 1);
#pragma unroll
            for (int j = 0; j < 16; ++j) b[2 + j] = __ldg(qs + j);
        }
    }
}

// CUDA-core mat-vec over the split layout: one warp per row, block-wise
// s = sum (q - 1) * x over the block, then acc += d * s.
__global__ void __launch_bounds__(256) soa_mv_kernel(const uint8_t *__restrict__ qs,
                                                     const uint8_t *__restrict__ dsc,
                                                     const float *__restrict__ x,
                                                     float *__restrict__ y, int N, int K,
                                                     int ncols) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const int nb = K / 64;
    float acc[8];
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) acc[cc] = 0.0f;
    for (int b = lane; b < nb; b += 32) {
        const size_t i = size_t(row) * nb + b;
        const float d = half_bits_to_float(uint32_t(dsc[2 * i]) | (uint32_t(dsc[2 * i + 1]) << 8));
        float s[8];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) s[cc] = 0.0f;
        for (int wi = 0; wi < 4; ++wi) {
            const uint8_t *pw = qs + 16 * i + 4 * wi;
            const uint32_t word = uint32_t(pw[0]) | (uint32_t(pw[1]) << 8) |
                                  (uint32_t(pw[2]) << 16) | (uint32_t(pw[3]) << 24);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float q1 = float(int((word >> (2 * e)) & 3u) - 1);
                const int k = b * 64 + wi * 16 + e;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                    if (cc < ncols) s[cc] = fmaf(q1, x[size_t(cc) * K + k], s[cc]);
            }
        }
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) acc[cc] = fmaf(d, s[cc], acc[cc]);
    }
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[cc] += __shfl_xor_sync(0xffffffffu, acc[cc], o);
    }
    if (lane == 0)
        for (int cc = 0; cc < ncols; ++cc) y[size_t(cc) * N + row] = acc[cc];
}

unsigned move_grid(int64_t n_blocks) {
    int64_t g = (n_blocks + 255) / 256;
    const int64_t cap = int64_t(sm_count()) * 16;
    if (g > cap) g = cap;
    return unsigned(g < 1 ? 1 : g);
}

}  // namespace

size_t soa_qs_bytes(int64_t N, int64_t K) { return (size_t(N) * (K / 64) * 16 + 255) & ~size_t(255); }

size_t soa_bytes(int64_t N, int64_t K) {
    return soa_qs_bytes(N, K) + ((size_t(N) * (K / 64) * 2 + 255) & ~size_t(255));
}

cudaError_t launch_soa_generic(const uint8_t *soa, const float *x, float *y, int64_t N, int64_t K,
                               int ncols, cudaStream_t s) {
    soa_mv_kernel<<<unsigned((N + 7) / 8), 256, 0, s>>>(soa, soa + soa_qs_bytes(N, K), x, y,
                                                        int(N), int(K), ncols);
    return cudaGetLastError();
}

cudaError_t launch_soa_move(const uint8_t *src, uint8_t *dst, int64_t N, int64_t K, bool to_soa,
                            cudaStream_t s) {
    const int64_t n_blocks = N * (K / 64);
    const int64_t d_off = int64_t(soa_qs_bytes(N, K));
    if (to_soa)
        soa_move_kernel<true><<<move_grid(n_blocks), 256, 0, s>>>(src, dst, n_blocks, d_off);
    else
        soa_move_kernel<false><<<move_grid(n_blocks), 256, 0, s>>>(src, dst, n_blocks, d_off);
    return cudaGetLastError();
}

}  // namespace q2
