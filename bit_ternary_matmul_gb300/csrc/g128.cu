// Group-128 Q2_0 (34-byte blocks of 128 weights).
//
// Source: "Llama.cpp umí dvoubitový Q2_0 i na kartách NVIDIA" (aisvetem.cz),
// section "Šest procent, o která se vedl spor" — the packing the format's
// authors use for their own models has 128 weights per block, 34 bytes, 2.125
// bits per weight — and its closing section: files named Q2_0.gguf without the
// _g64 suffix are that older packing. The pages give only the size; the layout
// read here is the 64-weight block extended to eight words: fp16 scale d at +0,
// then eight little-endian words, element 16w+i in bits 2i..2i+1 of word w,
// code q -> (q - 1) * d.
//
// The fast kernels read group-128 matrices in two ways: repacked once, exactly,
// into the 64-weight layout (each block becomes two blocks with the same scale,
// 36 bytes instead of 34), after which every fast path applies; or directly,
// for the ncols = 1 mat-vec, by the fp4 tensor-core kernel of matvec.cu with
// 272-byte stage boxes. get_rows reads the 34-byte blocks directly
// (get_rows.cu), and a CUDA-core mat-vec serves the other shapes.
#include "q2_0_device.cuh"
#include "q2_0_internal.h"

namespace q2 {
namespace {

constexpr int kG128Bytes = 34;

// One thread per output byte: output block 2i + h (18 bytes) = scale of block
// i, then its code bytes 16h .. 16h+15.
__global__ void __launch_bounds__(256) g128_to_g64_kernel(const uint8_t *__restrict__ src,
                                                          uint8_t *__restrict__ dst,
                                                          int64_t n_blocks) {
    const int64_t total = n_blocks * 36;
    for (int64_t o = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; o < total;
         o += int64_t(gridDim.x) * blockDim.x) {
        const int64_t i = o / 36;
        const int r = int(o - i * 36);
        const int h = r >= 18 ? 1 : 0;
        const int ob = r - 18 * h;  // byte within the 18-byte output block
        const uint8_t *b = src + i * kG128Bytes;
        dst[o] = ob < 2 ? __ldg(b + ob) : __ldg(b + 2 + 16 * h + (ob - 2));
    }
}

// CUDA-core mat-vec over 34-byte blocks: one warp per row, block-wise
// s = sum (q - 1) * x over the block, then acc += d * s.
__global__ void __launch_bounds__(256) g128_mv_kernel(const uint8_t *__restrict__ w,
                                                      const float *__restrict__ x,
                                                      float *__restrict__ y, int N, int K,
                                                      int ncols) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const int nb = K / 128;
    float acc[8];
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) acc[cc] = 0.0f;
    for (int b = lane; b < nb; b += 32) {
        const uint8_t *blk = w + (size_t(row) * nb + b) * kG128Bytes;
        const float d = half_bits_to_float(uint32_t(blk[0]) | (uint32_t(blk[1]) << 8));
        float s[8];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) s[cc] = 0.0f;
        for (int wi = 0; wi < 8; ++wi) {
            const uint8_t *pw = blk + 2 + 4 * wi;
            const uint32_t word = uint32_t(pw[0]) | (uint32_t(pw[1]) << 8) |
                                  (uint32_t(pw[2]) << 16) | (uint32_t(pw[3]) << 24);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float q1 = float(int((word >> (2 * i)) & 3u) - 1);
                const int k = b * 128 + wi * 16 + i;
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

inline bool valid_k128(int64_t K) { return K >= 128 && K % 128 == 0 && K <= (int64_t(1) << 30); }

}  // namespace

cudaError_t launch_g128_generic(const uint8_t *w, const float *x, float *y, int64_t N, int64_t K,
                                int ncols, cudaStream_t s) {
    g128_mv_kernel<<<unsigned((N + 7) / 8), 256, 0, s>>>(w, x, y, int(N), int(K), ncols);
    return cudaGetLastError();
}

}  // namespace q2

using namespace q2;

extern "C" {

int q2_0_g128_to_g64(const void *src, void *dst, int64_t nrows, int64_t K, void *stream) {
    if (!src || !dst || nrows < 1 || nrows > (int64_t(1) << 31) - 1 || !valid_k128(K))
        return Q2_0_EINVAL;
    int st = check_device(nullptr);
    if (st != Q2_0_OK) return st;
    const int64_t n_blocks = nrows * (K / 128);
    int64_t grid = (n_blocks * 36 + 255) / 256;
    const int64_t cap = int64_t(sm_count()) * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    g128_to_g64_kernel<<<unsigned(grid), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(src), static_cast<uint8_t *>(dst), n_blocks);
    return cuda_status(cudaGetLastError());
}

int q2_0_g128_get_rows(const void *table, int64_t n_rows, int64_t K, const int32_t *ids,
                      int64_t n_ids, float *out, void *stream) {
    if (n_ids < 0 || n_rows < 1 || !valid_k128(K)) return Q2_0_EINVAL;
    if (n_ids == 0) return Q2_0_OK;
    if (!table || !ids || !out || n_ids > (int64_t(1) << 31) - 1) return Q2_0_EINVAL;
    int st = check_device(nullptr);
    if (st != Q2_0_OK) return st;
    unsigned long long *err = error_word_ptr();
    if (!err) return Q2_0_ECUDA;
    return cuda_status(launch_get_rows(static_cast<const uint8_t *>(table), n_rows, K, ids, n_ids,
                                       out, err, reinterpret_cast<cudaStream_t>(stream), 128));
}

}  // extern "C"
