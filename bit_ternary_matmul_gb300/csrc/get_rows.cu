// q2_0_get_rows: gather rows of a Q2_0 table into F32, bit-exact.
//
// Source: "WebGPU: add Q2_0 support" (bisque.today write-up of llama.cpp
// PR 30914), shader paragraph — the get-rows shader copies rows out of a Q2_0
// tensor and writes 64 floats per block; format paragraph — code q decodes to
// (q - 1) * d.
//
// Element e of a block is code byte e/4 (block bytes 2..17), bits 2*(e%4):
// with little-endian words, bits 2i of word w are bits 2*(i%4) of byte
// 2 + 4w + i/4, and 16w + i = 4*(4w + i/4) + i%4.
//
// Layout: one thread per output float4 (4 elements = one code byte), so a warp
// writes 512 contiguous bytes; the kernel is write-bound (4 B written per
// 0.28 B read). Grid-stride over (id, float4) pairs.
#include "q2_0_device.cuh"
#include "q2_0_internal.h"

namespace q2 {

namespace {

// kGroup: weights per block (64: 18-byte blocks; 128: the 34-byte group-128
// packing, whose 32 code bytes follow the same byte rule).
template <bool kVec4, int kGroup>
__global__ void __launch_bounds__(256) get_rows_kernel(const uint8_t *__restrict__ table,
                                                       int64_t n_rows, int64_t K,
                                                       const int32_t *__restrict__ ids,
                                                       int64_t n_ids, float *__restrict__ out,
                                                       unsigned long long *err) {
    constexpr int kCodeBytes = kGroup / 4;
    constexpr int kBlockBytes = 2 + kCodeBytes;
    const int64_t q4_per_row = K / 4;  // float4 per output row
    const int64_t nb = K / kGroup;
    const int64_t total = n_ids * q4_per_row;
    for (int64_t t = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; t < total;
         t += int64_t(gridDim.x) * blockDim.x) {
        const int64_t r = t / q4_per_row;
        const int64_t j = t - r * q4_per_row;  // float4 index within the row
        const int64_t id = ids[r];
        if (id < 0 || id >= n_rows) {
            if (j == 0) record_error(err, Q2_0_DEVERR_BAD_ID, r);
            continue;
        }
        const int64_t b = j / kCodeBytes;                  // block within the row
        const int byte_in_codes = int(j % kCodeBytes);     // elements 4*byte .. +3
        const uint8_t *blk = table + (id * nb + b) * kBlockBytes;
        const uint32_t dbits = uint32_t(__ldg(blk)) | (uint32_t(__ldg(blk + 1)) << 8);
        const uint32_t codes = __ldg(blk + 2 + byte_in_codes);
        const float d = half_bits_to_float(dbits);
        float4 v;
        // IEEE product f32(q - 1) * f32(d): exact, keeps signed zeros.
        v.x = __fmul_rn(float(int(codes & 3u) - 1), d);
        v.y = __fmul_rn(float(int((codes >> 2) & 3u) - 1), d);
        v.z = __fmul_rn(float(int((codes >> 4) & 3u) - 1), d);
        v.w = __fmul_rn(float(int((codes >> 6) & 3u) - 1), d);
        if (kVec4) {
            reinterpret_cast<float4 *>(out + r * K)[j] = v;
        } else {
            float *o = out + r * K + 4 * j;
            o[0] = v.x;
            o[1] = v.y;
            o[2] = v.z;
            o[3] = v.w;
        }
    }
}

}  // namespace

cudaError_t launch_get_rows(const uint8_t *table, int64_t n_rows, int64_t K, const int32_t *ids,
                            int64_t n_ids, float *out, unsigned long long *err, cudaStream_t s,
                            int group) {
    const int64_t total = n_ids * (K / 4);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = int64_t(sm_count()) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    // Rows are K*4 bytes (a multiple of 256), so every row is 16-byte aligned
    // when `out` is; otherwise the same kernel stores scalars.
    const bool vec = (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
    const unsigned g = unsigned(blocks);
    if (group == 128) {
        if (vec)
            get_rows_kernel<true, 128><<<g, 256, 0, s>>>(table, n_rows, K, ids, n_ids, out, err);
        else
            get_rows_kernel<false, 128><<<g, 256, 0, s>>>(table, n_rows, K, ids, n_ids, out, err);
    } else {
        if (vec)
            get_rows_kernel<true, 64><<<g, 256, 0, s>>>(table, n_rows, K, ids, n_ids, out, err);
        else
            get_rows_kernel<false, 64><<<g, 256, 0, s>>>(table, n_rows, K, ids, n_ids, out, err);
    }
    return cudaGetLastError();
}

}  // namespace q2
