// Host-side internals shared by the translation units of libq2_0: launch
// helpers, TMA descriptor encoding and the kernel entry points each .cu file
// exposes to the C-ABI layer (api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/q2_0.h"

namespace q2 {

// Status of the last CUDA call -> q2_0_status.
inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? Q2_0_OK : Q2_0_ECUDA; }

// Checks the current device (cached per device): compute capability 10.3.
int check_device(int *device_out);

// Number of SMs of the current device (cached per device).
int sm_count();

// Device address of the current device's error word (2 x u64), or nullptr.
unsigned long long *error_word_ptr();

// Encodes a 2-D tiled tensor map; returns false on failure.
//   dtype: CU_TENSOR_MAP_DATA_TYPE_*; dims/strides in elements/bytes as the
//   driver API defines them (dim0 innermost; stride1 = bytes between rows).
bool encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t dim0,
                    uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
                    CUtensorMapSwizzle swizzle);

// ---- kernels' host launchers -------------------------------------------------
// group: 64 (18-byte blocks) or 128 (34-byte blocks)
cudaError_t launch_get_rows(const uint8_t *table, int64_t n_rows, int64_t K, const int32_t *ids,
                            int64_t n_ids, float *out, unsigned long long *err, cudaStream_t s,
                            int group = 64);

cudaError_t launch_quantize(const float *src, uint8_t *dst, int64_t nrows, int64_t K,
                            cudaStream_t s);

// activation element types
constexpr int kXF32 = 0;
constexpr int kXF16 = 1;

// mat-vec (x is F32 or F16 by xtype)
size_t matvec_workspace_bytes(int64_t K, int ncols);
bool matvec_fast_path_ok(const void *w, int64_t K);
int matvec_run(const uint8_t *w, const void *x, int xtype, float *y, int64_t N, int64_t K,
               int ncols, void *ws, size_t ws_bytes, cudaStream_t s);

// split layout: codes [N][K/64][16], then (256-byte aligned) fp16 scales [N][K/64]
size_t soa_qs_bytes(int64_t N, int64_t K);
size_t soa_bytes(int64_t N, int64_t K);
cudaError_t launch_soa_move(const uint8_t *src, uint8_t *dst, int64_t N, int64_t K, bool to_soa,
                            cudaStream_t s);
cudaError_t launch_soa_generic(const uint8_t *soa, const float *x, float *y, int64_t N, int64_t K,
                               int ncols, cudaStream_t s);
// mat-vec on the split layout: ncols 1 with K % 512 == 0 on the fp4 kernel
// (scratch: matvec_workspace_bytes(K, 1)); other shapes on CUDA cores
int matvec_split_run(const uint8_t *soa, const float *x, float *y, int64_t N, int64_t K,
                     int ncols, void *ws, size_t ws_bytes, cudaStream_t s);

// group-128 (34-byte blocks) mat-vec: ncols 1 with K % 1024 == 0 and w 16-byte
// aligned on the fp4 kernel (scratch: matvec_g128_workspace_bytes(K, ncols),
// 0 for the other shapes, which run on CUDA cores)
cudaError_t launch_g128_generic(const uint8_t *w, const float *x, float *y, int64_t N, int64_t K,
                                int ncols, cudaStream_t s);
size_t matvec_g128_workspace_bytes(int64_t K, int ncols);
int matvec_g128_run(const uint8_t *w, const float *x, float *y, int64_t N, int64_t K, int ncols,
                    void *ws, size_t ws_bytes, cudaStream_t s);

// expert mat-vec (mul_mat_id), F32 x: one fp4 prep region per activation vector
size_t matvec_moe_workspace_bytes(int64_t K, int64_t n_xvec);
int matvec_moe_run(const uint8_t *w, int64_t n_expert, int64_t N, int64_t K, const float *x,
                   int64_t n_x, const int32_t *ids, int64_t n_used, int64_t n_tokens, float *y,
                   void *ws, size_t ws_bytes, cudaStream_t s);

// batched mat-vec plans (opaque to the C ABI)
int mv_plan_create(const q2_0_mv_desc *descs, int n, int ncols, q2_0_mv_plan **plan);
int mv_plan_execute(const q2_0_mv_plan *plan, cudaStream_t s);
int mv_plan_launches(const q2_0_mv_plan *plan);
void mv_plan_destroy(q2_0_mv_plan *plan);

// GEMM (x is F32 or F16 by xtype; F16 runs the single-operand precision)
size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int prec);
int gemm_run(const uint8_t *w, const void *x, int xtype, float *y, int64_t N, int64_t K,
             int64_t M, int prec, void *ws, size_t ws_bytes, cudaStream_t s);

// grouped GEMM plans (opaque to the C ABI); F32 x
int mm_plan_create(const q2_0_mm_desc *descs, int n, int prec, q2_0_mm_plan **plan);
int mm_plan_execute(const q2_0_mm_plan *plan, cudaStream_t s);
int mm_plan_launches(const q2_0_mm_plan *plan);
void mm_plan_destroy(q2_0_mm_plan *plan);

}  // namespace q2
