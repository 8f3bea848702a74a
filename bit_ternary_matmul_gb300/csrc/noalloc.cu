// q2_0_mul_mat_vec_noalloc: the decode mat-vec with its scratch in a fixed,
// file-scope device array instead of memory obtained at call time.
//
// Some callers cannot allocate device memory when they run the mat-vec: an
// inference server or framework that reserves the whole of HBM for its own
// allocator up front leaves nothing for cudaMalloc or the default memory pool,
// and latency-critical decode loops must not pay for (or be serialised by) an
// allocator call. This entry point gives them the same result as
// q2_0_mul_mat_vec without any allocation: the activation fragments that the
// mat-vec prepares go into g_mv_noalloc_scratch, a static array that every GPU
// loading the library holds until the process exits.
#include <mutex>

#include "q2_0_device.cuh"
#include "q2_0_internal.h"

namespace q2 {
namespace {

// Q2_0_NOALLOC_SCRATCH_BYTES (1 MiB): enough for K up to 126,976 at ncols = 1,
// 63,488 at ncols 2..3, 31,744 at ncols 4..6 and 21,504 at ncols 7..8 (the
// scratch grows with K and ncols).
constexpr size_t kNoAllocScratchBytes = Q2_0_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_mv_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device. Looked up once per
// device, on the first call made with that device current; host code must not
// use the array's name as a device address.
int scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q2_0_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return Q2_0_EUNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_mv_noalloc_scratch) != cudaSuccess || !p)
            return Q2_0_ECUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return Q2_0_OK;
}

}  // namespace
}  // namespace q2

extern "C" int q2_0_mul_mat_vec_noalloc(const void *w, const float *x, float *y, int64_t N,
                                        int64_t K, int ncols, void *stream) {
    if (!w || !x || !y || N < 1 || N > (int64_t(1) << 31) - 1 || K < 64 || K % 64 != 0 ||
        K > (int64_t(1) << 30) || ncols < 1 || ncols > 8)
        return Q2_0_EINVAL;
    // The tensor-core path's scratch must fit the static array; the CUDA-core
    // path (K % 512 != 0 or w not 16-byte aligned) uses none.
    if (q2::matvec_fast_path_ok(w, K) &&
        q2::matvec_workspace_bytes(K, ncols) > q2::kNoAllocScratchBytes)
        return Q2_0_ENOSPACE;
    int st = q2::check_device(nullptr);
    if (st != Q2_0_OK) return st;
    void *scratch = nullptr;
    st = q2::scratch_for_current_device(&scratch);
    if (st != Q2_0_OK) return st;
    return q2::matvec_run(static_cast<const uint8_t *>(w), x, q2::kXF32, y, N, K, ncols, scratch,
                          q2::kNoAllocScratchBytes, reinterpret_cast<cudaStream_t>(stream));
}
