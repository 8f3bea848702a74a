// C-ABI entry points of libq2_0: argument validation, device checks, scratch
// handling and the device error word. Kernels live in the other .cu files.
#include <mutex>

#include "q2_0_device.cuh"
#include "q2_0_internal.h"

namespace q2 {

// Per-device error word (first error wins until q2_0_get_error clears it).
__device__ unsigned long long g_error_word[2];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_dev_state[kMaxDevices];  // 0 unknown, 1 ok, 2 unsupported
int g_sm_count[kMaxDevices];
unsigned long long *g_err_ptr[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn get_encode() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return g_encode;
}

}  // namespace

int check_device(int *device_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q2_0_ECUDA;
    if (device_out) *device_out = dev;
    if (dev < 0 || dev >= kMaxDevices) return Q2_0_EUNSUPPORTED;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_dev_state[dev] == 1) return Q2_0_OK;
        if (g_dev_state[dev] == 2) return Q2_0_EUNSUPPORTED;
    }
    cudaDeviceProp p;
    if (cudaGetDeviceProperties(&p, dev) != cudaSuccess) return Q2_0_ECUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    g_dev_state[dev] = (p.major == 10 && p.minor == 3) ? 1 : 2;
    g_sm_count[dev] = p.multiProcessorCount;
    return g_dev_state[dev] == 1 ? Q2_0_OK : Q2_0_EUNSUPPORTED;
}

int sm_count() {
    int dev = 0;
    if (check_device(&dev) != Q2_0_OK) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    return g_sm_count[dev];
}

unsigned long long *error_word_ptr() {
    int dev = 0;
    if (check_device(&dev) != Q2_0_OK) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<unsigned long long *>(p);
    }
    return g_err_ptr[dev];
}

bool encode_tmap_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t dim0,
                    uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
                    CUtensorMapSwizzle swizzle) {
    EncodeTiledFn f = get_encode();
    if (!f) return false;
    cuuint64_t dims[2] = {dim0, dim1};
    cuuint64_t strides[1] = {stride1_bytes};
    cuuint32_t box[2] = {box0, box1};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = f(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace q2

using namespace q2;

namespace {

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool valid_k(int64_t K) { return K >= 64 && K % 64 == 0 && K <= (int64_t(1) << 30); }

// Stream-ordered scratch from the device's default memory pool.
struct PoolScratch {
    void *ptr = nullptr;
    cudaStream_t s = nullptr;
    int alloc(size_t bytes, cudaStream_t st) {
        s = st;
        if (bytes == 0) return Q2_0_OK;
        return cuda_status(cudaMallocAsync(&ptr, bytes, st));
    }
    int release() {
        if (!ptr) return Q2_0_OK;
        cudaError_t e = cudaFreeAsync(ptr, s);
        ptr = nullptr;
        return cuda_status(e);
    }
};

}  // namespace

extern "C" {

const char *q2_0_version(void) { return "q2_0-gb300 0.1.0 (sm_103a)"; }

int q2_0_device_check(void) { return check_device(nullptr); }

size_t q2_0_mul_mat_vec_workspace_size(int64_t K, int ncols) {
    if (!valid_k(K) || ncols < 1 || ncols > 8) return 0;
    return matvec_workspace_bytes(K, ncols);
}

int q2_0_mul_mat_vec_ws(const void *w, const float *x, float *y, int64_t N, int64_t K, int ncols,
                        void *workspace, size_t workspace_bytes, void *stream) {
    if (!w || !x || !y || N < 1 || N > (int64_t(1) << 31) - 1 || !valid_k(K) || ncols < 1 ||
        ncols > 8)
        return Q2_0_EINVAL;
    size_t need = matvec_workspace_bytes(K, ncols);
    if (workspace_bytes < need || (need && !workspace) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return Q2_0_EINVAL;
    int st = check_device(nullptr);
    if (st != Q2_0_OK) return st;
    return matvec_run(static_cast<const uint8_t *>(w), x, kXF32, y, N, K, ncols, workspace,
                      workspace_bytes, as_stream(stream));
}

}  // extern "C"

namespace {

int mul_mat_vec_pool(const void *w, const void *x, int xtype, float *y, int64_t N, int64_t K,
                     int ncols, void *stream) {
    if (!w || !x || !y || N < 1 || N > (int64_t(1) << 31) - 1 || !valid_k(K) || ncols < 1 ||
        ncols > 8)
        return Q2_0_EINVAL;
    int st = check_device(nullptr);
    if (st != Q2_0_OK) return st;
    size_t need = matvec_workspace_bytes(K, ncols);
    PoolScratch ws;
    st = ws.alloc(need, as_stream(stream));
    if (st != Q2_0_OK) return st;
    st = matvec_run(static_cast<const uint8_t *>(w), x, xtype, y, N, K, ncols, ws.ptr, need,
                    as_stream(stream));
    int st2 = ws.release();
    return st != Q2_0_OK ? st : st2;
}

int mul_mat_impl(const void *w, const void *x, int xtype, float *y, int64_t N, int64_t K,
                 int64_t M, int prec, void *workspace, size_t workspace_bytes, void *stream) {
    if (!w || !x || !y || N < 1 || M < 1 || N > (int64_t(1) << 31) - 1 ||
        M > (int64_t(1) << 31) - 1 || !valid_k(K) ||
        (prec != Q2_0_PREC_F16_SPLIT && prec != Q2_0_PREC_F16))
        return Q2_0_EINVAL;
    size_t need = gemm_workspace_bytes(M, N, K, prec);
    if (workspace && (workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return Q2_0_EINVAL;
    int st = check_device(nullptr);
    if (st != Q2_0_OK) return st;
    if (workspace || need == 0)
        return gemm_run(static_cast<const uint8_t *>(w), x, xtype, y, N, K, M, prec, workspace,
                        workspace_bytes, as_stream(stream));
    PoolScratch ws;
    st = ws.alloc(need, as_stream(stream));
    if (st != Q2_0_OK) return st;
    st = gemm_run(static_cast<const uint8_t *>(w), x, xtype, y, N, K, M, prec, ws.ptr, need,
                  as_stream(stream));
    int st2 = ws.release();
    return st != Q2_0_OK ? st : st2;
}

}  // namespace

extern "C" {

int q2_0_mul_mat_vec(const void *w, const float *x, float *y, int64_t N, int64_t K, int ncols,
                     void *stream) {
    return mul_mat_vec_pool(w, x, kXF32, y, N, K, ncols, stream);
}

int q2_0_mul_mat_vec_f16(const void *w, const void *x, float *y, int64_t N, int64_t K, int ncols,
                         void *stream) {
    return mul_mat_vec_pool(w, x, kXF16, y, N, K, ncols, stream);
}

int q2_0_mv_plan_create(const q2_0_mv_desc *descs, int n_desc, int ncols, q2_0_mv_plan **plan) {
    if (!plan) return Q2_0_EINVAL;
    *plan = nullptr;
    if (!descs || n_desc < 1 || ncols < 1 || ncols > 8) return Q2_0_EINVAL;
    for (int i = 0; i < n_desc; ++i) {
        const q2_0_mv_desc &d = descs[i];
        if (!d.w || !d.x || !d.y || d.N < 1 || d.N > (int64_t(1) << 31) - 1 || !valid_k(d.K))
            return Q2_0_EINVAL;
    }
    int st = check_device(nullptr);
    if (st != Q2_0_OK) return st;
    return mv_plan_create(descs, n_desc, ncols, plan);
}

int q2_0_mv_plan_execute(const q2_0_mv_plan *plan, void *stream) {
    if (!plan) return Q2_0_EINVAL;
    return mv_plan_execute(plan, as_stream(stream));
}

int q2_0_mv_plan_launches(const q2_0_mv_plan *plan) { return plan ? mv_plan_launches(plan) : 0; }

void q2_0_mv_plan_destroy(q2_0_mv_plan *plan) {
    if (plan) mv_plan_destroy(plan);
}

size_t q2_0_mul_mat_workspace_size(int64_t M, int64_t N, int64_t K, int prec) {
    if (M < 1 || N < 1 || !valid_k(K) || (prec != Q2_0_PREC_F16_SPLIT && prec != Q2_0_PREC_F16))
        return 0;
    return gemm_workspace_bytes(M, N, K, prec);
}

int q2_0_mul_mat(const void *w, const float *x, float *y, int64_t N, int64_t K, int64_t M, int prec,
                 void *workspace, size_t workspace_bytes, void *stream) {
    return mul_mat_impl(w, x, kXF32, y, N, K, M, prec, workspace, workspace_bytes, stream);
}

int q2_0_mul_mat_f16(const void *w, const void *x, float *y, int64_t N, int64_t K, int64_t M,
                     void *workspace, size_t workspace_bytes, void *stream) {
    return mul_mat_impl(w, x, kXF16, y, N, K, M, Q2_0_PREC_F16, workspace, workspace_bytes, stream);
}

int q2_0_mm_plan_create(const q2_0_mm_desc *descs, int n_desc, int prec, q2_0_mm_plan **plan) {
    if (!plan) return Q2_0_EINVAL;
    *plan = nullptr;
    if (!descs || n_desc < 1 || (prec != Q2_0_PREC_F16_SPLIT && prec != Q2_0_PREC_F16))
        return Q2_0_EINVAL;
    for (int i = 0; i < n_desc; ++i) {
        const q2_0_mm_desc &d = descs[i];
        if (!d.w || !d.x || !d.y || d.N < 1 || d.M < 1 || d.N > (int64_t(1) << 31) - 1 ||
            d.M > (int64_t(1) << 31) - 1 || !valid_k(d.K))
            return Q2_0_EINVAL;
    }
    int st = check_device(nullptr);
    if (st != Q2_0_OK) return st;
    return mm_plan_create(descs, n_desc, prec, plan);
}

int q2_0_mm_plan_execute(const q2_0_mm_plan *plan, void *stream) {
    if (!plan) return Q2_0_EINVAL;
    return mm_plan_execute(plan, as_stream(stream));
}

int q2_0_mm_plan_launches(const q2_0_mm_plan *plan) { return plan ? mm_plan_launches(plan) : 0; }

void q2_0_mm_plan_destroy(q2_0_mm_plan *plan) {
    if (plan) mm_plan_destroy(plan);
}

size_t q2_0_split_bytes(int64_t N, int64_t K) {
    if (N < 1 || N > (int64_t(1) << 31) - 1 || !valid_k(K)) return 0;
    return soa_bytes(N, K);
}

int q2_0_split_layout(const void *w, void *dst, int64_t N, int64_t K, void *stream) {
    if (!w || !dst || N < 1 || N > (int64_t(1) << 31) - 1 || !valid_k(K)) return Q2_0_EINVAL;
    int st = check_device(nullptr);
    if (st != Q2_0_OK) return st;
    return cuda_status(launch_soa_move(static_cast<const uint8_t *>(w), static_cast<uint8_t *>(dst),
                                       N, K, true, as_stream(stream)));
}

int q2_0_join_layout(const void *src, void *w, int64_t N, int64_t K, void *stream) {
    if (!src || !w || N < 1 || N > (int64_t(1) << 31) - 1 || !valid_k(K)) return Q2_0_EINVAL;
    int st = check_device(nullptr);
    if (st != Q2_0_OK) return st;
    return cuda_status(launch_soa_move(static_cast<const uint8_t *>(src), static_cast<uint8_t *>(w),
                                       N, K, false, as_stream(stream)));
}

int q2_0_mul_mat_vec_split(const void *w, const float *x, float *y, int64_t N, int64_t K,
                           int ncols, void *stream) {
    if (!w || !x || !y || N < 1 || N > (int64_t(1) << 31) - 1 || !valid_k(K) || ncols < 1 ||
        ncols > 8)
        return Q2_0_EINVAL;
    int st = check_device(nullptr);
    if (st != Q2_0_OK) return st;
    const size_t need = ncols == 1 ? matvec_workspace_bytes(K, 1) : 0;
    PoolScratch ws;
    st = ws.alloc(need, as_stream(stream));
    if (st != Q2_0_OK) return st;
    st = matvec_split_run(static_cast<const uint8_t *>(w), x, y, N, K, ncols, ws.ptr, need,
                          as_stream(stream));
    int st2 = ws.release();
    return st != Q2_0_OK ? st : st2;
}

int q2_0_g128_mul_mat_vec(const void *w, const float *x, float *y, int64_t N, int64_t K, int ncols,
                         void *stream) {
    if (!w || !x || !y || N < 1 || N > (int64_t(1) << 31) - 1 || K < 128 || K % 128 != 0 ||
        K > (int64_t(1) << 30) || ncols < 1 || ncols > 8)
        return Q2_0_EINVAL;
    int st = check_device(nullptr);
    if (st != Q2_0_OK) return st;
    const size_t need = matvec_g128_workspace_bytes(K, ncols);
    PoolScratch ws;
    st = ws.alloc(need, as_stream(stream));
    if (st != Q2_0_OK) return st;
    st = matvec_g128_run(static_cast<const uint8_t *>(w), x, y, N, K, ncols, ws.ptr, need,
                         as_stream(stream));
    int st2 = ws.release();
    return st != Q2_0_OK ? st : st2;
}

// Expert mat-vec shapes: n_expert * N rows must fit a tensor-map coordinate,
// and the activation vectors a grid dimension.
static bool valid_moe(int64_t n_expert, int64_t N, int64_t K, int64_t n_x, int64_t n_used,
                      int64_t n_tokens) {
    return n_expert >= 1 && N >= 1 && valid_k(K) && n_used >= 1 && n_tokens >= 0 &&
           (n_x == 1 || n_x == n_used) && n_expert * N <= (int64_t(1) << 31) - 1 &&
           n_tokens * n_x <= 65535 && n_tokens * n_used <= 65535;
}

size_t q2_0_mul_mat_id_workspace_size(int64_t K, int64_t n_tokens, int64_t n_x) {
    if (!valid_k(K) || n_tokens < 0 || n_x < 1) return 0;
    return matvec_moe_workspace_bytes(K, n_tokens * n_x);
}

int q2_0_mul_mat_id(const void *w, int64_t n_expert, int64_t N, int64_t K, const float *x,
                    int64_t n_x, const int32_t *ids, int64_t n_used, int64_t n_tokens, float *y,
                    void *workspace, size_t workspace_bytes, void *stream) {
    if (!valid_moe(n_expert, N, K, n_x, n_used, n_tokens)) return Q2_0_EINVAL;
    if (n_tokens == 0) return Q2_0_OK;
    if (!w || !x || !ids || !y) return Q2_0_EINVAL;
    const size_t need = matvec_moe_workspace_bytes(K, n_tokens * n_x);
    if (matvec_fast_path_ok(w, K) &&
        (workspace_bytes < need || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return Q2_0_EINVAL;
    int st = check_device(nullptr);
    if (st != Q2_0_OK) return st;
    return matvec_moe_run(static_cast<const uint8_t *>(w), n_expert, N, K, x, n_x, ids, n_used,
                          n_tokens, y, workspace, workspace_bytes, as_stream(stream));
}

int q2_0_get_rows(const void *table, int64_t n_rows, int64_t K, const int32_t *ids, int64_t n_ids,
                  float *out, void *stream) {
    if (n_ids < 0 || n_rows < 1 || !valid_k(K)) return Q2_0_EINVAL;
    if (n_ids == 0) return Q2_0_OK;
    if (!table || !ids || !out || n_ids > (int64_t(1) << 31) - 1) return Q2_0_EINVAL;
    int st = check_device(nullptr);
    if (st != Q2_0_OK) return st;
    unsigned long long *err = error_word_ptr();
    if (!err) return Q2_0_ECUDA;
    return cuda_status(launch_get_rows(static_cast<const uint8_t *>(table), n_rows, K, ids, n_ids,
                                       out, err, as_stream(stream)));
}

int q2_0_quantize_ref(const float *src, void *dst, int64_t nrows, int64_t K, void *stream) {
    if (!src || !dst || nrows < 1 || !valid_k(K) || nrows > (int64_t(1) << 31) - 1)
        return Q2_0_EINVAL;
    int st = check_device(nullptr);
    if (st != Q2_0_OK) return st;
    return cuda_status(launch_quantize(src, static_cast<uint8_t *>(dst), nrows, K,
                                       as_stream(stream)));
}

int q2_0_get_error(void *stream, int64_t *info) {
    if (check_device(nullptr) != Q2_0_OK) return -1;
    cudaStream_t s = as_stream(stream);
    unsigned long long host[2] = {0, 0};
    const unsigned long long zero[2] = {0, 0};
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbolAsync(host, g_error_word, sizeof(host), 0, cudaMemcpyDeviceToHost, s) !=
        cudaSuccess)
        return -1;
    if (cudaMemcpyToSymbolAsync(g_error_word, zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
        return -1;
    if (cudaStreamSynchronize(s) != cudaSuccess) return -1;
    if (info) *info = static_cast<int64_t>(host[1]);
    return static_cast<int>(host[0]);
}

}  // extern "C"
