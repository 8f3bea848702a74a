/*
 * q2_0.h — C ABI of the GB300 (sm_103a) Q2_0 dequantize-fused matmul library.
 *
 * Q2_0 format. Sources: "WebGPU: add Q2_0 support" (bisque.today write-up of
 * llama.cpp PR 30914), format paragraph; "Llama.cpp umí dvoubitový Q2_0 i na
 * kartách NVIDIA" (aisvetem.cz), section "Osmnáct bajtů na čtyřiašedesát vah".
 *   A block packs 64 weights into 18 bytes: a little-endian IEEE fp16 scale d at
 *   byte 0, then four little-endian u32 words at bytes 2, 6, 10, 14. Element
 *   16*w + i of the block is the code q = (word_w >> 2i) & 3, and decodes to
 *   (q - 1) * d: codes 0/1/2/3 give -d / 0 / +d / +2d (3 is reserved by the
 *   format but decoded by the same rule).
 *   A weight matrix W has N rows of K weights (K a multiple of 64) stored as
 *   N * K/64 consecutive blocks, row-major: block b of row n is at byte offset
 *   (n * K/64 + b) * 18. No alignment is required of W.
 *
 * Activations and outputs follow ggml's mul_mat(src0 = W, src1 = X):
 *   X is F32 [C][K] row-major (C = ncols or M), Y is F32 [C][N] row-major,
 *   Y[c][n] = sum_k W[n][k] * X[c][k].
 *
 * Conventions for every call:
 *   - All pointers are device pointers owned by the caller, unless stated.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are
 *     asynchronous on it; nothing synchronises the host except
 *     q2_0_get_error().
 *   - The calls act on the device current to the calling thread. That device
 *     must be compute capability 10.3 (GB300); otherwise Q2_0_EUNSUPPORTED.
 *   - Argument errors return Q2_0_EINVAL before anything is launched. A failed
 *     launch or runtime call returns Q2_0_ECUDA. No exception crosses the ABI.
 *     There is no CPU fallback: every result is computed by a CUDA kernel.
 *   - Data-dependent errors found by a kernel (an id out of range in get_rows,
 *     a pipeline wait that timed out) are recorded in a per-device error word;
 *     q2_0_get_error() reads and clears it.
 */
#ifndef Q2_0_H
#define Q2_0_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define Q2_0_BLOCK_WEIGHTS 64
#define Q2_0_BLOCK_BYTES 18

typedef enum q2_0_status {
    Q2_0_OK = 0,
    Q2_0_EINVAL = 1,       /* bad argument; nothing was launched */
    Q2_0_ECUDA = 2,        /* a CUDA runtime call or kernel launch failed */
    Q2_0_EUNSUPPORTED = 3, /* the current device is not compute capability 10.3 */
    Q2_0_EDEVICE = 4,      /* a kernel recorded an error: see q2_0_get_error() */
    Q2_0_ENOSPACE = 5      /* q2_0_mul_mat_vec_noalloc: the call needs more scratch than
                              Q2_0_NOALLOC_SCRATCH_BYTES; nothing was launched */
} q2_0_status;

/* Device error codes (first error wins until cleared). */
#define Q2_0_DEVERR_NONE 0
#define Q2_0_DEVERR_BAD_ID 1  /* get_rows / mul_mat_id: ids[info] out of range */
#define Q2_0_DEVERR_TIMEOUT 2 /* a pipeline wait gave up; info = kernel tag */

/* GEMM activation precision. F32 activations are used by the tensor cores as
 * fp16 operands (the weights (q-1)*d are exact in fp16). Each token row is first
 * scaled by an exact power of two that puts its largest |x| in [2^14, 2^15), and
 * the f32 result is scaled back, so any finite x is in range:
 *   Q2_0_PREC_F16_SPLIT: x = hi + lo with hi = fp16(x), lo = fp16(x - hi); two
 *     tensor-core products. Each element x is held to within 2^-22 |x| + 2^-39 M
 *     (M its row's largest |x|): 22 bits of its own value down to 2^-18 M;
 *     tolerance |y - exact| <= 1e-5 * sum|w*x| + 1e-7. The products are exact; the f32 accumulation over K/16 tensor-core
 *     steps adds rounding that is far below that in practice, but whose
 *     worst-case bound grows as (K/16) * 2^-24 * sum|w*x|.
 *   Q2_0_PREC_F16: x rounded once to fp16, within 2^-11 |x| + 2^-39 M.
 *     Tolerance <= 4e-3 * sum|w*x|.
 * Precondition of both: finite x, and |2d| <= 65504 (so that (q-1)*d is finite
 * in fp16). */
typedef enum q2_0_prec { Q2_0_PREC_F16_SPLIT = 0, Q2_0_PREC_F16 = 1 } q2_0_prec;

/* Library version string (static storage). */
const char *q2_0_version(void);

/* Checks that the current device is a compute capability 10.3 GPU.
 * Returns Q2_0_OK, Q2_0_EUNSUPPORTED or Q2_0_ECUDA. */
int q2_0_device_check(void);

/*
 * q2_0_mul_mat_vec — decode mat-vec, Y[c][n] = sum_k W[n][k] X[c][k].
 * Source: the mat-vec kernel of "WebGPU: add Q2_0 support" (each block's codes
 * are multiplied by the activations and the scale d is applied once per block
 * sum).
 *   w      N x K Q2_0 matrix (N*K/64*18 bytes), any alignment.
 *   x      F32 [ncols][K].   y  F32 [ncols][N] (written, not accumulated).
 *   N >= 1, K >= 64 with K % 64 == 0, 1 <= ncols <= 8.
 * Precision (finite x; M_b = the largest |x| of the activation block of 64
 * that holds element k; the tensor-core paths have K % 512 == 0 and w 16-byte
 * aligned, other shapes run f32 on CUDA cores):
 *   ncols 1 and 2, tensor cores (fp4): each element of x is represented to
 *     within 2^-33 M_b; zero weights contribute exactly nothing; the rest is
 *     f32 rounding: |y - exact| <= 2^-33 sum_k |W[n][k]| M_b + 2^-20 sum_k |W X|;
 *   ncols 3..8, tensor cores (e4m3): each element keeps 20 bits of its own value,
 *     with a floor of 2^-33 M_b: |y - exact| <= 2^-33 sum_k |W[n][k]| M_b +
 *     2^-17 sum_k |W X|;
 *   CUDA cores: f32 products and sums, |y - exact| <= 2^-17 sum_k |W X| for
 *     K <= 65536.
 * The tensor-core paths meet the tolerance |y - exact| <= 1e-5 *
 * sum_k |W[n][k] X[c][k]| + 1e-7 unless, weighted by |W|, the activations sit
 * on average more than ~2e4 times below the largest element of their own block
 * of 64.
 * Scratch: the call takes q2_0_mul_mat_vec_workspace_size(K, ncols) bytes of
 * stream-ordered memory from the device's default memory pool
 * (cudaMallocAsync/cudaFreeAsync on `stream`); use q2_0_mul_mat_vec_ws to
 * supply it instead.
 */
int q2_0_mul_mat_vec(const void *w, const float *x, float *y, int64_t N, int64_t K, int ncols,
                     void *stream);

/*
 * q2_0_mul_mat_vec_f16 — q2_0_mul_mat_vec with F16 (IEEE binary16)
 * activations x [ncols][K], any alignment; y F32. The pages' WebGPU port
 * supports F32 activations only and lists F16 ones as missing ("WebGPU: add
 * Q2_0 support", limitations paragraph); this is that variant. Each fp16
 * value is read exactly, so the F32 precision statement applies with x read
 * as the exact fp16 values. Scratch as q2_0_mul_mat_vec (default memory pool).
 */
int q2_0_mul_mat_vec_f16(const void *w, const void *x, float *y, int64_t N, int64_t K, int ncols,
                         void *stream);

/* Scratch bytes q2_0_mul_mat_vec_ws needs for (K, ncols); 0 on bad arguments. */
size_t q2_0_mul_mat_vec_workspace_size(int64_t K, int ncols);

/* As q2_0_mul_mat_vec, with caller-owned scratch `workspace` (device memory,
 * 256-byte aligned, at least workspace_size bytes; contents are overwritten and
 * must not be used by other work in flight). */
int q2_0_mul_mat_vec_ws(const void *w, const float *x, float *y, int64_t N, int64_t K, int ncols,
                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * q2_0_mul_mat_vec_noalloc — q2_0_mul_mat_vec for callers that cannot allocate
 * device memory at call time. (The Q2_0 pages have no counterpart: this is a
 * deployment variant of the decode mat-vec above, with the same arguments and
 * the same result and error bound.)
 *   Who needs it: an inference server or framework that reserves all of HBM
 *   for its own allocator leaves nothing for cudaMalloc or the default memory
 *   pool, and a latency-critical decode loop should not call an allocator at
 *   all. This call allocates nothing: its scratch (the prepared activation
 *   fragments) lives in a static device array of Q2_0_NOALLOC_SCRATCH_BYTES
 *   that every GPU which loads the library holds until the process exits.
 *   Limit: shapes on the tensor-core path (K % 512 == 0 and w 16-byte
 *   aligned) need q2_0_mul_mat_vec_workspace_size(K, ncols) bytes of scratch;
 *   if that exceeds Q2_0_NOALLOC_SCRATCH_BYTES the call returns Q2_0_ENOSPACE
 *   and launches nothing (1 MiB covers K up to 126,976 for ncols = 1, 63,488
 *   for ncols 2..3, 31,744 for ncols 4..6 and 21,504 for ncols 7..8). Other
 *   shapes run the CUDA-core kernel, which needs no scratch, at any K.
 *   Set-up: the first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current and keeps it for the life
 *   of the process; make that first call before any stream capture, and do not
 *   call the entry point again after a cudaDeviceReset of that device (the
 *   kept address belongs to the context the reset destroyed).
 *   Sharing: every call uses the same array and leaves its contents behind.
 *   Each call rewrites all of the scratch it reads, so nothing needs clearing,
 *   but calls whose executions overlap on the GPU (e.g. on two streams) race
 *   on the array: serialise them.
 */
#define Q2_0_NOALLOC_SCRATCH_BYTES ((size_t)1 << 20)
int q2_0_mul_mat_vec_noalloc(const void *w, const float *x, float *y, int64_t N, int64_t K,
                             int ncols, void *stream);

/*
 * Batched decode mat-vec: many independent (W, x, y) products, e.g. all the
 * projections of one decoder step, run by one persistent launch with a static,
 * cost-balanced schedule of row tiles over the GPU's SMs.
 * q2_0_mv_plan_create records the descriptors (the pointers are kept, not the
 * data), encodes per-matrix TMA descriptors, builds the schedule and allocates
 * the plan's device memory and scratch. q2_0_mv_plan_execute launches the work
 * on `stream` (two kernels: activation preparation, then the mat-vecs); it
 * allocates nothing and may be captured in a CUDA graph. Each descriptor
 * obeys q2_0_mul_mat_vec's rules; all share ncols.
 */
typedef struct q2_0_mv_desc {
    const void *w; /* N x K Q2_0 matrix */
    const float *x; /* F32 [ncols][K] */
    float *y;       /* F32 [ncols][N] */
    int64_t N;
    int64_t K;
} q2_0_mv_desc;

typedef struct q2_0_mv_plan q2_0_mv_plan;

int q2_0_mv_plan_create(const q2_0_mv_desc *descs, int n_desc, int ncols, q2_0_mv_plan **plan);
int q2_0_mv_plan_execute(const q2_0_mv_plan *plan, void *stream);
/* Number of kernel launches one execute performs. */
int q2_0_mv_plan_launches(const q2_0_mv_plan *plan);
void q2_0_mv_plan_destroy(q2_0_mv_plan *plan);

/*
 * q2_0_mul_mat — prefill GEMM, Y[m][n] = sum_k W[n][k] X[m][k], M tokens.
 * Source: the tiled matrix multiply of "WebGPU: add Q2_0 support" (codes are
 * unpacked into shared memory as half precision before the product).
 *   w      N x K Q2_0 matrix.  x  F32 [M][K].  y  F32 [M][N] (written).
 *   N, M >= 1, K >= 64 with K % 64 == 0. prec is a q2_0_prec.
 * workspace: device memory of at least q2_0_mul_mat_workspace_size(M, N, K,
 * prec) bytes, 256-byte aligned, or NULL to take it from the device's default
 * memory pool on `stream` (stream-ordered).
 */
size_t q2_0_mul_mat_workspace_size(int64_t M, int64_t N, int64_t K, int prec);
int q2_0_mul_mat(const void *w, const float *x, float *y, int64_t N, int64_t K, int64_t M, int prec,
                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * q2_0_mul_mat_f16 — q2_0_mul_mat with F16 activations x [M][K] (the missing
 * F16 path of the same limitations paragraph). fp16 x is already an exact fp16
 * tensor-core operand, so one product per weight suffices and the bound is
 * |y - exact| <= 1e-5 * sum_k |W[n][k] X[m][k]| + 1e-7 with X the fp16 values.
 * workspace: at least q2_0_mul_mat_workspace_size(M, N, K, Q2_0_PREC_F16)
 * bytes, 256-byte aligned, or NULL for the default memory pool. Fast path:
 * K % 512 == 0, w and x 16-byte aligned; otherwise a CUDA-core kernel.
 */
int q2_0_mul_mat_f16(const void *w, const void *x, float *y, int64_t N, int64_t K, int64_t M,
                     void *workspace, size_t workspace_bytes, void *stream);

/*
 * Grouped prefill GEMM: several independent products Y = W X^T (e.g. the
 * gate and up projections of one layer, which read the same X) run as one
 * launch of the tensor-core kernel over the pooled output tiles, with one
 * activation prepass and one stream-K reduction for all of them.
 * q2_0_mm_plan_create records the descriptors (the pointers are kept, not the
 * data), prepares each distinct activation matrix once (descriptors with the
 * same x, M and K share it), encodes the TMA descriptors and allocates the
 * plan's device memory: per distinct X, the fp16 hi (and lo) copies and the
 * row exponents; the stream-K partial tiles (2 x 128 KB per SM). Each
 * descriptor obeys q2_0_mul_mat's rules and its bound; all share prec. A
 * descriptor outside the fast path (K % 512 != 0, w or x not 16-byte aligned)
 * runs the CUDA-core kernel inside execute. q2_0_mm_plan_execute launches the
 * work on `stream` (the prepass, one launch per 8 distinct X; the tensor-core
 * kernel; the reduction; one launch per CUDA-core descriptor); it allocates
 * nothing and may be captured in a CUDA graph. Each execute reads the
 * current contents of every w and x and writes every y, so the caller may
 * refill x between executes. Products must not write to memory that another
 * product of the same plan reads or writes, and two executes of one plan must
 * not overlap on the GPU (they share the plan's scratch).
 * Ownership: the plan belongs to the device current at creation; execute it
 * on a stream of that device. q2_0_mm_plan_destroy frees its device memory;
 * call it after the last execute has completed.
 * Errors: Q2_0_EINVAL for a null pointer, n_desc < 1, N or M outside
 * [1, 2^31), K not a multiple of 64 in [64, 2^30] or an unknown prec;
 * Q2_0_EUNSUPPORTED for a device that is not compute capability 10.3;
 * Q2_0_ECUDA when an allocation, a copy or a TMA descriptor fails.
 */
typedef struct q2_0_mm_desc {
    const void *w;  /* N x K Q2_0 matrix */
    const float *x; /* F32 [M][K] */
    float *y;       /* F32 [M][N] */
    int64_t N;
    int64_t K;
    int64_t M;
} q2_0_mm_desc;

typedef struct q2_0_mm_plan q2_0_mm_plan;

int q2_0_mm_plan_create(const q2_0_mm_desc *descs, int n_desc, int prec, q2_0_mm_plan **plan);
int q2_0_mm_plan_execute(const q2_0_mm_plan *plan, void *stream);
/* Number of kernel launches one execute performs. */
int q2_0_mm_plan_launches(const q2_0_mm_plan *plan);
void q2_0_mm_plan_destroy(q2_0_mm_plan *plan);

/*
 * Split layout — scales and codes in separate arrays, as the loader in
 * "kopitiam_runtime::gpu_offload" (section "Why the weight has to stay
 * quantized") splits a block format's scales from its quants. For an N x K
 * Q2_0 matrix with nb = K/64 blocks per row, the split buffer holds
 *   qs[n][b][16]  the 16 code bytes of block (n, b), row-major, then, from
 *                 byte round_up(N * nb * 16, 256),
 *   d[n][b]       its fp16 scale (2 bytes, little-endian), row-major;
 * q2_0_split_bytes(N, K) bytes in all. The code and scale rules are the
 * 18-byte block's. The split is a load-time option; q2_0_mul_mat_vec_split
 * computes what q2_0_mul_mat_vec computes on the 18-byte layout.
 *   q2_0_split_layout  18-byte blocks w -> split buffer dst (bit-exact move).
 *   q2_0_join_layout   split buffer src -> 18-byte blocks w (its inverse).
 *   q2_0_mul_mat_vec_split  y = W x with W in the split layout; same bound as
 *       q2_0_mul_mat_vec. Fast path (fp4 tensor cores): ncols 1, K % 512 == 0,
 *       the buffer 16-byte aligned; otherwise a CUDA-core kernel. Scratch is
 *       stream-ordered, from the default memory pool.
 * Returns 0 from q2_0_split_bytes and Q2_0_EINVAL from the others for N < 1,
 * N >= 2^31 or K not a positive multiple of 64. Device pointers, owned by the
 * caller.
 */
size_t q2_0_split_bytes(int64_t N, int64_t K);
int q2_0_split_layout(const void *w, void *dst, int64_t N, int64_t K, void *stream);
int q2_0_join_layout(const void *src, void *w, int64_t N, int64_t K, void *stream);
int q2_0_mul_mat_vec_split(const void *w, const float *x, float *y, int64_t N, int64_t K,
                           int ncols, void *stream);

/*
 * q2_0_mul_mat_id — expert mat-vec of a mixture-of-experts layer (ggml
 * mul_mat_id; the limitations paragraph of "WebGPU: add Q2_0 support" names
 * MUL_MAT_ID as not ported).
 *   w    n_expert Q2_0 matrices of N x K, one after another (expert e starts
 *        at byte e * N * K/64 * 18).
 *   x    F32 [n_tokens][n_x][K]: n_x = 1 (one vector per token, shared by its
 *        experts) or n_x = n_used (one vector per slot).
 *   ids  int32 [n_tokens][n_used], expert of each slot.
 *   y    F32 [n_tokens][n_used][N]:
 *        y[t][i][n] = sum_k W_{ids[t][i]}[n][k] * x[t][n_x == 1 ? 0 : i][k].
 * Bound: |y - exact| <= 1e-5 * sum_k |W x| + 1e-7, as q2_0_mul_mat_vec.
 * workspace: at least q2_0_mul_mat_id_workspace_size(K, n_tokens, n_x) bytes,
 * 256-byte aligned (the size is 0, and NULL allowed, off the fast path).
 * Fast path: K % 512 == 0 and w 16-byte aligned; otherwise a CUDA-core kernel.
 * Limits: n_expert * N < 2^31, n_tokens * n_used and n_tokens * n_x <= 65535.
 * An id outside [0, n_expert) leaves its slot's output unwritten and records
 * Q2_0_DEVERR_BAD_ID with info = the slot index t * n_used + i.
 * n_tokens == 0 is a no-op. All pointers are device memory owned by the caller.
 */
size_t q2_0_mul_mat_id_workspace_size(int64_t K, int64_t n_tokens, int64_t n_x);
int q2_0_mul_mat_id(const void *w, int64_t n_expert, int64_t N, int64_t K, const float *x,
                    int64_t n_x, const int32_t *ids, int64_t n_used, int64_t n_tokens, float *y,
                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * q2_0_get_rows — gather rows of a Q2_0 table into F32, bit-exact.
 * Source: the get-rows shader of "WebGPU: add Q2_0 support" (copies rows of a
 * Q2_0 tensor out, 64 floats per block).
 *   table  n_rows x K Q2_0 matrix.  ids  int32 [n_ids] (repeats allowed).
 *   out    F32 [n_ids][K]: out[r][k] = f32(q - 1) * f32(d), the IEEE product
 *          (signed zeros kept).
 * An id outside [0, n_rows) leaves its output row unwritten and records
 * Q2_0_DEVERR_BAD_ID with info = its position r. n_ids == 0 is a no-op.
 */
int q2_0_get_rows(const void *table, int64_t n_rows, int64_t K, const int32_t *ids, int64_t n_ids,
                  float *out, void *stream);

/*
 * Group-128 Q2_0: 34-byte blocks of 128 weights (fp16 d, then eight
 * little-endian words of sixteen 2-bit codes; element 16w+i in bits 2i..2i+1
 * of word w; code q -> (q - 1) * d). Source: "Llama.cpp umí dvoubitový Q2_0 i
 * na kartách NVIDIA" (aisvetem.cz), "Šest procent, o která se vedl spor" (34
 * bytes per 128 weights) and its closing section (Q2_0.gguf files without the
 * _g64 suffix use this packing). The pages fix only the size; the word layout
 * is the 64-weight block's, extended. K % 128 == 0 for all three calls.
 *
 * q2_0_g128_to_g64 — exact repack: src is an nrows x K group-128 matrix
 * (nrows*K/128*34 bytes), dst (nrows*K/64*18 bytes, written) the same matrix in
 * the 64-weight layout: block i becomes blocks 2i and 2i+1 with i's scale and
 * its code bytes 0..15 and 16..31. Every q2_0_* call then applies to dst.
 */
int q2_0_g128_to_g64(const void *src, void *dst, int64_t nrows, int64_t K, void *stream);

/* q2_0_g128_get_rows — as q2_0_get_rows over a group-128 table, bit-exact. */
int q2_0_g128_get_rows(const void *table, int64_t n_rows, int64_t K, const int32_t *ids,
                      int64_t n_ids, float *out, void *stream);

/* q2_0_g128_mul_mat_vec — as q2_0_mul_mat_vec over a group-128 matrix, for
 * callers that keep the 128-weight packing. ncols = 1 with K % 1024 == 0 and w
 * 16-byte aligned runs the fp4 tensor-core kernel directly on the 34-byte
 * blocks (one 272-byte box per row and 1024 weights; activations scaled per
 * 128 elements), with scratch of 1024 + K/1024 * 8320 bytes (256-aligned) from
 * the device's default memory pool on `stream`; its bound is the ncols = 1 one
 * with M_b the largest |x| of the 128-element block. Other shapes run on CUDA
 * cores (f32, the same error bound as the CUDA-core mat-vec) without scratch. */
int q2_0_g128_mul_mat_vec(const void *w, const float *x, float *y, int64_t N, int64_t K, int ncols,
                         void *stream);

/*
 * q2_0_quantize_ref — the reference quantizer, bit-exact.
 * Source: "Llama.cpp umí dvoubitový Q2_0 i na kartách NVIDIA" (aisvetem.cz),
 * section "Na běžný model to není": the block's largest |w| is the scale and
 * each weight is rounded to the nearest of the four levels.
 *   src  F32 [nrows][K] (finite).  dst  nrows x K Q2_0 matrix (written).
 * Per block: amax = max |w|; d = fp16(amax) rounded to nearest even; code 2 if
 * 2w >= amax, code 0 if 2w <= -amax, else code 1 (ties away from zero; the
 * decisions use the unrounded amax); amax == 0 gives d = 0 and code 1.
 */
int q2_0_quantize_ref(const float *src, void *dst, int64_t nrows, int64_t K, void *stream);

/*
 * q2_0_get_error — synchronises `stream`, then reads and clears the current
 * device's error word. Returns a Q2_0_DEVERR_* code; *info (if not NULL)
 * receives its detail. Returns -1 if the read itself failed.
 */
int q2_0_get_error(void *stream, int64_t *info);

/*
 * q2_0_test_inject_stall — TEST ONLY: exercises the bounded pipeline waits.
 * (No counterpart on the pages: the failure-detection path of this library.)
 * The next fp4 mat-vec launch on the current device (ncols 1 or 2 on the
 * tensor-core path: q2_0_mul_mat_vec, _ws, _noalloc, _f16, a plan; ncols 1:
 * _split or q2_0_mul_mat_id) stops feeding its pipeline before pipeline stage `stage`
 * of each CTA (0 = the first), and every pipeline wait of that launch gives up
 * after wait_limit_ns instead of about one second. The consumers' waits on
 * the missing stage then run out: the kernel records Q2_0_DEVERR_TIMEOUT with
 * info 111 (the wait for a stage's copies), lets the copies it issued land,
 * frees its tensor memory and returns; its outputs are incomplete. Later
 * launches are unaffected. Returns Q2_0_EINVAL for stage < 0 or a limit of 0
 * or above 10 s.
 */
int q2_0_test_inject_stall(int stage, uint64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* Q2_0_H */
