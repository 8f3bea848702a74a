// Q2_0 decode mat-vec: Y[c][n] = sum_k W[n][k] X[c][k] for ncols = 1..8.
//
// Source: "WebGPU: add Q2_0 support" (bisque.today write-up of llama.cpp
// PR 30914), mat-vec kernel excerpt: four threads share a 64-weight block, each
// owning one 32-bit word of 16 codes; codes are shifted out of the word two
// bits at a time, (q - 1) multiplies the activation, and the scale d is applied
// once per block sum. This file keeps that structure — a thread owns word c of
// a block, d is applied once per block — but does the multiply-accumulate on
// the tensor cores (mma.sync m16n8k16, fp16 in, fp32 accumulate):
//
// Decode without shifts. For field m (0..3) the mask 0x00030003 << 2m picks,
// from one word, the codes of elements i = m and i = 8 + m into the two fp16
// halves of a register; read as fp16 these are the subnormals q * 4^m * 2^-24,
// exact. (word >> 8) with the same masks picks elements 4 + m and 12 + m. So a
// word becomes 8 A-operand registers with one logic op each (+1 shift). The
// per-field factor 4^m is removed by scaling the activations of field m by
// 4^-m, and the "- 1" of (q - 1) by starting each block's accumulation at
// -sum(activation * 4^m * 2^-24) of that block (the value all-ones codes give).
//
// Activations (F32) enter as fp16 hi + lo pairs: per column j, u = x * 2^s_j
// with 2^s_j chosen so max|u| lies in [2^14, 2^15); for element e of a block,
// v = u * 2^-2(e%4), hi = fp16(v), lo = fp16(v - hi). MMA n-tile t carries
// activation columns 4t..4t+3: its B column 2i is the hi part of column 4t+i
// and B column 2i+1 the lo part, so the lanes that carry data are consecutive
// (lanes 0..7 for one column) and a thread's two accumulator registers of a row
// hold hi and lo of the same column. A small kernel (mv_prep) writes these
// fragments once per call, in register order; the mat-vec kernel only loads them.
//
// Streaming. Each CTA (16 consumer warps of 16 rows + 1 producer warp) owns row
// tiles of 256 rows. A pipeline stage is one 2-D TMA box of 256 rows x 144 bytes
// (8 blocks = 512 weights per row) plus the 8 blocks' fragment records (1-D
// bulk copy); as many stages as fit in shared memory. 144-byte rows make the
// shared-memory words of the 8 rows of an MMA group fall in distinct banks.
// Block pairs (36 bytes) start 4-byte aligned: the odd block's words are
// aligned, the even block's words straddle two aligned words and are rebuilt
// with one byte-permute. The consumer loop is limited by shared-memory
// wavefronts, so the record layout is chosen for dense 16-byte fragment loads.
//
// Requirements of the TMA path: K % 512 == 0 (row stride a multiple of 16 B)
// and W 16-byte aligned. Other shapes run mv_generic_kernel (CUDA cores, f32).
// Activations are F32 or F16 (the prep kernels and the generic kernel read
// either; F16 values are converted exactly).
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <queue>
#include <vector>

#include "q2_0_device.cuh"
#include "q2_0_internal.h"
#include "q2_0_tcgen05.cuh"

namespace q2 {

namespace {

constexpr int kTileRows = 256;
constexpr int kChunkBlocks = 8;
constexpr int kChunkBytes = kChunkBlocks * 18;  // 144
constexpr int kWStageBytes = kTileRows * kChunkBytes;  // 36864
constexpr int kPrepHeader = 64;  // float out_scale[8] (+ pad)
constexpr int kMaxStages = 12;
constexpr int kPrepThreads = 512;
// Dynamic shared memory the ring may use: the opt-in maximum less the static
// part and the barriers.
constexpr int kSmemBudget = 232448 - 1024 - 2 * kMaxStages * 8;

// Timeout tags (info of Q2_0_DEVERR_TIMEOUT).
constexpr int kTagMvFull = 101;
constexpr int kTagMvEmpty = 102;

struct MvPrepJob {
    const void *x;   // [ncols][K], F32 or F16 (the prep kernel's template argument)
    uint8_t *prep;   // prepared fragments
    int K;
    // fp4 prep only, launched without a job list: grid row j prepares the vector
    // at x + j * x_stride into prep + j * prep_stride (bytes)
    long long x_stride;
    long long prep_stride;
};

struct MvJob {  // 64-byte aligned through its CUtensorMap member
    CUtensorMap tmap;  // W as uint8 [N][K/64*18], box {144, 256}
    const uint8_t *prep;
    float *y;
    int N;
    int nb;        // K / 64
    int n_chunks;  // K / 512
    int n_tiles;   // ceil(N / 256)
    CUtensorMap tmap_d;  // split layout only: fp16 scales [N][K/64], box {16, 128}
};

struct MvItem {
    int job;
    int tile;
};

// Expert mat-vec (mul_mat_id) on the fp4 kernel: the single job's tensor map
// spans all experts' rows; output vector v = t * n_used + i takes expert
// ids[v]. ids == nullptr for every other launch.
struct MvMoe {
    const int32_t *ids;     // [n_vec]
    int n_vec;              // n_tokens * n_used
    int n_used;
    int n_x;                // activation vectors per token: 1 (shared) or n_used
    int n_expert;
    long long prep_stride;  // bytes between consecutive activation vectors' prep
};

struct MvParams {
    const MvJob *jobs;        // nullptr: the single job passed by value
    const MvItem *items;      // per-CTA work lists (schedule), when jobs != nullptr
    const int *cta_begin;     // [gridDim.x + 1]
    const int *cta_stages;    // [gridDim.x] stages (512-column chunks) per CTA, plan only
    int ncols;
    int n_stages;             // pipeline depth (n_stages_for(ncols))
    unsigned long long *err;
    MvMoe moe;
    int split;                // fp4 kernel only: 1 = the split layout (codes and scales apart)
};

// Record per block per n-tile, for S = lane slots carrying data (8 per column of
// the tile; the tiles of ncols 5..8 both use 32): B-fragment registers 0..3 of
// lanes 0..S-1 (16 B each), registers 4..7 of those lanes, then for each lane
// group c the accumulator starts (hi, lo) of column 4t + c (8 B each).
__host__ __device__ constexpr int n_tiles_for(int ncols) { return ncols <= 4 ? 1 : 2; }
__host__ __device__ constexpr int used_slots(int ncols) { return ncols <= 4 ? 8 * ncols : 32; }
__host__ __device__ constexpr int rec_bytes(int ncols) { return 32 * used_slots(ncols) + 32; }
__host__ __device__ constexpr int rstage_bytes(int ncols) {
    return kChunkBlocks * n_tiles_for(ncols) * rec_bytes(ncols);
}
constexpr int n_stages_for(int ncols) {
    return kSmemBudget / (kWStageBytes + rstage_bytes(ncols)) < kMaxStages
               ? kSmemBudget / (kWStageBytes + rstage_bytes(ncols))
               : kMaxStages;
}
constexpr int smem_bytes_for(int ncols) {
    return n_stages_for(ncols) * (kWStageBytes + rstage_bytes(ncols)) + 2 * kMaxStages * 8;
}

size_t prep_bytes_for(int64_t K, int ncols) {
    size_t b = kPrepHeader + size_t(K / 64) * n_tiles_for(ncols) * rec_bytes(ncols);
    return (b + 255) & ~size_t(255);
}


// v * 2^e for |e| <= 252 with two exact power-of-two factors (each a normal f32).
__device__ __forceinline__ float mul_pow2(float v, int e) {
    const int e1 = e / 2, e2 = e - e1;
    return v * __int_as_float((127 + e1) << 23) * __int_as_float((127 + e2) << 23);
}

// Activation element load: F32 as is, F16 (IEEE binary16) converted exactly.
__device__ __forceinline__ float ld_x(const float *p) { return *p; }
__device__ __forceinline__ float ld_x(const __half *p) { return __half2float(*p); }

// ---------------------------------------------------------------------------
// Activation preparation: grid (ncols, n_jobs), kPrepThreads threads.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
    return uint32_t(__half_as_ushort(lo)) | (uint32_t(__half_as_ushort(hi)) << 16);
}

template <int NT, typename XT>
__global__ void __launch_bounds__(kPrepThreads) mv_prep_kernel(
    const __grid_constant__ MvPrepJob single, const MvPrepJob *__restrict__ jobs, int ncols) {
    // The mat-vec kernel that follows may start its prologue (barrier set-up,
    // weight loads) now; it waits for this grid before reading the fragments.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Launched as a programmatic dependent of the kernel before it on the stream
    // (a mat-vec that may still read this buffer, or the producer of x): wait
    // for that grid before reading x or writing the prep buffer.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const MvPrepJob &J = jobs ? jobs[blockIdx.y] : single;
    const int K = J.K;
    const int j = blockIdx.x;  // activation column
    const XT *xj = static_cast<const XT *>(J.x) + size_t(j) * K;
    const int tid = threadIdx.x;
    const int nb = K / 64;

    // 1) column scale 2^s with max|x * 2^s| in [2^14, 2^15). The thread's first
    //    16-element group stays in registers for step 2.
    float first[16];
    float m = 0.0f;
    if (tid < nb * 4) {
        if (sizeof(XT) == 4 && (reinterpret_cast<uintptr_t>(xj) & 15u) == 0) {
            const float4 *src = reinterpret_cast<const float4 *>(xj + tid * 16);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const float4 f = src[q4];
                first[4 * q4] = f.x;
                first[4 * q4 + 1] = f.y;
                first[4 * q4 + 2] = f.z;
                first[4 * q4 + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) first[i] = ld_x(xj + tid * 16 + i);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(first[i]));
    }
    for (int k = (kPrepThreads + tid) * 16; k < K; k += kPrepThreads * 16)
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(ld_x(xj + k + i)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float red[kPrepThreads / 32];
    if ((tid & 31) == 0) red[tid >> 5] = m;
    __syncthreads();
    float amax = red[0];
#pragma unroll
    for (int w = 1; w < kPrepThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    int s = 0;
    if (amax > 0.0f && amax <= 3.4e38f) {
        int e;
        frexpf(amax, &e);  // amax = f * 2^e, f in [0.5, 1)
        s = min(max(15 - e, -100), 126);
    }
    float *out_scale = reinterpret_cast<float *>(J.prep);
    if (tid == 0) out_scale[j] = ldexpf(1.0f, 24 - s);
    if (j == 0 && tid < 8 && tid >= ncols) out_scale[tid] = 0.0f;

    // 2) fragments. Thread handles (block b, word c): the 16 elements 16c..16c+15.
    const float fscale[4] = {ldexpf(1.0f, s), ldexpf(1.0f, s - 2), ldexpf(1.0f, s - 4),
                             ldexpf(1.0f, s - 6)};
    const int lane = tid & 31;
    const int su = used_slots(ncols), rb = rec_bytes(ncols);
    const int t = j >> 2, jc = j & 3;  // n-tile and column within it
    for (int idx = tid; idx < nb * 4; idx += kPrepThreads) {
        const int b = idx >> 2, c = idx & 3;
        const XT *xe = xj + b * 64 + c * 16;
        __half hi[16], lo[16];
        float base_hi = 0.0f, base_lo = 0.0f;  // sum over the block of part * 4^m * 2^-24
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float xv = idx == tid ? first[i] : ld_x(xe + i);
            const float v = xv * fscale[i & 3];
            hi[i] = __float2half_rn(v);
            lo[i] = __float2half_rn(v - __half2float(hi[i]));
            const float wgt = ldexpf(1.0f, 2 * (i & 3) - 24);
            base_hi += __half2float(hi[i]) * wgt;
            base_lo += __half2float(lo[i]) * wgt;
        }
        uint32_t rh[8], rl[8];
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
            rh[2 * mm] = pack_half2(hi[mm], hi[8 + mm]);
            rh[2 * mm + 1] = pack_half2(hi[4 + mm], hi[12 + mm]);
            rl[2 * mm] = pack_half2(lo[mm], lo[8 + mm]);
            rl[2 * mm + 1] = pack_half2(lo[4 + mm], lo[12 + mm]);
        }
        // full-block sums over the 4 threads (b, c = 0..3) = consecutive lanes
        const unsigned grp = 0xFu << (lane & ~3);
        base_hi += __shfl_xor_sync(grp, base_hi, 1);
        base_hi += __shfl_xor_sync(grp, base_hi, 2);
        base_lo += __shfl_xor_sync(grp, base_lo, 1);
        base_lo += __shfl_xor_sync(grp, base_lo, 2);

        // B column 2*jc (hi) is lane group 2*jc, column 2*jc+1 (lo) group 2*jc+1.
        uint8_t *rec = J.prep + kPrepHeader + (size_t(b) * NT + t) * rb;
        const int l_hi = 4 * (2 * jc) + c, l_lo = 4 * (2 * jc + 1) + c;
        *reinterpret_cast<uint4 *>(rec + l_hi * 16) = make_uint4(rh[0], rh[1], rh[2], rh[3]);
        *reinterpret_cast<uint4 *>(rec + 16 * su + l_hi * 16) = make_uint4(rh[4], rh[5], rh[6], rh[7]);
        *reinterpret_cast<uint4 *>(rec + l_lo * 16) = make_uint4(rl[0], rl[1], rl[2], rl[3]);
        *reinterpret_cast<uint4 *>(rec + 16 * su + l_lo * 16) = make_uint4(rl[4], rl[5], rl[6], rl[7]);
        if (c == 0)
            *reinterpret_cast<float2 *>(rec + 32 * su + 8 * jc) = make_float2(-base_hi, -base_lo);
        // Column 0's CTA also clears the slots and starts of columns past ncols
        // in the last tile (the tiles of ncols 5..8 share the 32-slot layout).
        if (j == 0) {
            const int last_t = NT - 1;
            uint8_t *rl_rec = J.prep + kPrepHeader + (size_t(b) * NT + last_t) * rb;
            for (int jj = ncols - 4 * last_t; jj < 4; ++jj) {
                if (8 * jj + 8 > su) break;
                for (int part = 0; part < 2; ++part) {
                    const int l = 4 * (2 * jj + part) + c;
                    *reinterpret_cast<uint4 *>(rl_rec + l * 16) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4 *>(rl_rec + 16 * su + l * 16) = make_uint4(0, 0, 0, 0);
                }
            }
            if (c == 0)
                for (int jj = ncols - 4 * last_t; jj < 4; ++jj)
                    *reinterpret_cast<float2 *>(rl_rec + 32 * su + 8 * jj) = make_float2(0.f, 0.f);
        }
    }
}

// ---------------------------------------------------------------------------
// Tensor-core mat-vec kernel
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1, float c0, float c1,
                                          float c2, float c3) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2),
          "f"(c3));
}

__device__ __forceinline__ uint32_t pick(const uint4 &a, const uint4 &b, int r) {
    switch (r) {
        case 0: return a.x;
        case 1: return a.y;
        case 2: return a.z;
        case 3: return a.w;
        case 4: return b.x;
        case 5: return b.y;
        case 6: return b.z;
        default: return b.w;
    }
}

// fp16 scale at a shared-memory address, as f32.
__device__ __forceinline__ float lds_half_as_float(const uint8_t *p) {
    return __half2float(*reinterpret_cast<const __half *>(p));
}

// Code words and scales of one block pair for a thread's two rows (a, b):
// element u = 0 is the even block (words straddle two aligned words), u = 1 the
// odd block (words aligned).
struct PairRegs {
    uint32_t wa[2], wb[2];
    float da[2], db[2];
};

__device__ __forceinline__ PairRegs load_pair(const uint8_t *row_a, const uint8_t *row_b, int pr,
                                              int c) {
    PairRegs r;
    const uint8_t *pa = row_a + 36 * pr;
    const uint8_t *pb = row_b + 36 * pr;
    r.wa[0] = __byte_perm(*reinterpret_cast<const uint32_t *>(pa + 4 * c),
                          *reinterpret_cast<const uint32_t *>(pa + 4 * c + 4), 0x5432);
    r.wb[0] = __byte_perm(*reinterpret_cast<const uint32_t *>(pb + 4 * c),
                          *reinterpret_cast<const uint32_t *>(pb + 4 * c + 4), 0x5432);
    r.wa[1] = *reinterpret_cast<const uint32_t *>(pa + 20 + 4 * c);
    r.wb[1] = *reinterpret_cast<const uint32_t *>(pb + 20 + 4 * c);
    r.da[0] = lds_half_as_float(pa);
    r.db[0] = lds_half_as_float(pb);
    r.da[1] = lds_half_as_float(pa + 18);
    r.db[1] = lds_half_as_float(pb + 18);
    return r;
}

// One pipeline stage (8 blocks of a thread's rows a = row_a, b = row_a + 8) as
// straight-line code: per block pair, the B fragments (data lanes only) and
// accumulator starts, the two code words and scales per row, then the four MMA
// steps issued step-major across the pair's two chains, then the scaling.
template <int NT>
__device__ __forceinline__ void mv_stage(float (&acc)[NT][4], uint4 (&fr0)[2][NT],
                                         uint4 (&fr1)[2][NT], const uint8_t *row_a,
                                         const uint8_t *rs, int rec_bytes, int su, int lane, int c,
                                         const bool (&lane_used)[NT]) {
    const uint8_t *row_b = row_a + 8 * kChunkBytes;
#pragma unroll
    for (int pr = 0; pr < kChunkBlocks / 2; ++pr) {
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const uint8_t *rec = rs + ((2 * pr + u) * NT + t) * rec_bytes;
                if (lane_used[t]) {  // other lanes keep their zero registers
                    fr0[u][t] = *reinterpret_cast<const uint4 *>(rec + lane * 16);
                    fr1[u][t] = *reinterpret_cast<const uint4 *>(rec + 16 * su + lane * 16);
                }
            }
        const PairRegs cur = load_pair(row_a, row_b, pr, c);
        uint32_t sa[2], sb[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            sa[u] = cur.wa[u] >> 8;
            sb[u] = cur.wb[u] >> 8;
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            float2 st[2];
#pragma unroll
            for (int u = 0; u < 2; ++u)
                st[u] = *reinterpret_cast<const float2 *>(rs + ((2 * pr + u) * NT + t) * rec_bytes +
                                                          32 * su + 8 * c);
            float cc[2][4];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                cc[u][0] = st[u].x;
                cc[u][1] = st[u].y;
                cc[u][2] = st[u].x;
                cc[u][3] = st[u].y;
            }
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const uint32_t mask = 0x00030003u << (2 * m);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    float dd[4];
                    mma_16816(dd, cur.wa[u] & mask, cur.wb[u] & mask, sa[u] & mask, sb[u] & mask,
                              pick(fr0[u][t], fr1[u][t], 2 * m), pick(fr0[u][t], fr1[u][t], 2 * m + 1),
                              cc[u][0], cc[u][1], cc[u][2], cc[u][3]);
                    cc[u][0] = dd[0];
                    cc[u][1] = dd[1];
                    cc[u][2] = dd[2];
                    cc[u][3] = dd[3];
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                acc[t][0] = fmaf(cur.da[u], cc[u][0], acc[t][0]);
                acc[t][1] = fmaf(cur.da[u], cc[u][1], acc[t][1]);
                acc[t][2] = fmaf(cur.db[u], cc[u][2], acc[t][2]);
                acc[t][3] = fmaf(cur.db[u], cc[u][3], acc[t][3]);
            }
        }
    }
}

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

constexpr int kConsumerWarps = kTileRows / 16;  // one 16-row MMA group per warp
constexpr int kCtaThreads = (kConsumerWarps + 1) * 32;

// NT: MMA n-tiles (1 for ncols <= 4, 2 for 5..8).
template <int NT>
__global__ void __launch_bounds__(kCtaThreads, 1)
    mv_tc_kernel(const __grid_constant__ MvJob single, const MvParams p) {
    // The next prep launch on the stream may become resident now; it waits for
    // this grid before it touches any buffer this kernel reads.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int kCW = kConsumerWarps;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int kStages = p.n_stages;
    const int su = used_slots(p.ncols), kRecBytes = rec_bytes(p.ncols);
    const int kRStageBytes = kChunkBlocks * NT * kRecBytes;
    uint8_t *w_stage = smem;                               // kStages x kWStageBytes
    uint8_t *r_stage = smem + kStages * kWStageBytes;      // kStages x kRStageBytes
    uint64_t *full = reinterpret_cast<uint64_t *>(r_stage + kStages * kRStageBytes);
    uint64_t *empty = full + kMaxStages;
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kCW);
        }
        s_abort = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // This CTA's work list.
    int n_items, item_base = 0;
    if (p.jobs) {
        item_base = p.cta_begin[blockIdx.x];
        n_items = p.cta_begin[blockIdx.x + 1] - item_base;
    } else {
        n_items = blockIdx.x < unsigned(single.n_tiles)
                      ? (single.n_tiles - 1 - int(blockIdx.x)) / int(gridDim.x) + 1
                      : 0;
    }
    auto item_at = [&](int i, const MvJob *&J, int &tile) {
        if (p.jobs) {
            const MvItem it = p.items[item_base + i];
            J = &p.jobs[it.job];
            tile = it.tile;
        } else {
            J = &single;
            tile = int(blockIdx.x) + i * int(gridDim.x);
        }
    };

    if (warp == kCW) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true, prep_ready = false;
            for (int i = 0; i < n_items && ok; ++i) {
                const MvJob *J;
                int tile;
                item_at(i, J, tile);
                const int nch = J->n_chunks;
                for (int ch = 0; ch < nch; ++ch) {
                    if (!mbar_wait(&empty[stage], ph ^ 1u, p.err, kTagMvEmpty) ||
                        *(volatile int *)&s_abort) {
                        ok = false;
                        s_abort = 1;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], kWStageBytes + kRStageBytes);
                    tma_load_2d(w_stage + stage * kWStageBytes, &J->tmap, ch * kChunkBytes,
                                tile * kTileRows, &full[stage]);
                    if (!prep_ready) {
                        // The activation fragments come from the preceding kernel.
                        grid_dependency_wait();
                        prep_ready = true;
                    }
                    bulk_g2s(r_stage + stage * kRStageBytes,
                             J->prep + kPrepHeader + size_t(ch) * kRStageBytes, kRStageBytes,
                             &full[stage]);
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Let copies already issued land before the CTA exits (bounded).
                int st = stage, pp = ph;
                for (int k = 0; k < kStages && k < issued; ++k) {
                    if (--st < 0) {
                        st = kStages - 1;
                        pp ^= 1;
                    }
                    mbar_wait(&full[st], uint32_t(pp), p.err, kTagMvFull);
                }
            }
        }
        return;
    }

    // ------------------------------ consumers ------------------------------
    grid_dependency_wait();  // the epilogue reads the column scales written by prep
    const int g = lane >> 2, c = lane & 3;
    // Lane groups g < 2 * (columns of tile t) carry B data.
    bool lane_used[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) lane_used[t] = g < 2 * min(4, p.ncols - 4 * t);

    // B-fragment registers of a block pair; lanes that carry no column keep zeros.
    uint4 fr0[2][NT], fr1[2][NT];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int t = 0; t < NT; ++t) fr0[u][t] = fr1[u][t] = make_uint4(0, 0, 0, 0);

    int stage = 0;
    uint32_t ph = 0;
    for (int i = 0; i < n_items; ++i) {
        const MvJob *J;
        int tile;
        item_at(i, J, tile);
        const int n_chunks = J->n_chunks;
        float acc[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[t][k] = 0.0f;

        bool ok = true;
        for (int ch = 0; ch < n_chunks; ++ch) {
            const bool got = mbar_wait(&full[stage], ph, p.err, kTagMvFull) &&
                             !*(volatile int *)&s_abort;
            if (!__all_sync(0xffffffffu, got)) {  // warp-uniform decision
                s_abort = 1;
                ok = false;
                break;
            }
            mv_stage<NT>(acc, fr0, fr1, w_stage + stage * kWStageBytes + (warp * 16 + g) * kChunkBytes,
                         r_stage + stage * kRStageBytes, kRecBytes, su, lane, c, lane_used);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == kStages) {
                stage = 0;
                ph ^= 1u;
            }
        }
        if (!ok) break;

        // ---- epilogue: hi + lo of column 4t + c, undo the column scale, store ----
        const float *out_scale = reinterpret_cast<const float *>(J->prep);
        const int N = J->N;
        const int row_a = tile * kTileRows + warp * 16 + g;
        const int row_b = row_a + 8;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int col = 4 * t + c;
            if (col < p.ncols) {
                const float sc = out_scale[col];
                if (row_a < N) J->y[size_t(col) * N + row_a] = (acc[t][0] + acc[t][1]) * sc;
                if (row_b < N) J->y[size_t(col) * N + row_b] = (acc[t][2] + acc[t][3]) * sc;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// tcgen05 mat-vec (ncols 1..3)
//
// The codes become tensor-core operands without any arithmetic: byte j of a
// code word holds elements 4j..4j+3 at bits 0-1, 2-3, 4-5, 6-7, and read as
// e4m3 a byte whose only set bits are 0-1 is the subnormal q * 2^-9, one whose
// only set bits are 2-3 is q * 2^-7 (bit 2 is the top mantissa bit, bit 3 the
// lowest exponent bit: 0, 2^-7, 2^-6, 1.5 * 2^-6). So word & 0x03030303,
// word & 0x0C0C0C0C, (word >> 4) & 0x03030303 and (word >> 4) & 0x0C0C0C0C are
// four registers of exact e4m3 weights, one logic op each. Four expansion
// warps per 128-row tile store them into tensor memory (one row per TMEM lane)
// and one thread issues tcgen05.mma kind::f8f6f4 (M = 128, N = 16, K = 32)
// with A in TMEM and B = the activations as e4m3 pieces in shared memory.
//
// Activations as e4m3 pieces. Per column j, u = x * 2^s_j with max|u| in
// [2^-2, 2^-1); element e gives v = u * 2^9 (codes at bits 0-1) or u * 2^7
// (bits 2-3), split into kT5Pieces e4m3 values: piece p = e4m3(r_p * 2^4p),
// r_0 = v, r_{p+1} = r_p - piece_p * 2^-4p; each rounding keeps 4 significant
// bits, so the residual after 5 pieces is below 2^-20 |v|. Piece p of column j
// is B row n = 5j + p. A block's MMA result per row is then C_n = sum q *
// piece_n / (2^9 or 2^7).
//
// Per block accumulators. d changes every 64 weights of a row, so each block
// gets its own accumulator columns; the epilogue loads them and forms, per
// row and column,
//   t = sum_p 2^-4p C_(5j+p) - beta_j,   acc_j += d * t,
// where beta_j is the same sum for all-ones codes (the "- 1" of (q - 1)),
// computed by the preparation kernel with the same f32 operations from exact
// per-piece sums, so that all-ones blocks give exactly 0. With one column
// (5 pieces) two blocks share a 16-column accumulator: the even block's pieces
// are B rows 0-4 and the odd block's rows 8-12, each block's other rows zero,
// and the odd block's MMAs accumulate onto the even block's result. With 2-3
// columns each block has its own 16 columns.
//
// Pipeline per CTA (persistent over 128-row tiles), stage = 8 blocks:
//   warp 2      streams the stage's TMA box (144 B x 128 rows) and, by bulk
//               copy, its B image and betas into an 8-deep shared-memory ring;
//   warps 4-11  expand the stage's codes into a TMEM A buffer (3 buffers with
//               one column, 2 with 2-3; warps 4-7 blocks 0-3, warps 8-11 blocks
//               4-7; warp w owns TMEM lanes 32 (w % 4) .. +31, i.e. those rows);
//   warp 3      issues the stage's 16 MMAs into one of two TMEM D buffers and
//               commits them to the expansion (A free) and epilogue (D full)
//               barriers. The whole warp runs the loop and waits, and the
//               elected lane issues: from a lone lane each MMA cost ~70 cycles
//               to issue, and a warp diverged around the waits took ~200 cycles
//               to reconverge;
//   warps 12-15 epilogue, one row per thread: D, the row's d values from the
//               ring and the betas; they release the D buffer and the ring slot.
// The expansion of a stage waits for the MMAs that last read its A buffer, so
// the A buffer count sets how far expansion runs ahead of the tensor core.
// ---------------------------------------------------------------------------
constexpr int kT5Rows = 128;
constexpr int kT5Pieces = 5;
constexpr int kT5MaxCols = 3;                         // 5 * 3 pieces fit N = 16
constexpr int kT5N = 16;
constexpr int kT5Stages = 8;
constexpr int kT5RawBytes = kT5Rows * kChunkBytes;   // 18432
constexpr int kT5ImgBytes = kT5N * kChunkBlocks * 64; // 8192: 16 rows x 512 K bytes, SW128
constexpr int kT5BetaBytes = kChunkBlocks * 4 * 4;   // beta[8 blocks][4 columns] f32
constexpr int kT5PrepHeader = 1024;                  // int col_shift[8], images 1024-aligned
constexpr int kT5ExpWarps = 4;
constexpr int kT5EpiWarps = 4;
// Warp roles. A warp reaches only the TMEM lanes of its quarter (warp % 4), so
// each quarter hosts 1 expansion warp and 1 epilogue warp (12 warps in all: a
// second expansion warp per quarter measured slower at ncols 2 and no faster
// at 3). Two MMA issuers (even and odd stages) sit on warps 1 and 3, the
// producer on warp 2.
constexpr int kT5ProdWarp = 2;
constexpr int kT5MmaWarp = 3;    // even stages; allocates TMEM
constexpr int kT5MmaWarp2 = 1;   // odd stages
constexpr int kT5ExpWarp0 = 4;   // warps 4-7
constexpr int kT5EpiWarp0 = 8;   // warps 8-11
constexpr int kT5Warps = kT5EpiWarp0 + kT5EpiWarps;
constexpr int kT5Threads = kT5Warps * 32;
constexpr int kT5MaxABufs = 3;
constexpr int kT5Smem = 1024 /* alignment slack */ +
                        kT5Stages * (kT5ImgBytes + kT5RawBytes + kT5BetaBytes) +
                        (2 * kT5Stages + 2 * kT5MaxABufs + 4) * 8;
// TMEM columns (512): A buffers of 128 (8 blocks x 16 columns of 4 e4m3), then
// two D buffers of 64 (one column: 4 block pairs x 16) or 128 (8 blocks x 16).
__host__ __device__ constexpr int t5_abufs(int nc) { return nc == 1 ? 3 : 2; }
__host__ __device__ constexpr int t5_dcols(int nc) { return nc == 1 ? 64 : 128; }
static_assert(t5_abufs(1) * 128 + 2 * t5_dcols(1) <= 512, "TMEM budget");
static_assert(t5_abufs(2) * 128 + 2 * t5_dcols(2) <= 512, "TMEM budget");
constexpr int kTagT5Full = 111;
constexpr int kTagT5Empty = 112;
constexpr int kTagT5AFull = 113;
constexpr int kTagT5DFull = 114;
constexpr int kTagT5DEmpty = 115;

size_t t5_prep_bytes(int64_t K) {
    const size_t n_chunks = size_t(K / 512);
    size_t b = kT5PrepHeader + n_chunks * (kT5ImgBytes + kT5BetaBytes);
    return (b + 255) & ~size_t(255);
}

// Byte offset of element (row n, K position kc) of one stage's B image: K-major
// rows of 128 bytes in atoms of 8 rows (1024 B); the 16-byte chunk index is
// XOR-ed with the row within the atom (128-byte swizzle); 4 atom columns of
// 128 K bytes (2 KB each: rows 0-7, then rows 8-15).
__host__ __device__ constexpr int t5_img_offset(int n, int kc) {
    return (kc >> 7) * 2048 + (n >> 3) * 1024 + (n & 7) * 128 +
           ((((kc & 127) >> 4) ^ (n & 7)) << 4) + (kc & 15);
}

// Preparation: grid (ncols, n_jobs), kPrepThreads threads. Thread (block b,
// word c, r) handles the 4 elements 16c + 4jj + r (jj = 0..3) of block b and
// writes, per piece, one 32-bit word of the B image: K positions 64 (b % 8) +
// 16c + 4r + jj (the order the expansion warps store codes in TMEM: column
// 4c + r of a block holds elements 16c + 4jj + r in byte jj). The per-piece
// all-ones sums are exact integers in units of 2^-18 (a piece is a multiple of
// 2^-9, divided by 2^9 or 2^7; |sum| < 64 * 448 * 2^-7), rounded once to f32.
constexpr int kT5PrepThreads = 256;

template <typename XT>
__global__ void __launch_bounds__(kT5PrepThreads) t5_prep_kernel(
    const __grid_constant__ MvPrepJob single, const MvPrepJob *__restrict__ jobs, int ncols) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Launched as a programmatic dependent of the kernel before it on the stream
    // (a mat-vec that may still read this buffer, or the producer of x): wait
    // for that grid before reading x or writing the prep buffer.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const MvPrepJob &J = jobs ? jobs[blockIdx.y] : single;
    const int K = J.K;
    const int j = blockIdx.x;
    const XT *xj = static_cast<const XT *>(J.x) + size_t(j) * K;
    const int tid = threadIdx.x;
    const int nb = K / 64;
    const int n_chunks = K / 512;
    // grid z splits a column's 16 * nb items (one per thread, grid-stride for
    // very long columns); the CTAs past this column's items have nothing to do
    if (int(blockIdx.z) * kT5PrepThreads >= nb * 16) return;

    // 1) column scale 2^s with max|x * 2^s| in [2^-2, 2^-1) (each CTA of the
    //    column reads the whole column)
    float m = 0.0f;
    if (sizeof(XT) == 4 && (reinterpret_cast<uintptr_t>(xj) & 15u) == 0) {
        const float4 *x4 = reinterpret_cast<const float4 *>(xj);
        for (int k = tid; k < K / 4; k += kT5PrepThreads) {
            const float4 f = x4[k];
            m = fmaxf(m, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
        }
    } else {
        for (int k = tid; k < K; k += kT5PrepThreads) m = fmaxf(m, fabsf(ld_x(xj + k)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float red[kT5PrepThreads / 32];
    if ((tid & 31) == 0) red[tid >> 5] = m;
    __syncthreads();
    float amax = red[0];
#pragma unroll
    for (int w = 1; w < kT5PrepThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    int s = 0;
    if (amax > 0.0f && amax <= 3.4e38f) {
        int e;
        frexpf(amax, &e);  // amax = f * 2^e, f in [0.5, 1)
        s = -e - 1;
    }
    int *col_shift = reinterpret_cast<int *>(J.prep);
    if (blockIdx.z == 0 && tid == 0) col_shift[j] = s;

    // 2) pieces
    uint8_t *img = J.prep + kT5PrepHeader;
    float *beta = reinterpret_cast<float *>(img + size_t(n_chunks) * kT5ImgBytes);
    const int lane = tid & 31;
    const unsigned grp = 0xFFFFu << (lane & 16);  // the block's 16 threads
    for (int idx = int(blockIdx.z) * kT5PrepThreads + tid; idx < nb * 16;
         idx += int(gridDim.z) * kT5PrepThreads) {
        const int b = idx >> 4, c = (idx >> 2) & 3, r = idx & 3;
        const XT *xe = xj + b * 64 + c * 16 + r;
        const int e_in = s + ((r & 1) ? 7 : 9);    // v = x * 2^e_in
        const float to_int = (r & 1) ? 2048.0f : 512.0f;  // piece / (2^7 or 2^9) in 2^-18 units
        float v[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) v[jj] = mul_pow2(ld_x(xe + 4 * jj), e_in);
        uint8_t *bimg = img + size_t(b >> 3) * kT5ImgBytes;
        const int kc = 64 * (b & 7) + 16 * c;
        int isum[kT5Pieces];
#pragma unroll
        for (int p = 0; p < kT5Pieces; ++p) {
            const float up = __int_as_float((127 + 4 * p) << 23);
            const float down = __int_as_float((127 - 4 * p) << 23);
            const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                make_float2(v[0] * up, v[1] * up), __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                make_float2(v[2] * up, v[3] * up), __NV_SATFINITE, __NV_E4M3);
            const float2 plo = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(lo, __NV_E4M3)));
            const float2 phi = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3)));
            v[0] -= plo.x * down;
            v[1] -= plo.y * down;
            v[2] -= phi.x * down;
            v[3] -= phi.y * down;
            isum[p] = __float2int_rn(plo.x * to_int) + __float2int_rn(plo.y * to_int) +
                      __float2int_rn(phi.x * to_int) + __float2int_rn(phi.y * to_int);
            // one column: the block's pieces are rows 0-4 (even block) or 8-12 (odd)
            const int n = ncols == 1 ? 8 * (b & 1) + p : kT5Pieces * j + p;
            *reinterpret_cast<uint32_t *>(bimg + t5_img_offset(n, kc) + 4 * r) =
                uint32_t(lo) | (uint32_t(hi) << 16);
        }
        if (ncols == 1) {
            // the rows the other block of the pair reads its result from stay zero
            for (int n = 8 * (1 - (b & 1)); n < 8 * (1 - (b & 1)) + 8; ++n)
                *reinterpret_cast<uint32_t *>(bimg + t5_img_offset(n, kc) + 4 * r) = 0u;
        }
        float base[kT5Pieces];
#pragma unroll
        for (int p = 0; p < kT5Pieces; ++p) {
            int t = isum[p];
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) t += __shfl_xor_sync(grp, t, o);
            base[p] = float(t) * 0x1p-18f;
        }
        if ((idx & 15) == 0) {
            // the epilogue's combination, applied to the all-ones results
            float t = base[4] * 0x1p-16f;
            t = fmaf(base[3], 0x1p-12f, t);
            t = fmaf(base[2], 0x1p-8f, t);
            t = fmaf(base[1], 0x1p-4f, t);
            t = t + base[0];
            beta[size_t(b >> 3) * (kT5BetaBytes / 4) + (b & 7) * 4 + j] = t;
        }
    }
}

// kind::f8f6f4 instruction descriptor: D f32, A and B e4m3, both K-major, N, M.
__host__ __device__ constexpr uint32_t idesc_e4m3(int m, int n) {
    return (1u << 4) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

// NC: activation columns (1..3).
template <int NC>
__global__ void __launch_bounds__(kT5Threads, 1)
    mv_t5_kernel(const __grid_constant__ MvJob single, const MvParams p) {
    // The next prep launch on the stream may become resident now; it waits for
    // this grid before it touches any buffer this kernel reads.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int kABufs = t5_abufs(NC);
    constexpr int kDCols = t5_dcols(NC);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *img_ring = smem;                                      // kT5Stages x 8 KB
    uint8_t *raw_ring = img_ring + kT5Stages * kT5ImgBytes;         // kT5Stages x 18 KB
    uint8_t *beta_ring = raw_ring + kT5Stages * kT5RawBytes;        // kT5Stages x 128 B
    uint64_t *full = reinterpret_cast<uint64_t *>(beta_ring + kT5Stages * kT5BetaBytes);
    uint64_t *empty = full + kT5Stages;        // arrived by the 4 epilogue warps
    uint64_t *a_full = empty + kT5Stages;      // [kABufs] arrived by the 8 expansion warps
    uint64_t *a_empty = a_full + kT5MaxABufs;  // [kABufs] tcgen05.commit
    uint64_t *d_full = a_empty + kT5MaxABufs;  // [2] tcgen05.commit
    uint64_t *d_empty = d_full + 2;            // [2] arrived by the 4 epilogue warps
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kT5Stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kT5EpiWarps);
        }
        for (int i = 0; i < kABufs; ++i) {
            mbar_init(&a_full[i], kT5ExpWarps);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], kT5EpiWarps);
        }
        s_abort = 0;
        fence_barrier_init();
    }
    if (warp == kT5MmaWarp) {
        tmem_alloc(&s_tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    int n_items, item_base = 0;
    if (p.jobs) {
        item_base = p.cta_begin[blockIdx.x];
        n_items = p.cta_begin[blockIdx.x + 1] - item_base;
    } else {
        n_items = blockIdx.x < unsigned(single.n_tiles)
                      ? (single.n_tiles - 1 - int(blockIdx.x)) / int(gridDim.x) + 1
                      : 0;
    }
    auto item_at = [&](int i, const MvJob *&J, int &tile) {
        if (p.jobs) {
            const MvItem it = p.items[item_base + i];
            J = &p.jobs[it.job];
            tile = it.tile;
        } else {
            J = &single;
            tile = int(blockIdx.x) + i * int(gridDim.x);
        }
    };
    auto stage_parity = [](int s) { return uint32_t(s / kT5Stages) & 1u; };
    // A buffer of stage s and the parity of its use; D buffer likewise
    auto a_buf = [](int s) { return s % kABufs; };
    auto a_use = [](int s) { return uint32_t(s / kABufs) & 1u; };
    auto a_col = [&](int s) { return uint32_t(a_buf(s) * 128); };
    auto d_col = [&](int s) { return uint32_t(kABufs * 128 + (s & 1) * kDCols); };

    if (warp == kT5ProdWarp) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            int s = 0;
            bool ok = true, prep_ready = false;
            for (int i = 0; i < n_items && ok; ++i) {
                const MvJob *J;
                int tile;
                item_at(i, J, tile);
                const uint8_t *img = J->prep + kT5PrepHeader;
                const uint8_t *beta = img + size_t(J->n_chunks) * kT5ImgBytes;
                const int nch = J->n_chunks;
                for (int ch = 0; ch < nch; ++ch, ++s) {
                    const int st = s % kT5Stages;
                    if (!mbar_wait(&empty[st], stage_parity(s) ^ 1u, p.err, kTagT5Empty, true) ||
                        *(volatile int *)&s_abort) {
                        ok = false;
                        s_abort = 1;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[st], kT5RawBytes + kT5ImgBytes + kT5BetaBytes);
                    tma_load_2d(raw_ring + st * kT5RawBytes, &J->tmap, ch * kChunkBytes,
                                tile * kT5Rows, &full[st]);
                    if (!prep_ready) {
                        grid_dependency_wait();  // the B images come from the prep kernel
                        prep_ready = true;
                    }
                    bulk_g2s(img_ring + st * kT5ImgBytes, img + size_t(ch) * kT5ImgBytes,
                             kT5ImgBytes, &full[st]);
                    bulk_g2s(beta_ring + st * kT5BetaBytes, beta + size_t(ch) * kT5BetaBytes,
                             kT5BetaBytes, &full[st]);
                }
            }
            if (!ok) {
                // let copies already issued land (bounded) before the CTA exits
                for (int k = 1; k <= kT5Stages && s - k >= 0; ++k)
                    mbar_wait(&full[(s - k) % kT5Stages], stage_parity(s - k), p.err, kTagT5Full);
            }
        }
    } else if (warp == kT5MmaWarp || warp == kT5MmaWarp2) {
        // ------------------------------ MMA issuers ------------------------------
        // Each issuer's per-stage control path (barrier checks, fence, issue,
        // commits) takes about a stage's worth of time, so two issuers take
        // the even and the odd stages (D buffer = stage parity; consecutive
        // uses of an A buffer are ordered through its expansion). The whole
        // warp runs the loop and waits (addresses and descriptors stay
        // warp-uniform, and the warp stays converged); the elected lane issues
        // the MMAs and commits them.
        constexpr uint32_t idesc = idesc_e4m3(kT5Rows, kT5N);
        const bool leader = elect_one();
        const int parity = warp == kT5MmaWarp ? 0 : 1;
        const uint64_t desc0 = sw128_desc(smem_addr(img_ring));
        int s = 0, last = -1;
        bool ok = true;
        for (int i = 0; i < n_items && ok; ++i) {
            const MvJob *J;
            int tile;
            item_at(i, J, tile);
            const int nch = J->n_chunks;
            for (int ch = 0; ch < nch; ++ch, ++s) {
                if ((s & 1) != parity) continue;
                const int st = s % kT5Stages;
                const bool got =
                    mbar_wait(&full[st], stage_parity(s), p.err, kTagT5Full) &&
                    mbar_wait(&a_full[a_buf(s)], a_use(s), p.err, kTagT5AFull) &&
                    mbar_wait(&d_empty[s & 1], (uint32_t(s >> 1) & 1u) ^ 1u, p.err,
                              kTagT5DEmpty) &&
                    !*(volatile int *)&s_abort;
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a_base = tmem + a_col(s);
                const uint32_t d_base = tmem + d_col(s);
                // descriptor start-address field advanced by the byte offset / 16
                const uint64_t dst = desc0 + uint64_t((st * kT5ImgBytes) >> 4);
                if (leader) {
#pragma unroll
                    for (int b = 0; b < kChunkBlocks; ++b)
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            // one column: blocks 2i, 2i+1 share accumulator i
                            const uint32_t dcol = NC == 1 ? (b >> 1) * kT5N : b * kT5N;
                            const uint32_t accum = NC == 1 ? uint32_t((b & 1) | kk) : uint32_t(kk);
                            tc_mma_f8f6f4_ta(d_base + dcol, a_base + b * 16 + kk * 8,
                                             dst + uint64_t(((b >> 1) * 2048 + (b & 1) * 64 +
                                                             kk * 32) >> 4),
                                             idesc, accum);
                        }
                    tc_commit(&a_empty[a_buf(s)]);
                    tc_commit(&d_full[s & 1]);
                }
                __syncwarp();
                last = s;
            }
        }
        if (last >= 0)  // TMEM is freed only after the last MMAs completed
            mbar_wait(&d_full[last & 1], uint32_t(last >> 1) & 1u, p.err, kTagT5DFull);
    } else if (warp >= kT5ExpWarp0 && warp < kT5ExpWarp0 + kT5ExpWarps) {
        // ------------------------------ expansion ------------------------------
        // warp w: TMEM lane quarter w % 4 (rows 32 (w % 4) ..), all 8 blocks
        const int qd = warp & 3;
        const int row = 32 * qd + lane;
        const uint32_t lane_base = uint32_t(32 * qd) << 16;
        int s = 0;
        bool ok = true;
        for (int i = 0; i < n_items && ok; ++i) {
            const MvJob *J;
            int tile;
            item_at(i, J, tile);
            const int nch = J->n_chunks;
            for (int ch = 0; ch < nch; ++ch, ++s) {
                const int st = s % kT5Stages;
                const bool got =
                    mbar_wait(&full[st], stage_parity(s), p.err, kTagT5Full) &&
                    mbar_wait(&a_empty[a_buf(s)], a_use(s) ^ 1u, p.err, kTagT5AFull) &&
                    !*(volatile int *)&s_abort;
                if (!__all_sync(0xffffffffu, got)) {
                    s_abort = 1;
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int G = 0; G < 2; ++G) {
                    const uint8_t *rp = raw_ring + st * kT5RawBytes + row * kChunkBytes + G * 72;
                    uint32_t u[18];
#pragma unroll
                    for (int k = 0; k < 9; ++k) {
                        const uint2 v = *reinterpret_cast<const uint2 *>(rp + 8 * k);
                        u[2 * k] = v.x;
                        u[2 * k + 1] = v.y;
                    }
                    const uint32_t a_base = tmem + lane_base + a_col(s) + 4 * G * 16;
#pragma unroll
                    for (int bi = 0; bi < 4; ++bi) {
                        uint32_t a[16];
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint32_t w;
                            if (bi == 0) w = __byte_perm(u[c], u[c + 1], 0x5432);
                            else if (bi == 1) w = u[5 + c];
                            else if (bi == 2) w = __byte_perm(u[9 + c], u[10 + c], 0x5432);
                            else w = u[14 + c];
                            const uint32_t hw = w >> 4;
                            a[4 * c + 0] = w & 0x03030303u;
                            a[4 * c + 1] = w & 0x0C0C0C0Cu;
                            a[4 * c + 2] = hw & 0x03030303u;
                            a[4 * c + 3] = hw & 0x0C0C0C0Cu;
                        }
                        tmem_st16(a_base + bi * 16, a);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[a_buf(s)]);
            }
        }
    } else if (warp >= kT5EpiWarp0) {
        // ------------------------------ epilogue ------------------------------
        // warp w: TMEM lane quarter w % 4; one row per thread, all 8 blocks.
        grid_dependency_wait();  // reads the column shifts written by prep
        const int qd = warp & 3;
        const int row = 32 * qd + lane;
        const uint32_t lane_base = uint32_t(32 * qd) << 16;
        float acc[NC];
#pragma unroll
        for (int j = 0; j < NC; ++j) acc[j] = 0.0f;
        int s = 0;
        bool ok = true;
        for (int i = 0; i < n_items && ok; ++i) {
            const MvJob *J;
            int tile;
            item_at(i, J, tile);
            const int nch = J->n_chunks;
            for (int ch = 0; ch < nch; ++ch, ++s) {
                const int st = s % kT5Stages;
                const bool got =
                    mbar_wait(&full[st], stage_parity(s), p.err, kTagT5Full) &&
                    mbar_wait(&d_full[s & 1], uint32_t(s >> 1) & 1u, p.err, kTagT5DFull) &&
                    !*(volatile int *)&s_abort;
                if (!__all_sync(0xffffffffu, got)) {
                    s_abort = 1;
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_base = tmem + lane_base + d_col(s);
                const uint8_t *rp = raw_ring + st * kT5RawBytes + row * kChunkBytes;
                const float *bt = reinterpret_cast<const float *>(beta_ring + st * kT5BetaBytes);
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {
                    // blocks 4hb .. 4hb+3: C[bi][n] = accumulator column n of block 4hb+bi
                    float C[4][NC * 5];
                    if (NC == 1) {
                        uint32_t r[2][16];
#pragma unroll
                        for (int pi = 0; pi < 2; ++pi)
                            tmem_ld16(d_base + (2 * hb + pi) * kT5N, r[pi]);
                        tmem_wait_ld();
#pragma unroll
                        for (int bi = 0; bi < 4; ++bi)
#pragma unroll
                            for (int n = 0; n < 5; ++n)
                                C[bi][n] = __uint_as_float(r[bi >> 1][8 * (bi & 1) + n]);
                    } else {
                        uint32_t r[4][16];
#pragma unroll
                        for (int bi = 0; bi < 4; ++bi)
                            tmem_ld16(d_base + (4 * hb + bi) * kT5N, r[bi]);
                        tmem_wait_ld();
#pragma unroll
                        for (int bi = 0; bi < 4; ++bi)
#pragma unroll
                            for (int n = 0; n < NC * 5; ++n) C[bi][n] = __uint_as_float(r[bi][n]);
                    }
#pragma unroll
                    for (int bi = 0; bi < 4; ++bi) {
                        const int b = 4 * hb + bi;
                        const float d = lds_half_as_float(rp + 18 * b);
#pragma unroll
                        for (int j = 0; j < NC; ++j) {
                            const float *c = &C[bi][5 * j];
                            float t = c[4] * 0x1p-16f;
                            t = fmaf(c[3], 0x1p-12f, t);
                            t = fmaf(c[2], 0x1p-8f, t);
                            t = fmaf(c[1], 0x1p-4f, t);
                            t = t + c[0];
                            acc[j] = fmaf(d, t - bt[b * 4 + j], acc[j]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&d_empty[s & 1]);
                    mbar_arrive(&empty[st]);
                }
                if (ch == nch - 1) {
                    const int *col_shift = reinterpret_cast<const int *>(J->prep);
                    const int r = tile * kT5Rows + row;
                    if (r < J->N)
#pragma unroll
                        for (int j = 0; j < NC; ++j)
                            J->y[size_t(j) * J->N + r] = mul_pow2(acc[j], -col_shift[j]);
#pragma unroll
                    for (int j = 0; j < NC; ++j) acc[j] = 0.0f;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kT5MmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// tcgen05 mat-vec on packed fp4 (ncols = 1)
//
// The codes are exact e2m1 values without arithmetic as well: e2m1 is sign,
// two exponent bits, one mantissa bit, and a nibble whose only set bits are
// the low two (exponent bit 0, mantissa) reads as 0, 0.5, 1, 1.5 = q / 2. With
// each code at bits 2i of a word, word & 0x33333333 holds the even elements
// 0, 2, .., 14 as eight packed e2m1 values and (word >> 2) & 0x33333333 the odd
// ones: 16 weights per shift and two logic ops. tcgen05.mma kind::mxf4 takes
// K = 64 (a whole block) per instruction with A in TMEM; its per-32-element
// ue8m0 scales are all 1.0 (0x7F), so it multiplies the e2m1 values as they are.
//
// Activations, block by block. For block b of the vector (64 elements) with
// M_b = max |x| over the block, M_b = f * 2^e (f in [0.5, 1)), the prep kernel
// forms v = x * 2^(2 - e) (max |v| in [2, 4)) and splits it into 16 e2m1 pieces:
// piece p = e2m1(r_p * 4^p), r_0 = v, r_(p+1) = r_p - piece_p * 4^-p. Every
// subtraction is exact, the scaled residual after the first piece stays within
// [-2, 2], and |r_16| <= 2^-32, so each element keeps its value to 2^-33 of its
// own block's maximum (not of the whole vector's). Piece p is B row p.
//
// The "- 1" of (q - 1) without cancellation. With A = q / 2 the MMA gives, per
// row and piece, C_p = sum_k (q_k / 2) piece_pk, an exact f32 (multiples of 1/4
// below 2^9). The prep kernel computes the same sums for all-ones codes,
// B_p = sum_k piece_pk / 2, and stores them combined in three groups,
//   H = sum_{p<6} 4^-p B_p,  M = sum_{6<=p<12} 4^-p B_p,  L = sum_{p>=12} 4^-p B_p,
// each of which spans fewer than 24 bits and is therefore exact in f32. The
// epilogue forms the same three groups of C (also exact) and subtracts group by
// group, so the element of a zero weight cancels exactly however large it is;
// the one rounding left, (H_C - H) + (M_C - M) + (L_C - L), is relative to the
// sum over the nonzero weights. The block's contribution is d * t * 2^(e - 1).
// Per stage the 8 block contributions are summed in f32 and the stage sums are
// added with a compensated (two-sum) accumulation, so the accumulated rounding
// does not grow with K.
// ---------------------------------------------------------------------------
constexpr int kT4Pieces = 16;
constexpr int kT4ImgBytes = kT5N * kChunkBlocks * 32;  // 4096: 16 rows x 256 bytes (512 e2m1)
// per block of a stage: float {2^(e - 1), H, M, L}
constexpr int kT4BlockRec = 4;
constexpr int kT4BetaBytes = kChunkBlocks * kT4BlockRec * 4;  // 128
constexpr int kT4ABufs = 3;
constexpr int kT4ACol = 256;                           // A buffers at 256 + 64 i
constexpr int kT4ScaleCol = 448;                       // scales A 448..451, B 452..455
// mbarriers: full / empty per stage, a_full / a_empty per A buffer, d_full /
// d_empty per D buffer, a drain per MMA issuer
constexpr int kT4Barriers = 2 * kT5Stages + 2 * kT4ABufs + 2 * 2 + 2;
constexpr int kT4Smem = 1024 /* alignment slack */ +
                        kT5Stages * (kT4ImgBytes + kT5RawBytes + kT4BetaBytes) +
                        kT4Barriers * 8;
static_assert(kT4Pieces == kT5N, "one B row per piece");

size_t t4_prep_bytes(int64_t K) {
    const size_t n_chunks = size_t(K / 512);
    size_t b = kT5PrepHeader + n_chunks * (kT4ImgBytes + kT4BetaBytes);
    return (b + 255) & ~size_t(255);
}

// kind::mxf4 instruction descriptor: A and B e2m1 (1), N, scales ue8m0, M.
__host__ __device__ constexpr uint32_t idesc_mxf4(int m, int n) {
    return (1u << 7) | (1u << 10) | (uint32_t(n >> 3) << 17) | (1u << 23) |
           (uint32_t(m >> 4) << 24);
}

// 2^k as a float for k in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float pow2f(int k) {
    return k >= -126 ? __int_as_float((127 + k) << 23) : __int_as_float(1 << (149 + k));
}

// Preparation: grid (1, n_jobs, z), kT5PrepThreads threads. Item (block b,
// word c, parity h): the 8 elements 16c + 2j + h (j = 0..7) of block b, one
// 32-bit word of the B image per piece (K positions 64 (b % 8) + 16c + 8h + j,
// nibble j). The 8 items of a block are 8 consecutive lanes: they share the
// block maximum and sum the all-ones groups H, M, L by shuffles (every partial
// sum is exact).
template <typename XT>
__global__ void __launch_bounds__(kT5PrepThreads) t4_prep_kernel(
    const __grid_constant__ MvPrepJob single, const MvPrepJob *__restrict__ jobs) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Launched as a programmatic dependent of the kernel before it on the stream
    // (a mat-vec that may still read this buffer, or the producer of x): wait
    // for that grid before reading x or writing the prep buffer.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    MvPrepJob J = jobs ? jobs[blockIdx.y] : single;
    if (!jobs) {  // a strided batch of vectors, one per grid row
        J.x = static_cast<const uint8_t *>(single.x) + size_t(blockIdx.y) * single.x_stride;
        J.prep = single.prep + size_t(blockIdx.y) * single.prep_stride;
    }
    const int K = J.K;
    const XT *xj = static_cast<const XT *>(J.x);
    const int nb = K / 64;
    const int n_chunks = K / 512;
    uint8_t *img = J.prep + kT5PrepHeader;
    float *brec = reinterpret_cast<float *>(img + size_t(n_chunks) * kT4ImgBytes);
    const int lane = threadIdx.x & 31;
    const unsigned grp = 0xFFu << (lane & 24);  // the block's 8 threads
    // 8 items per block and nb blocks: whole warps share a block range, so the
    // shuffles below always run with all 8 lanes of a block present
    for (int idx = int(blockIdx.z) * kT5PrepThreads + int(threadIdx.x); idx < nb * 8;
         idx += int(gridDim.z) * kT5PrepThreads) {
        const int b = idx >> 3, c = (idx >> 1) & 3, h = idx & 1;
        const XT *xe = xj + b * 64 + c * 16 + h;
        float v[8];
        float m = 0.0f;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            v[jj] = ld_x(xe + 2 * jj);
            m = fmaxf(m, fabsf(v[jj]));
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(grp, m, o));
        // v = x * 2^(2 - e), max |v| over the block in [2, 4); all-zero (or
        // non-finite) blocks keep e = 0
        int e = 0;
        if (m > 0.0f && m <= 3.402823466e38f) frexpf(m, &e);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) v[jj] = mul_pow2(v[jj], 2 - e);
        uint8_t *bimg = img + size_t(b >> 3) * kT4ImgBytes;
        const int kbyte = 32 * (b & 7) + 8 * c + 4 * h;  // byte of K position 64(b%8)+16c+8h
        float grp_sum[3] = {0.0f, 0.0f, 0.0f};  // this item's share of H, M, L
#pragma unroll
        for (int p = 0; p < kT4Pieces; ++p) {
            const float up = __int_as_float((127 + 2 * p) << 23);
            const float down = __int_as_float((127 - 2 * p) << 23);
            uint32_t word = 0;
            int acc2 = 0;  // sum of 2 * piece (exact small integers)
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
                const __nv_fp4x2_storage_t pc = __nv_cvt_float2_to_fp4x2(
                    make_float2(v[2 * q2] * up, v[2 * q2 + 1] * up), __NV_E2M1, cudaRoundNearest);
                const float2 pv =
                    __half22float2(__half2(__nv_cvt_fp4x2_to_halfraw2(pc, __NV_E2M1)));
                v[2 * q2] -= pv.x * down;
                v[2 * q2 + 1] -= pv.y * down;
                acc2 += __float2int_rn(2.0f * pv.x) + __float2int_rn(2.0f * pv.y);
                word |= uint32_t(pc) << (8 * q2);
            }
            *reinterpret_cast<uint32_t *>(bimg + t5_img_offset(p, kbyte)) = word;
            // sum of piece / 2 = acc2 / 4, weighted by 4^-p, into its group
            const int gi = p < 6 ? 0 : p < 12 ? 1 : 2;
            grp_sum[gi] = fmaf(float(acc2) * 0.25f, down, grp_sum[gi]);
        }
#pragma unroll
        for (int gi = 0; gi < 3; ++gi)
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) grp_sum[gi] += __shfl_xor_sync(grp, grp_sum[gi], o);
        if ((idx & 7) == 0)
            *reinterpret_cast<float4 *>(brec + size_t(b) * kT4BlockRec) =
                make_float4(pow2f(e - 1), grp_sum[0], grp_sum[1], grp_sum[2]);
    }
}

// Where the epilogue writes the tile a ring stage belongs to; the producer fills
// one per slot before the slot's barrier arrive.
struct T4StageMeta {
    float *y;              // nullptr: the tile is not written (an expert id out of range)
    int row0;              // first row of the tile
    int n_rows;            // rows of the matrix
    int flags;             // kT4FirstOfTile | kT4LastOfTile
    int pad;
};
constexpr int kT4FirstOfTile = 1;
constexpr int kT4LastOfTile = 2;

// Warp roles of the fp4 kernel. A warp reaches only the TMEM lanes of its
// quarter (warp % 4, which is also its SM sub-partition):
//   warp 2       producer;
//   warps 3, 1   MMA issuers of the even / odd stages (warp 3 allocates TMEM);
//   warps 4-7    expansion, one per lane quarter, all 8 blocks of a stage;
//   warps 8-11   epilogue, one per lane quarter, all 8 blocks of a stage.
// Measured: more warps per sub-partition (two expansion or two epilogue warps
// per quarter) lengthened the stage period; 12 warps gave the shortest.
constexpr int kT4SplitCodeBytes = kT5Rows * 128;  // 16 KB of codes, then 2 KB of scales
static_assert(kT4SplitCodeBytes + kT5Rows * 16 == kT5RawBytes, "split stage = block stage bytes");
constexpr int kT4ProdWarp = 2;
constexpr int kT4MmaWarp = 3;
constexpr int kT4MmaWarp2 = 1;
constexpr int kT4ExpWarp0 = 4;
constexpr int kT4ExpWarps = 4;
constexpr int kT4EpiWarp0 = 8;
constexpr int kT4EpiWarps = 4;
constexpr int kT4Threads = 12 * 32;

// kSplit: the weights are in the split layout (codes [N][K/64][16], scales
// [N][K/64]); the stage's code box is 128 bytes x 128 rows with 128-byte swizzle
// and its scale box 16 bytes x 128 rows, together the same 18 KB as the block
// box of the 18-byte layout.
// At most 128 registers a thread (384 x 128 = 48K of the SM's 64K), so a CTA of
// the next prep kernel (256 threads x 64 registers) can be resident beside it
// and the programmatic launch overlaps the two.
template <bool kSplit>
__global__ void __maxnreg__(128)
    mv_t4_kernel(const __grid_constant__ MvJob single, const MvParams p) {
    // The next prep launch on the stream may become resident now; it waits for
    // this grid before it touches any buffer this kernel reads.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *img_ring = smem;                                      // kT5Stages x 4 KB
    uint8_t *raw_ring = img_ring + kT5Stages * kT4ImgBytes;         // kT5Stages x 18 KB
    uint8_t *beta_ring = raw_ring + kT5Stages * kT5RawBytes;        // kT5Stages x 32 B
    uint64_t *full = reinterpret_cast<uint64_t *>(beta_ring + kT5Stages * kT4BetaBytes);
    uint64_t *empty = full + kT5Stages;
    uint64_t *a_full = empty + kT5Stages;
    uint64_t *a_empty = a_full + kT5MaxABufs;
    uint64_t *d_full = a_empty + kT5MaxABufs;
    uint64_t *d_empty = d_full + 2;
    uint64_t *drain = d_empty + 2;  // [2] one per MMA issuer: its final commit
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    // per ring slot, written by the producer before the slot's barrier arrive:
    // where the epilogue writes the tile that the stage belongs to
    __shared__ T4StageMeta s_meta[kT5Stages];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kT5Stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kT4EpiWarps);
        }
        for (int i = 0; i < kT4ABufs; ++i) {
            mbar_init(&a_full[i], kT4ExpWarps);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], kT4EpiWarps);
        }
        for (int i = 0; i < 2; ++i) mbar_init(&drain[i], 1);
        s_abort = 0;
        fence_barrier_init();
    }
    if (warp == kT4MmaWarp) {
        tmem_alloc(&s_tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    int n_items, item_base = 0;
    if (p.jobs) {
        item_base = p.cta_begin[blockIdx.x];
        n_items = p.cta_begin[blockIdx.x + 1] - item_base;
    } else {
        // one matrix: its tiles; expert mat-vec: (output vector, tile) pairs
        const int total = p.moe.ids ? p.moe.n_vec * single.n_tiles : single.n_tiles;
        n_items = blockIdx.x < unsigned(total) ? (total - 1 - int(blockIdx.x)) / int(gridDim.x) + 1
                                               : 0;
    }
    auto item_at = [&](int i, const MvJob *&J, int &tile) {
        if (p.jobs) {
            const MvItem it = p.items[item_base + i];
            J = &p.jobs[it.job];
            tile = it.tile;
        } else {
            J = &single;
            tile = int(blockIdx.x) + i * int(gridDim.x);
        }
    };
    // stages of this CTA (every role but the producer runs a flat stage loop)
    const int n_stages = p.jobs ? p.cta_stages[blockIdx.x] : n_items * single.n_chunks;
    auto stage_parity = [](int s) { return uint32_t(s / kT5Stages) & 1u; };
    auto a_buf = [](int s) { return s % kT4ABufs; };
    auto a_use = [](int s) { return uint32_t(s / kT4ABufs) & 1u; };
    auto a_col = [](int s) { return uint32_t(kT4ACol + (s % kT4ABufs) * 64); };
    auto d_col = [](int s) { return uint32_t((s & 1) * 128); };

    if (warp == kT4ProdWarp) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            int s = 0, last = -1;
            bool ok = true, prep_ready = false;
            for (int i = 0; i < n_items && ok; ++i) {
                const MvJob *J;
                int tile;
                item_at(i, J, tile);
                const uint8_t *prep = J->prep;
                float *y_out = J->y;
                int row_base = 0;  // first tensor-map row of the matrix
                if (p.moe.ids) {
                    // item = (output vector v, tile): expert ids[v], that expert's
                    // rows of the stacked tensor map, the vector's prep and y
                    const int v = tile / J->n_tiles;
                    tile -= v * J->n_tiles;
                    int e = p.moe.ids[v];
                    if (e < 0 || e >= p.moe.n_expert) {
                        if (tile == 0) record_error(p.err, Q2_0_DEVERR_BAD_ID, v);
                        e = 0;            // stream a valid matrix, write nothing
                        y_out = nullptr;
                    } else {
                        y_out += size_t(v) * J->N;
                    }
                    row_base = e * J->N;
                    const int xv = p.moe.n_x == 1 ? v / p.moe.n_used : v;
                    prep += size_t(xv) * p.moe.prep_stride;
                }
                const uint8_t *img = prep + kT5PrepHeader;
                const uint8_t *beta = img + size_t(J->n_chunks) * kT4ImgBytes;
                const int nch = J->n_chunks;
                for (int ch = 0; ch < nch; ++ch, ++s) {
                    const int st = s % kT5Stages;
                    if (!mbar_wait(&empty[st], stage_parity(s) ^ 1u, p.err, kTagT5Empty, true) ||
                        *(volatile int *)&s_abort) {
                        ok = false;
                        s_abort = 1;
                        break;
                    }
                    T4StageMeta &m = s_meta[st];
                    m.y = y_out;
                    m.row0 = tile * kT5Rows;
                    m.n_rows = J->N;
                    m.flags = (ch == 0 ? kT4FirstOfTile : 0) | (ch == nch - 1 ? kT4LastOfTile : 0);
                    mbar_arrive_expect_tx(&full[st], kT5RawBytes + kT4ImgBytes + kT4BetaBytes);
                    if (kSplit) {
                        tma_load_2d(raw_ring + st * kT5RawBytes, &J->tmap, ch * 128,
                                    row_base + tile * kT5Rows, &full[st]);
                        tma_load_2d(raw_ring + st * kT5RawBytes + kT4SplitCodeBytes, &J->tmap_d,
                                    ch * 16, row_base + tile * kT5Rows, &full[st]);
                    } else {
                        tma_load_2d(raw_ring + st * kT5RawBytes, &J->tmap, ch * kChunkBytes,
                                    row_base + tile * kT5Rows, &full[st]);
                    }
                    if (!prep_ready) {
                        grid_dependency_wait();  // the B images come from the prep kernel
                        prep_ready = true;
                    }
                    bulk_g2s(img_ring + st * kT4ImgBytes, img + size_t(ch) * kT4ImgBytes,
                             kT4ImgBytes, &full[st]);
                    bulk_g2s(beta_ring + st * kT4BetaBytes, beta + size_t(ch) * kT4BetaBytes,
                             kT4BetaBytes, &full[st]);
                    last = s;
                }
            }
            if (!ok) {
                // let the copies in flight land (bounded) before the CTA exits
                for (int t = last; t >= 0 && t > last - kT5Stages; --t)
                    mbar_wait(&full[t % kT5Stages], stage_parity(t), p.err, kTagT5Full);
            }
        }
    } else if (warp == kT4MmaWarp || warp == kT4MmaWarp2) {
        // ------------------------------ MMA issuers ------------------------------
        // even / odd stages; the whole warp runs the loop and waits (so it stays
        // converged), the elected lane issues (one K = 64 MMA per block) and commits
        constexpr uint32_t idesc = idesc_mxf4(kT5Rows, kT5N);
        const bool leader = elect_one();
        const int mine = warp == kT4MmaWarp ? 0 : 1;
        const uint64_t desc0 = sw128_desc(smem_addr(img_ring));
        const uint32_t sfa = tmem + kT4ScaleCol, sfb = tmem + kT4ScaleCol + 4;
        int last = -1;
        {
            for (int s = mine; s < n_stages; s += 2) {
                const int st = s % kT5Stages;
                const bool got =
                    mbar_wait(&full[st], stage_parity(s), p.err, kTagT5Full) &&
                    mbar_wait(&a_full[a_buf(s)], a_use(s), p.err, kTagT5AFull) &&
                    mbar_wait(&d_empty[s & 1], (uint32_t(s >> 1) & 1u) ^ 1u, p.err,
                              kTagT5DEmpty) &&
                    !*(volatile int *)&s_abort;
                if (!__all_sync(0xffffffffu, got)) {
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a_base = tmem + a_col(s);
                const uint32_t d_base = tmem + d_col(s);
                const uint64_t dst = desc0 + uint64_t((st * kT4ImgBytes) >> 4);
                if (leader) {
#pragma unroll
                    for (int b = 0; b < kChunkBlocks; ++b)
                        tc_mma_mxf4_ta(d_base + b * kT5N, a_base + b * 8,
                                       dst + uint64_t(((b >> 2) * 2048 + (b & 3) * 32) >> 4), idesc,
                                       sfa, sfb, 0u);
                    tc_commit(&a_empty[a_buf(s)]);
                    tc_commit(&d_full[s & 1]);
                }
                __syncwarp();
                last = s;
            }
        }
        // TMEM is freed only after this issuer's MMAs completed: one more commit
        // tracks all of them
        if (last >= 0) {
            if (leader) tc_commit(&drain[mine]);
            __syncwarp();
            if (leader) mbar_wait(&drain[mine], 0u, p.err, kTagT5DFull);
            __syncwarp();
        }
    } else if (warp >= kT4ExpWarp0 && warp < kT4ExpWarp0 + kT4ExpWarps) {
        // ------------------------------ expansion ------------------------------
        // warp w: TMEM lane quarter w % 4 (rows 32 (w % 4) ..), all 8 blocks
        const int qd = warp & 3;
        const int row = 32 * qd + lane;
        const uint32_t lane_base = uint32_t(32 * qd) << 16;
        {  // scale factors 1.0 (ue8m0 127) for this quarter's lanes
            const uint32_t one = 0x7F7F7F7Fu;
            tmem_st4(tmem + lane_base + kT4ScaleCol, one, one, one, one);
            tmem_st4(tmem + lane_base + kT4ScaleCol + 4, one, one, one, one);
        }
        {
            for (int s = 0; s < n_stages; ++s) {
                const int st = s % kT5Stages;
                const bool got =
                    mbar_wait(&full[st], stage_parity(s), p.err, kTagT5Full) &&
                    mbar_wait(&a_empty[a_buf(s)], a_use(s) ^ 1u, p.err, kTagT5AFull) &&
                    !*(volatile int *)&s_abort;
                if (!__all_sync(0xffffffffu, got)) {
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int G = 0; G < 2; ++G) {
                    uint32_t a[32];
                    if (kSplit) {
                        // block 4G+bi is 16-byte chunk 4G+bi of the row, stored at
                        // chunk (4G+bi) ^ (row % 8) by the 128-byte swizzle
                        const uint8_t *rp = raw_ring + st * kT5RawBytes + row * 128;
#pragma unroll
                        for (int bi = 0; bi < 4; ++bi) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(
                                rp + (((4 * G + bi) ^ (row & 7)) << 4));
                            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                a[8 * bi + 2 * c + 0] = wv[c] & 0x33333333u;
                                a[8 * bi + 2 * c + 1] = (wv[c] >> 2) & 0x33333333u;
                            }
                        }
                    } else {
                        const uint8_t *rp =
                            raw_ring + st * kT5RawBytes + row * kChunkBytes + G * 72;
                        uint32_t u[18];
#pragma unroll
                        for (int k = 0; k < 9; ++k) {
                            const uint2 v = *reinterpret_cast<const uint2 *>(rp + 8 * k);
                            u[2 * k] = v.x;
                            u[2 * k + 1] = v.y;
                        }
#pragma unroll
                        for (int bi = 0; bi < 4; ++bi) {
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                uint32_t w;
                                if (bi == 0) w = __byte_perm(u[c], u[c + 1], 0x5432);
                                else if (bi == 1) w = u[5 + c];
                                else if (bi == 2) w = __byte_perm(u[9 + c], u[10 + c], 0x5432);
                                else w = u[14 + c];
                                a[8 * bi + 2 * c + 0] = w & 0x33333333u;
                                a[8 * bi + 2 * c + 1] = (w >> 2) & 0x33333333u;
                            }
                        }
                    }
                    tmem_st32(tmem + lane_base + a_col(s) + 32 * G, a);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[a_buf(s)]);
            }
        }
    } else if (warp >= kT4EpiWarp0 && warp < kT4EpiWarp0 + kT4EpiWarps) {
        // ------------------------------ epilogue ------------------------------
        // warp w: TMEM lane quarter w % 4, all 8 blocks of each stage; it writes y
        // at the tile's last stage. Every wait is bounded; a warp whose wait
        // fails leaves the loop.
        const int qd = warp & 3;
        const int row = 32 * qd + lane;
        const uint32_t lane_base = uint32_t(32 * qd) << 16;
        float acc = 0.0f, comp = 0.0f;  // compensated sum of the stage sums
        for (int s = 0; s < n_stages; ++s) {
            const int st = s % kT5Stages;
            const bool got = !*(volatile int *)&s_abort &&
                             mbar_wait(&full[st], stage_parity(s), p.err, kTagT5Full) &&
                             mbar_wait(&d_full[s & 1], uint32_t(s >> 1) & 1u, p.err, kTagT5DFull);
            if (!__all_sync(0xffffffffu, got)) {
                s_abort = 1;
                break;
            }
            tc_fence_after();
            const T4StageMeta m = s_meta[st];
            const uint32_t d_base = tmem + lane_base + d_col(s);
            const uint8_t *rp = raw_ring + st * kT5RawBytes + row * kChunkBytes;
            const float4 *brec = reinterpret_cast<const float4 *>(beta_ring + st * kT4BetaBytes);
            float stage_sum = 0.0f;
            // blocks 4 hb .. 4 hb + 3: their 16 pieces each (64 registers)
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                uint32_t r[4][16];
#pragma unroll
                for (int bi = 0; bi < 4; ++bi) tmem_ld16(d_base + (4 * hb + bi) * kT5N, r[bi]);
                tmem_wait_ld();
                if (hb == 1) {  // the stage's accumulators are all in registers
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&d_empty[s & 1]);
                }
#pragma unroll
                for (int bi = 0; bi < 4; ++bi) {
                    const int b = 4 * hb + bi;
                    auto C = [&](int pp) { return __uint_as_float(r[bi][pp]); };
                    // the three exact groups of sum_p 4^-p C_p
                    float gh = C(5) * 0x1p-10f, gm = C(11) * 0x1p-22f, gl = C(15) * 0x1p-30f;
#pragma unroll
                    for (int pp = 4; pp >= 0; --pp) gh = fmaf(C(pp), __int_as_float((127 - 2 * pp) << 23), gh);
#pragma unroll
                    for (int pp = 10; pp >= 6; --pp) gm = fmaf(C(pp), __int_as_float((127 - 2 * pp) << 23), gm);
#pragma unroll
                    for (int pp = 14; pp >= 12; --pp) gl = fmaf(C(pp), __int_as_float((127 - 2 * pp) << 23), gl);
                    const float4 br = brec[b];  // {2^(e - 1), H, M, L}
                    const float t = ((gh - br.y) + (gm - br.z)) + (gl - br.w);
                    const float d =
                        kSplit ? lds_half_as_float(raw_ring + st * kT5RawBytes + kT4SplitCodeBytes +
                                                   row * 16 + 2 * b)
                               : lds_half_as_float(rp + 18 * b);
                    stage_sum = fmaf(d, t * br.x, stage_sum);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            // acc + comp += stage_sum (two-sum: the rounding error is kept)
            {
                const float sum = acc + stage_sum;
                const float bb = sum - acc;
                comp += (acc - (sum - bb)) + (stage_sum - bb);
                acc = sum;
            }
            if (m.flags & kT4LastOfTile) {
                const int rr = m.row0 + row;
                if (m.y && rr < m.n_rows) m.y[rr] = acc + comp;
                acc = 0.0f;
                comp = 0.0f;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kT4MmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// Generic mat-vec (any K % 64 == 0, any alignment): one warp per row, f32 on
// CUDA cores, block-wise: s = sum (q - 1) * x over the block, then acc += d*s.
// ---------------------------------------------------------------------------
template <typename XT>
__global__ void __launch_bounds__(256) mv_generic_kernel(const uint8_t *__restrict__ w,
                                                         const XT *__restrict__ x,
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
        const uint8_t *blk = w + (size_t(row) * nb + b) * 18;
        const float d = half_bits_to_float(uint32_t(blk[0]) | (uint32_t(blk[1]) << 8));
        float s[8];
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) s[cc] = 0.0f;
        for (int wi = 0; wi < 4; ++wi) {
            const uint8_t *pw = blk + 2 + 4 * wi;
            const uint32_t word = uint32_t(pw[0]) | (uint32_t(pw[1]) << 8) |
                                  (uint32_t(pw[2]) << 16) | (uint32_t(pw[3]) << 24);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float q1 = float(int((word >> (2 * i)) & 3u) - 1);
                const int k = b * 64 + wi * 16 + i;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                    if (cc < ncols) s[cc] = fmaf(q1, ld_x(x + size_t(cc) * K + k), s[cc]);
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

// Generic expert mat-vec (any K % 64 == 0, any alignment): grid (rows / 8,
// output vectors); one warp per row of the vector's expert, as above.
__global__ void __launch_bounds__(256) moe_generic_kernel(
    const uint8_t *__restrict__ w, const float *__restrict__ x, const int32_t *__restrict__ ids,
    float *__restrict__ y, int N, int K, int n_expert, int n_used, int n_x,
    unsigned long long *err) {
    const int v = blockIdx.y;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int e = ids[v];
    if (e < 0 || e >= n_expert) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_error(err, Q2_0_DEVERR_BAD_ID, v);
        return;
    }
    if (row >= N) return;
    const int nb = K / 64;
    const float *xv = x + size_t(n_x == 1 ? v / n_used : v) * K;
    const uint8_t *wr = w + (size_t(e) * N + row) * nb * 18;
    float acc = 0.0f;
    for (int b = lane; b < nb; b += 32) {
        const uint8_t *blk = wr + size_t(b) * 18;
        const float d = half_bits_to_float(uint32_t(blk[0]) | (uint32_t(blk[1]) << 8));
        float sum = 0.0f;
        for (int wi = 0; wi < 4; ++wi) {
            const uint8_t *pw = blk + 2 + 4 * wi;
            const uint32_t word = uint32_t(pw[0]) | (uint32_t(pw[1]) << 8) |
                                  (uint32_t(pw[2]) << 16) | (uint32_t(pw[3]) << 24);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                sum = fmaf(float(int((word >> (2 * i)) & 3u) - 1), xv[b * 64 + wi * 16 + i], sum);
        }
        acc = fmaf(d, sum, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) y[size_t(v) * N + row] = acc;
}

std::mutex g_attr_mu;
bool g_attr_done[64][2];
bool g_t5_attr_done[64][kT5MaxCols];

template <int NC>
cudaError_t set_t5_attr() {
    return cudaFuncSetAttribute(mv_t5_kernel<NC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kT5Smem);
}

bool g_t4_attr_done[64];

cudaError_t ensure_t4_attr() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (dev < 64 && g_t4_attr_done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(mv_t4_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kT4Smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mv_t4_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kT4Smem);
    if (e == cudaSuccess && dev < 64) g_t4_attr_done[dev] = true;
    return e;
}

cudaError_t ensure_t5_attrs(int ncols) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (dev < 64 && g_t5_attr_done[dev][ncols - 1]) return cudaSuccess;
    e = ncols == 1 ? set_t5_attr<1>() : ncols == 2 ? set_t5_attr<2>() : set_t5_attr<3>();
    if (e == cudaSuccess && dev < 64) g_t5_attr_done[dev][ncols - 1] = true;
    return e;
}

cudaError_t ensure_attrs(int nt) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (dev < 64 && g_attr_done[dev][nt - 1]) return cudaSuccess;
    if (nt == 1)
        e = cudaFuncSetAttribute(mv_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBudget + 2 * kMaxStages * 8);
    else
        e = cudaFuncSetAttribute(mv_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBudget + 2 * kMaxStages * 8);
    if (e == cudaSuccess && dev < 64) g_attr_done[dev][nt - 1] = true;
    return e;
}

// ncols = 1 runs the fp4 tcgen05 kernel, ncols 2-3 the e4m3 one (both 128-row
// tiles); more columns run the mma.sync kernel (256-row tiles).
bool use_t4(int ncols) { return ncols == 1; }
bool use_t5(int ncols) { return ncols <= kT5MaxCols; }
int tile_rows_for(int ncols) { return use_t5(ncols) ? kT5Rows : kTileRows; }

bool make_job(MvJob &J, const uint8_t *w, const uint8_t *prep, float *y, int64_t N, int64_t K,
              int rows) {
    std::memset(&J, 0, sizeof(J));
    const uint64_t row_bytes = uint64_t(K / 64) * 18;
    if (!encode_tmap_2d(&J.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, row_bytes, uint64_t(N), row_bytes,
                        kChunkBytes, rows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return false;
    J.prep = prep;
    J.y = y;
    J.N = int(N);
    J.nb = int(K / 64);
    J.n_chunks = int(K / 512);
    J.n_tiles = int((N + rows - 1) / rows);
    return true;
}

// max_k: the largest K among the jobs (sets the t5 prep's grid z).
template <typename XT>
// The prep kernels are launched as programmatic dependents of whatever precedes
// them on the stream: their launch overlaps that kernel's tail, and they wait
// for it (griddepcontrol.wait) before reading x or writing their buffers.
cudaError_t launch_prep_t(const MvPrepJob &single, const MvPrepJob *jobs, int n_jobs, int ncols,
                          int64_t max_k, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(ncols, n_jobs);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (use_t4(ncols)) {
        const int64_t items = max_k / 64 * 8;
        cfg.gridDim.z =
            unsigned(std::min<int64_t>((items + kT5PrepThreads - 1) / kT5PrepThreads, 65535));
        cfg.blockDim = dim3(kT5PrepThreads);
        return cudaLaunchKernelEx(&cfg, t4_prep_kernel<XT>, single, jobs);
    }
    if (use_t5(ncols)) {
        const int64_t items = max_k / 64 * 16;
        cfg.gridDim.z =
            unsigned(std::min<int64_t>((items + kT5PrepThreads - 1) / kT5PrepThreads, 65535));
        cfg.blockDim = dim3(kT5PrepThreads);
        return cudaLaunchKernelEx(&cfg, t5_prep_kernel<XT>, single, jobs, ncols);
    }
    cfg.blockDim = dim3(kPrepThreads);
    if (n_tiles_for(ncols) == 1) return cudaLaunchKernelEx(&cfg, mv_prep_kernel<1, XT>, single, jobs, ncols);
    return cudaLaunchKernelEx(&cfg, mv_prep_kernel<2, XT>, single, jobs, ncols);
}

cudaError_t launch_prep(const MvPrepJob &single, const MvPrepJob *jobs, int n_jobs, int ncols,
                        int64_t max_k, int xtype, cudaStream_t s) {
    return xtype == kXF16 ? launch_prep_t<__half>(single, jobs, n_jobs, ncols, max_k, s)
                          : launch_prep_t<float>(single, jobs, n_jobs, ncols, max_k, s);
}

// The tensor-core kernel is launched as a programmatic dependent of the prep
// kernel: its prologue and first weight loads overlap the prep's tail; its
// producer waits for the prep grid before loading any activation fragment.
cudaError_t launch_tc(const MvJob &single, const MvParams &prm, int grid, cudaStream_t s) {
    const int nt = n_tiles_for(prm.ncols);
    cudaError_t e = use_t4(prm.ncols)   ? ensure_t4_attr()
                    : use_t5(prm.ncols) ? ensure_t5_attrs(prm.ncols)
                                        : ensure_attrs(nt);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (use_t4(prm.ncols)) {
        cfg.blockDim = dim3(kT4Threads);
        cfg.dynamicSmemBytes = kT4Smem;
        e = prm.split ? cudaLaunchKernelEx(&cfg, mv_t4_kernel<true>, single, prm)
                      : cudaLaunchKernelEx(&cfg, mv_t4_kernel<false>, single, prm);
    } else if (use_t5(prm.ncols)) {
        cfg.blockDim = dim3(kT5Threads);
        cfg.dynamicSmemBytes = kT5Smem;
        if (prm.ncols == 1)
            e = cudaLaunchKernelEx(&cfg, mv_t5_kernel<1>, single, prm);
        else if (prm.ncols == 2)
            e = cudaLaunchKernelEx(&cfg, mv_t5_kernel<2>, single, prm);
        else
            e = cudaLaunchKernelEx(&cfg, mv_t5_kernel<3>, single, prm);
    } else if (nt == 1) {
        cfg.blockDim = dim3(kCtaThreads);
        cfg.dynamicSmemBytes = smem_bytes_for(prm.ncols);
        e = cudaLaunchKernelEx(&cfg, mv_tc_kernel<1>, single, prm);
    } else {
        cfg.blockDim = dim3(kCtaThreads);
        cfg.dynamicSmemBytes = smem_bytes_for(prm.ncols);
        e = cudaLaunchKernelEx(&cfg, mv_tc_kernel<2>, single, prm);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_generic(const uint8_t *w, const void *x, int xtype, float *y, int64_t N,
                           int64_t K, int ncols, cudaStream_t s) {
    const unsigned grid = unsigned((N + 7) / 8);
    if (xtype == kXF16)
        mv_generic_kernel<__half><<<grid, 256, 0, s>>>(w, static_cast<const __half *>(x), y,
                                                       int(N), int(K), ncols);
    else
        mv_generic_kernel<float><<<grid, 256, 0, s>>>(w, static_cast<const float *>(x), y,
                                                      int(N), int(K), ncols);
    return cudaGetLastError();
}

}  // namespace

size_t matvec_workspace_bytes(int64_t K, int ncols) {
    return use_t4(ncols) ? t4_prep_bytes(K) : use_t5(ncols) ? t5_prep_bytes(K)
                                                            : prep_bytes_for(K, ncols);
}

bool matvec_fast_path_ok(const void *w, int64_t K) {
    return K % 512 == 0 && (reinterpret_cast<uintptr_t>(w) & 15u) == 0;
}

int matvec_run(const uint8_t *w, const void *x, int xtype, float *y, int64_t N, int64_t K,
               int ncols, void *ws, size_t ws_bytes, cudaStream_t s) {
    if (!matvec_fast_path_ok(w, K))
        return cuda_status(launch_generic(w, x, xtype, y, N, K, ncols, s));
    if (ws_bytes < matvec_workspace_bytes(K, ncols)) return Q2_0_EINVAL;
    unsigned long long *err = error_word_ptr();
    if (!err) return Q2_0_ECUDA;
    uint8_t *prep = static_cast<uint8_t *>(ws);
    MvPrepJob pj{x, prep, int(K)};
    cudaError_t e = launch_prep(pj, nullptr, 1, ncols, K, xtype, s);
    if (e != cudaSuccess) return Q2_0_ECUDA;
    MvJob J;
    if (!make_job(J, w, prep, y, N, K, tile_rows_for(ncols))) return Q2_0_ECUDA;
    MvParams prm{nullptr, nullptr, nullptr, nullptr, ncols, n_stages_for(ncols), err};
    const int grid = std::max(1, std::min(J.n_tiles, sm_count()));
    return cuda_status(launch_tc(J, prm, grid, s));
}

int matvec_split_run(const uint8_t *soa, const float *x, float *y, int64_t N, int64_t K,
                     int ncols, void *ws, size_t ws_bytes, cudaStream_t s) {
    const uint8_t *dsc = soa + soa_qs_bytes(N, K);
    if (ncols != 1 || !matvec_fast_path_ok(soa, K))
        return cuda_status(launch_soa_generic(soa, x, y, N, K, ncols, s));
    if (ws_bytes < t4_prep_bytes(K)) return Q2_0_EINVAL;
    unsigned long long *err = error_word_ptr();
    if (!err) return Q2_0_ECUDA;
    uint8_t *prep = static_cast<uint8_t *>(ws);
    MvPrepJob pj{x, prep, int(K)};
    if (launch_prep(pj, nullptr, 1, 1, K, kXF32, s) != cudaSuccess) return Q2_0_ECUDA;
    MvJob J;
    std::memset(&J, 0, sizeof(J));
    const uint64_t nb = uint64_t(K / 64);
    // codes: 128 bytes (8 blocks) x 128 rows per box, 128-byte swizzle;
    // scales: 16 bytes x 128 rows per box
    if (!encode_tmap_2d(&J.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, soa, nb * 16, uint64_t(N), nb * 16,
                        128, kT5Rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&J.tmap_d, CU_TENSOR_MAP_DATA_TYPE_UINT8, dsc, nb * 2, uint64_t(N), nb * 2,
                        16, kT5Rows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return Q2_0_ECUDA;
    J.prep = prep;
    J.y = y;
    J.N = int(N);
    J.nb = int(nb);
    J.n_chunks = int(K / 512);
    J.n_tiles = int((N + kT5Rows - 1) / kT5Rows);
    MvParams prm{nullptr, nullptr, nullptr, nullptr, 1, n_stages_for(1), err, MvMoe{}, 1};
    const int grid = std::max(1, std::min(J.n_tiles, sm_count()));
    return cuda_status(launch_tc(J, prm, grid, s));
}

size_t matvec_moe_workspace_bytes(int64_t K, int64_t n_xvec) {
    return K % 512 == 0 ? size_t(n_xvec) * t4_prep_bytes(K) : 0;
}

int matvec_moe_run(const uint8_t *w, int64_t n_expert, int64_t N, int64_t K, const float *x,
                   int64_t n_x, const int32_t *ids, int64_t n_used, int64_t n_tokens, float *y,
                   void *ws, size_t ws_bytes, cudaStream_t s) {
    unsigned long long *err = error_word_ptr();
    if (!err) return Q2_0_ECUDA;
    const int64_t n_vec = n_tokens * n_used;
    if (!matvec_fast_path_ok(w, K)) {
        dim3 grid(unsigned((N + 7) / 8), unsigned(n_vec));
        moe_generic_kernel<<<grid, 256, 0, s>>>(w, x, ids, y, int(N), int(K), int(n_expert),
                                                int(n_used), int(n_x), err);
        return cuda_status(cudaGetLastError());
    }
    const int64_t n_xvec = n_tokens * n_x;
    if (ws_bytes < matvec_moe_workspace_bytes(K, n_xvec)) return Q2_0_EINVAL;
    uint8_t *prep = static_cast<uint8_t *>(ws);
    const long long stride = (long long)t4_prep_bytes(K);
    // one fp4 prep region per activation vector
    MvPrepJob pj{x, prep, int(K), (long long)K * 4, stride};
    if (launch_prep(pj, nullptr, int(n_xvec), 1, K, kXF32, s) != cudaSuccess) return Q2_0_ECUDA;
    // the tensor map spans all experts' rows; the kernel picks expert ids[v]
    MvJob J;
    if (!make_job(J, w, prep, y, n_expert * N, K, kT5Rows)) return Q2_0_ECUDA;
    J.N = int(N);
    J.n_tiles = int((N + kT5Rows - 1) / kT5Rows);
    MvParams prm{nullptr, nullptr, nullptr, nullptr, 1, n_stages_for(1), err,
                 MvMoe{ids, int(n_vec), int(n_used), int(n_x), int(n_expert), stride}};
    const int64_t items = n_vec * J.n_tiles;
    const int grid = int(std::max<int64_t>(1, std::min<int64_t>(items, sm_count())));
    return cuda_status(launch_tc(J, prm, grid, s));
}

}  // namespace q2

// ---------------------------------------------------------------------------
// Batched plans
// ---------------------------------------------------------------------------
struct q2_0_mv_plan {
    int device = 0;
    int ncols = 1;
    int n_fast = 0;
    int grid = 0;
    int64_t max_k = 0;  // largest K among the TMA-path jobs
    q2::MvJob *d_jobs = nullptr;
    q2::MvItem *d_items = nullptr;
    int *d_cta_begin = nullptr;
    int *d_cta_stages = nullptr;  // [grid] stages (512-column chunks) per CTA
    q2::MvPrepJob *d_prep_jobs = nullptr;
    uint8_t *d_prep = nullptr;
    unsigned long long *err = nullptr;
    std::vector<q2_0_mv_desc> generic;  // descriptors outside the TMA path
};

namespace q2 {

void mv_plan_destroy(q2_0_mv_plan *plan) {
    if (!plan) return;
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(plan->device);
    cudaFree(plan->d_jobs);
    cudaFree(plan->d_items);
    cudaFree(plan->d_cta_begin);
    cudaFree(plan->d_cta_stages);
    cudaFree(plan->d_prep_jobs);
    cudaFree(plan->d_prep);
    cudaSetDevice(cur);
    delete plan;
}

int mv_plan_create(const q2_0_mv_desc *descs, int n, int ncols, q2_0_mv_plan **out) {
    q2_0_mv_plan *P = new q2_0_mv_plan();
    cudaGetDevice(&P->device);
    P->ncols = ncols;
    P->err = error_word_ptr();
    if (!P->err) {
        delete P;
        return Q2_0_ECUDA;
    }
    std::vector<int> fast;
    for (int i = 0; i < n; ++i) {
        if (matvec_fast_path_ok(descs[i].w, descs[i].K))
            fast.push_back(i);
        else
            P->generic.push_back(descs[i]);
    }
    P->n_fast = int(fast.size());
    int st = Q2_0_OK;
    if (P->n_fast > 0) {
        // prep buffers, one per fast job
        std::vector<size_t> off(P->n_fast);
        size_t total = 0;
        for (int j = 0; j < P->n_fast; ++j) {
            off[j] = total;
            total += matvec_workspace_bytes(descs[fast[j]].K, ncols);
        }
        std::vector<MvJob> jobs(P->n_fast);
        std::vector<MvPrepJob> pjobs(P->n_fast);
        if (cudaMalloc(&P->d_prep, total) != cudaSuccess) st = Q2_0_ECUDA;
        for (int j = 0; j < P->n_fast && st == Q2_0_OK; ++j) {
            const q2_0_mv_desc &d = descs[fast[j]];
            if (!make_job(jobs[j], static_cast<const uint8_t *>(d.w), P->d_prep + off[j], d.y, d.N,
                          d.K, tile_rows_for(ncols)))
                st = Q2_0_ECUDA;
            pjobs[j] = MvPrepJob{d.x, P->d_prep + off[j], int(d.K)};
            P->max_k = std::max<int64_t>(P->max_k, d.K);
        }
        // Schedule of (job, tile) items over one CTA per SM. A tile costs its
        // stage count (K / 512): the pipeline takes the same time per stage
        // whatever the tile's valid rows. Longest-processing-time-first, then
        // moves and swaps between the most and the least loaded CTA while they
        // lower the larger of the two loads; each CTA then takes its items in
        // (job, tile) order, so consecutive items share a tensor map and
        // activation images.
        std::vector<MvItem> items;
        std::vector<int> cost;
        for (int j = 0; j < P->n_fast; ++j)
            for (int t = 0; t < jobs[j].n_tiles; ++t) {
                items.push_back(MvItem{j, t});
                cost.push_back(jobs[j].n_chunks);
            }
        std::vector<int> order(items.size());
        for (size_t k = 0; k < order.size(); ++k) order[k] = int(k);
        std::stable_sort(order.begin(), order.end(),
                         [&](int a, int b) { return cost[a] > cost[b]; });
        const int grid = std::max(1, std::min<int>(sm_count(), int(items.size())));
        using Load = std::pair<int64_t, int>;
        std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
        for (int c = 0; c < grid; ++c) heap.push(Load(0, c));
        std::vector<std::vector<int>> per_cta(grid);  // item indices
        std::vector<int64_t> load(grid, 0);
        for (int k : order) {
            Load l = heap.top();
            heap.pop();
            per_cta[l.second].push_back(k);
            load[l.second] += cost[k];
            heap.push(Load(load[l.second], l.second));
        }
        for (int iter = 0; iter < 4 * int(items.size()) && grid > 1; ++iter) {
            const int hi = int(std::max_element(load.begin(), load.end()) - load.begin());
            const int lo = int(std::min_element(load.begin(), load.end()) - load.begin());
            const int64_t gap = load[hi] - load[lo];
            // moving cost d from hi to lo lowers the larger of the two loads by
            // min(d, gap - d): take the move or swap that lowers it most
            int64_t best = 0, gain = 0;
            int bi = -1, bj = -1;
            for (int a = 0; a < int(per_cta[hi].size()); ++a) {
                const int64_t ca = cost[per_cta[hi][a]];
                if (std::min(ca, gap - ca) > gain) { gain = std::min(ca, gap - ca); best = ca; bi = a; bj = -1; }
                for (int b = 0; b < int(per_cta[lo].size()); ++b) {
                    const int64_t d = ca - cost[per_cta[lo][b]];
                    if (std::min(d, gap - d) > gain) { gain = std::min(d, gap - d); best = d; bi = a; bj = b; }
                }
            }
            if (bi < 0) break;
            const int ka = per_cta[hi][bi];
            per_cta[hi].erase(per_cta[hi].begin() + bi);
            per_cta[lo].push_back(ka);
            if (bj >= 0) {
                const int kb = per_cta[lo][bj];
                per_cta[lo].erase(per_cta[lo].begin() + bj);
                per_cta[hi].push_back(kb);
            }
            load[hi] -= best;
            load[lo] += best;
        }
        std::vector<MvItem> flat;
        std::vector<int> begin(grid + 1, 0), stages(grid, 0);
        for (int c = 0; c < grid; ++c) {
            std::sort(per_cta[c].begin(), per_cta[c].end());  // items are built in (job, tile) order
            begin[c] = int(flat.size());
            for (int k : per_cta[c]) {
                flat.push_back(items[k]);
                stages[c] += jobs[items[k].job].n_chunks;
            }
        }
        begin[grid] = int(flat.size());
        P->grid = grid;
        if (st == Q2_0_OK &&
            (cudaMalloc(&P->d_jobs, sizeof(MvJob) * jobs.size()) != cudaSuccess ||
             cudaMalloc(&P->d_items, sizeof(MvItem) * flat.size()) != cudaSuccess ||
             cudaMalloc(&P->d_cta_begin, sizeof(int) * begin.size()) != cudaSuccess ||
             cudaMalloc(&P->d_cta_stages, sizeof(int) * stages.size()) != cudaSuccess ||
             cudaMalloc(&P->d_prep_jobs, sizeof(MvPrepJob) * pjobs.size()) != cudaSuccess))
            st = Q2_0_ECUDA;
        if (st == Q2_0_OK &&
            (cudaMemcpy(P->d_jobs, jobs.data(), sizeof(MvJob) * jobs.size(),
                        cudaMemcpyHostToDevice) != cudaSuccess ||
             cudaMemcpy(P->d_items, flat.data(), sizeof(MvItem) * flat.size(),
                        cudaMemcpyHostToDevice) != cudaSuccess ||
             cudaMemcpy(P->d_cta_begin, begin.data(), sizeof(int) * begin.size(),
                        cudaMemcpyHostToDevice) != cudaSuccess ||
             cudaMemcpy(P->d_cta_stages, stages.data(), sizeof(int) * stages.size(),
                        cudaMemcpyHostToDevice) != cudaSuccess ||
             cudaMemcpy(P->d_prep_jobs, pjobs.data(), sizeof(MvPrepJob) * pjobs.size(),
                        cudaMemcpyHostToDevice) != cudaSuccess))
            st = Q2_0_ECUDA;
    }
    if (st != Q2_0_OK) {
        mv_plan_destroy(P);
        return st;
    }
    *out = P;
    return Q2_0_OK;
}

int mv_plan_launches(const q2_0_mv_plan *P) {
    return (P->n_fast > 0 ? 2 : 0) + int(P->generic.size());
}

int mv_plan_execute(const q2_0_mv_plan *P, cudaStream_t s) {
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != P->device) return Q2_0_EINVAL;
    if (P->n_fast > 0) {
        MvPrepJob none{nullptr, nullptr, 0};
        if (launch_prep(none, P->d_prep_jobs, P->n_fast, P->ncols, P->max_k, kXF32, s) !=
            cudaSuccess)
            return Q2_0_ECUDA;
        MvJob dummy;
        std::memset(&dummy, 0, sizeof(dummy));
        MvParams prm{P->d_jobs, P->d_items, P->d_cta_begin, P->d_cta_stages, P->ncols,
                     n_stages_for(P->ncols),
                     P->err};
        if (launch_tc(dummy, prm, P->grid, s) != cudaSuccess) return Q2_0_ECUDA;
    }
    for (const q2_0_mv_desc &d : P->generic)
        if (launch_generic(static_cast<const uint8_t *>(d.w), d.x, kXF32, d.y, d.N, d.K, P->ncols,
                           s) !=
            cudaSuccess)
            return Q2_0_ECUDA;
    return Q2_0_OK;
}

}  // namespace q2
