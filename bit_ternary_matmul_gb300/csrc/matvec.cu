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
// word becomes 8 A-operand registers with one LOP3 each (+1 shift). The
// per-field factor 4^m is removed by scaling the activations of field m by
// 4^-m, and the "- 1" of (q - 1) by starting each block's accumulation at
// -sum(activation * 4^m * 2^-24) of that block (the value all-ones codes give).
//
// Activations (F32) enter as fp16 hi + lo pairs: per column j, u = x * 2^s_j
// with 2^s_j chosen so max|u| lies in [2^14, 2^15); for element e of a block,
// v = u * 2^-2(e%4), hi = fp16(v), lo = fp16(v - hi). The B operand of an MMA
// has 8 columns: for ncols <= 4 they are (hi of cols 0..3, lo of cols 0..3);
// for 5..8 two MMAs use (hi of cols 0..7) and (lo of cols 0..7). A separate
// small kernel (mv_prep) writes these fragments, in exactly the register order
// the MMA wants, once per call; the mat-vec kernel then only loads them.
//
// Streaming. Each CTA (8 consumer warps + 1 producer warp) owns row tiles of
// 256 rows. A pipeline stage is one 2-D TMA box of 256 rows x 144 bytes (8
// blocks = 512 weights per row) plus the 8 blocks' activation fragments (1-D
// bulk copy). 144-byte rows make the shared-memory words of the 8 rows of an
// MMA group fall in distinct banks. Block pairs (36 bytes) start 4-byte
// aligned: the odd block's words are aligned, the even block's words straddle
// two aligned words and are rebuilt with one byte-permute.
//
// Requirements of the TMA path: K % 512 == 0 (row stride a multiple of 16 B)
// and W 16-byte aligned. Other shapes run mv_generic_kernel (CUDA cores, f32).
#include <algorithm>
#include <cstring>
#include <mutex>
#include <queue>
#include <vector>

#include "q2_0_device.cuh"
#include "q2_0_internal.h"

namespace q2 {

namespace {

constexpr int kTileRows = 256;
constexpr int kChunkBlocks = 8;
constexpr int kChunkBytes = kChunkBlocks * 18;  // 144
constexpr int kWStageBytes = kTileRows * kChunkBytes;  // 36864
// Record per block per n-tile, for S = lane slots that carry data (8 per column
// for ncols <= 4, 4 per column for 5..8): B-fragment registers 0..3 of the S
// slots (16 B each), registers 4..7 of the slots, then for each lane group c
// the accumulator start (s[2c], s[2c+1], s[2c], s[2c+1]) (64 B). Data lanes
// occupy consecutive slots, so their 16-byte loads are dense.
constexpr int kPrepHeader = 64;  // float out_scale[8] (+ pad)
constexpr int kMaxStages = 8;
// Dynamic shared memory the ring may use: the opt-in maximum less the static
// part and the barriers.
constexpr int kSmemBudget = 232448 - 1024 - 2 * kMaxStages * 8;
constexpr int kPrepThreads = 512;

// Timeout tags (info of Q2_0_DEVERR_TIMEOUT).
constexpr int kTagMvFull = 101;
constexpr int kTagMvEmpty = 102;

struct MvPrepJob {
    const float *x;  // [ncols][K]
    uint8_t *prep;   // prepared fragments
    int K;
};

struct MvJob {  // 64-byte aligned through its CUtensorMap member
    CUtensorMap tmap;  // W as uint8 [N][K/64*18], box {144, 256}
    const uint8_t *prep;
    float *y;
    int N;
    int nb;        // K / 64
    int n_chunks;  // K / 512
    int n_tiles;   // ceil(N / 256)
};

struct MvItem {
    int job;
    int tile;
};

struct MvParams {
    const MvJob *jobs;        // nullptr: the single job passed by value
    const MvItem *items;      // per-CTA work lists (schedule), when jobs != nullptr
    const int *cta_begin;     // [gridDim.x + 1]
    int ncols;
    int n_stages;             // pipeline depth (n_stages_for(ncols))
    unsigned long long *err;
};

__host__ __device__ constexpr int n_tiles_for(int ncols) { return ncols <= 4 ? 1 : 2; }
__host__ __device__ constexpr int used_slots(int ncols) {
    return n_tiles_for(ncols) == 1 ? 8 * ncols : 4 * ncols;
}
__host__ __device__ constexpr int rec_bytes(int ncols) { return 32 * used_slots(ncols) + 64; }
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

// ---------------------------------------------------------------------------
// Activation preparation: grid (ncols, n_jobs), 256 threads.
// ---------------------------------------------------------------------------
// Lane slot of MMA lane L = 4g + c in a record. NT == 1: column groups g < 4
// carry hi parts of columns 0..ncols-1, g >= 4 the lo parts; NT == 2: g < ncols.
__host__ __device__ __forceinline__ int lane_slot(int nt, int lane, int ncols) {
    const int g = lane >> 2, c = lane & 3;
    return nt == 1 ? (((g & 3) + (g >> 2) * ncols) * 4 + c) : lane;
}

// Accumulator start of MMA column n (the -sum for all-ones codes): stored at
// both places lane group n/2 loads it from.
__device__ __forceinline__ void put_start(uint8_t *rec, int s_used, int n, float v) {
    float *q = reinterpret_cast<float *>(rec + 32 * s_used + (n >> 1) * 16) + (n & 1);
    q[0] = v;
    q[2] = v;
}

__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
    return uint32_t(__half_as_ushort(lo)) | (uint32_t(__half_as_ushort(hi)) << 16);
}

template <int NT>
__global__ void __launch_bounds__(kPrepThreads) mv_prep_kernel(
    const __grid_constant__ MvPrepJob single, const MvPrepJob *__restrict__ jobs, int ncols) {
    // The mat-vec kernel that follows may start its prologue (barrier set-up,
    // weight loads) now; it waits for this grid before reading the fragments.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const MvPrepJob &J = jobs ? jobs[blockIdx.y] : single;
    const int K = J.K;
    const int j = blockIdx.x;  // activation column
    const float *xj = J.x + size_t(j) * K;
    const int tid = threadIdx.x;
    const int nb = K / 64;

    // 1) column scale 2^s with max|x * 2^s| in [2^14, 2^15). The thread's first
    //    16-element group stays in registers for step 2.
    float first[16];
    float m = 0.0f;
    if (tid < nb * 4) {
        if ((reinterpret_cast<uintptr_t>(xj) & 15u) == 0) {
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
            for (int i = 0; i < 16; ++i) first[i] = xj[tid * 16 + i];
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(first[i]));
    }
    for (int k = (kPrepThreads + tid) * 16; k < K; k += kPrepThreads * 16)
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(xj[k + i]));
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
    for (int idx = tid; idx < nb * 4; idx += kPrepThreads) {
        const int b = idx >> 2, c = idx & 3;
        const float *xe = xj + b * 64 + c * 16;
        __half hi[16], lo[16];
        float base_hi = 0.0f, base_lo = 0.0f;  // sum over the block of part * 4^m * 2^-24
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float xv = idx == tid ? first[i] : xe[i];
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

        const int su = used_slots(ncols), rb = rec_bytes(ncols);
        uint8_t *rec0 = J.prep + kPrepHeader + size_t(b) * NT * rb;
        int lane_hi, lane_lo, slot_hi, slot_lo;
        uint8_t *rec_hi, *rec_lo;
        if (NT == 1) {
            rec_hi = rec_lo = rec0;
            lane_hi = 4 * j + c;
            lane_lo = 4 * (4 + j) + c;
            slot_hi = j;
            slot_lo = 4 + j;
        } else {
            rec_hi = rec0;
            rec_lo = rec0 + rb;
            lane_hi = lane_lo = 4 * j + c;
            slot_hi = slot_lo = j;
        }
        const int sh = lane_slot(NT, lane_hi, ncols), sl = lane_slot(NT, lane_lo, ncols);
        *reinterpret_cast<uint4 *>(rec_hi + sh * 16) = make_uint4(rh[0], rh[1], rh[2], rh[3]);
        *reinterpret_cast<uint4 *>(rec_hi + 16 * su + sh * 16) = make_uint4(rh[4], rh[5], rh[6], rh[7]);
        *reinterpret_cast<uint4 *>(rec_lo + sl * 16) = make_uint4(rl[0], rl[1], rl[2], rl[3]);
        *reinterpret_cast<uint4 *>(rec_lo + 16 * su + sl * 16) = make_uint4(rl[4], rl[5], rl[6], rl[7]);
        if (c == 0) {
            put_start(rec_hi, su, slot_hi, -base_hi);
            put_start(rec_lo, su, slot_lo, -base_lo);
        }
        // Column 0's CTA also zeroes the column starts of unused columns.
        if (j == 0 && c == 0) {
            for (int t = 0; t < NT; ++t) {
                uint8_t *rt = rec0 + t * rb;
                for (int u = ncols; u < (NT == 1 ? 4 : 8); ++u) {
                    put_start(rt, su, u, 0.0f);
                    if (NT == 1) put_start(rt, su, 4 + u, 0.0f);
                }
            }
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

// fp16 scale at a shared-memory address, as f32 (16-bit load + convert).
__device__ __forceinline__ float lds_half_as_float(const uint8_t *p) {
    return __half2float(*reinterpret_cast<const __half *>(p));
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

// Consumer warps per CTA for RG 16-row groups per warp (256-row tiles).
template <int RG>
constexpr int consumer_warps() { return kTileRows / (16 * RG); }
template <int RG>
constexpr int cta_threads() { return (consumer_warps<RG>() + 1) * 32; }

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// NT: MMA n-tiles (1 for ncols <= 4, 2 for 5..8); RG: 16-row groups per warp.
template <int NT, int RG>
__global__ void __launch_bounds__(cta_threads<RG>(), 1)
    mv_tc_kernel(const __grid_constant__ MvJob single, const MvParams p) {
    constexpr int kCW = consumer_warps<RG>();
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
                for (int ch = 0; ch < J->n_chunks; ++ch) {
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
                             J->prep + kPrepHeader + size_t(ch) * kRStageBytes,
                             kRStageBytes, &full[stage]);
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
    // B lanes that carry data: NT==1 -> groups g < ncols (hi) and 4 <= g < 4+ncols (lo)
    bool lane_used[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t)
        lane_used[t] = (NT == 1) ? ((g & 3) < p.ncols) : (g < p.ncols);

    const int slot = lane_slot(NT, lane, p.ncols);
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
        float acc[RG][NT][4];
#pragma unroll
        for (int rg = 0; rg < RG; ++rg)
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[rg][t][k] = 0.0f;

        bool ok = true;
        for (int ch = 0; ch < n_chunks; ++ch) {
            const bool got = mbar_wait(&full[stage], ph, p.err, kTagMvFull) &&
                             !*(volatile int *)&s_abort;
            if (!__all_sync(0xffffffffu, got)) {  // warp-uniform decision
                s_abort = 1;
                ok = false;
                break;
            }
            const uint8_t *ws = w_stage + stage * kWStageBytes;
            const uint8_t *rs = r_stage + stage * kRStageBytes;
            // Block pairs (36 bytes per row). The words and scales of pair pr+1 are
            // loaded before pair pr's MMAs, which are issued step-major across the
            // pair's two accumulation chains.
            const int ra = warp * 16 + g;
            const uint8_t *row_a = ws + ra * kChunkBytes;
            const uint8_t *row_b = row_a + 8 * kChunkBytes;
            PairRegs nxt = load_pair(row_a, row_b, 0, c);
#pragma unroll
            for (int pr = 0; pr < kChunkBlocks / 2; ++pr) {
                const PairRegs cur = nxt;
                if (pr + 1 < kChunkBlocks / 2) nxt = load_pair(row_a, row_b, pr + 1, c);
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        const uint8_t *rec = rs + ((2 * pr + u) * NT + t) * kRecBytes;
                        if (lane_used[t]) {  // unused lanes keep their zero registers
                            fr0[u][t] = *reinterpret_cast<const uint4 *>(rec + slot * 16);
                            fr1[u][t] = *reinterpret_cast<const uint4 *>(rec + 16 * su + slot * 16);
                        }
                    }
                uint32_t sa[2], sb[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    sa[u] = __umulhi(cur.wa[u], 0x01000000u);  // >> 8 on the FMA pipe
                    sb[u] = __umulhi(cur.wb[u], 0x01000000u);
                }
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    float4 cc[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        cc[u] = *reinterpret_cast<const float4 *>(
                            rs + ((2 * pr + u) * NT + t) * kRecBytes + 32 * su + 16 * c);
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const uint32_t mask = 0x00030003u << (2 * m);
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            float dd[4];
                            mma_16816(dd, cur.wa[u] & mask, cur.wb[u] & mask, sa[u] & mask,
                                      sb[u] & mask, pick(fr0[u][t], fr1[u][t], 2 * m),
                                      pick(fr0[u][t], fr1[u][t], 2 * m + 1), cc[u].x, cc[u].y,
                                      cc[u].z, cc[u].w);
                            cc[u] = make_float4(dd[0], dd[1], dd[2], dd[3]);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        acc[0][t][0] = fmaf(cur.da[u], cc[u].x, acc[0][t][0]);
                        acc[0][t][1] = fmaf(cur.da[u], cc[u].y, acc[0][t][1]);
                        acc[0][t][2] = fmaf(cur.db[u], cc[u].z, acc[0][t][2]);
                        acc[0][t][3] = fmaf(cur.db[u], cc[u].w, acc[0][t][3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == kStages) {
                stage = 0;
                ph ^= 1u;
            }
        }
        if (!ok) break;

        // ---- epilogue: combine hi + lo, undo the column scale, store ----
        const float *out_scale = reinterpret_cast<const float *>(J->prep);
        const int N = J->N;
#pragma unroll
        for (int rg = 0; rg < RG; ++rg) {
            const int row_a = tile * kTileRows + warp * (16 * RG) + rg * 16 + g;
            const int row_b = row_a + 8;
            float v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (NT == 1)
                    v[k] = acc[rg][0][k] + __shfl_xor_sync(0xffffffffu, acc[rg][0][k], 2);
                else
                    v[k] = acc[rg][0][k] + acc[rg][NT - 1][k];
            }
            if (NT == 1 && c >= 2) continue;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int col = 2 * c + k;
                if (col < p.ncols) {
                    const float sc = out_scale[col];
                    if (row_a < N) J->y[size_t(col) * N + row_a] = v[k] * sc;
                    if (row_b < N) J->y[size_t(col) * N + row_b] = v[2 + k] * sc;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Generic mat-vec (any K % 64 == 0, any alignment): one warp per row, f32 on
// CUDA cores, block-wise: s = sum (q - 1) * x over the block, then acc += d*s.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) mv_generic_kernel(const uint8_t *__restrict__ w,
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

// One 16-row group per consumer warp: 16 consumer warps per CTA for both
// n-tile counts.
constexpr int kRG1 = 1;
constexpr int kRG2 = 1;

std::mutex g_attr_mu;
bool g_attr_done[64][2];

cudaError_t ensure_attrs(int nt) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (dev < 64 && g_attr_done[dev][nt - 1]) return cudaSuccess;
    if (nt == 1)
        e = cudaFuncSetAttribute(mv_tc_kernel<1, kRG1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBudget + 2 * kMaxStages * 8);
    else
        e = cudaFuncSetAttribute(mv_tc_kernel<2, kRG2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBudget + 2 * kMaxStages * 8);
    if (e == cudaSuccess && dev < 64) g_attr_done[dev][nt - 1] = true;
    return e;
}

bool make_job(MvJob &J, const uint8_t *w, const uint8_t *prep, float *y, int64_t N, int64_t K) {
    std::memset(&J, 0, sizeof(J));
    const uint64_t row_bytes = uint64_t(K / 64) * 18;
    if (!encode_tmap_2d(&J.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, row_bytes, uint64_t(N), row_bytes,
                        kChunkBytes, kTileRows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return false;
    J.prep = prep;
    J.y = y;
    J.N = int(N);
    J.nb = int(K / 64);
    J.n_chunks = int(K / 512);
    J.n_tiles = int((N + kTileRows - 1) / kTileRows);
    return true;
}

cudaError_t launch_prep(const MvPrepJob &single, const MvPrepJob *jobs, int n_jobs, int ncols,
                        cudaStream_t s) {
    dim3 grid(ncols, n_jobs);
    if (n_tiles_for(ncols) == 1)
        mv_prep_kernel<1><<<grid, kPrepThreads, 0, s>>>(single, jobs, ncols);
    else
        mv_prep_kernel<2><<<grid, kPrepThreads, 0, s>>>(single, jobs, ncols);
    return cudaGetLastError();
}

// The tensor-core kernel is launched as a programmatic dependent of the prep
// kernel: its prologue and first weight loads overlap the prep's tail; its
// producer waits for the prep grid before loading any activation fragment.
cudaError_t launch_tc(const MvJob &single, const MvParams &prm, int grid, cudaStream_t s) {
    const int nt = n_tiles_for(prm.ncols);
    cudaError_t e = ensure_attrs(nt);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (nt == 1) {
        cfg.blockDim = dim3(cta_threads<kRG1>());
        cfg.dynamicSmemBytes = smem_bytes_for(prm.ncols);
        e = cudaLaunchKernelEx(&cfg, mv_tc_kernel<1, kRG1>, single, prm);
    } else {
        cfg.blockDim = dim3(cta_threads<kRG2>());
        cfg.dynamicSmemBytes = smem_bytes_for(prm.ncols);
        e = cudaLaunchKernelEx(&cfg, mv_tc_kernel<2, kRG2>, single, prm);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_generic(const uint8_t *w, const float *x, float *y, int64_t N, int64_t K,
                           int ncols, cudaStream_t s) {
    mv_generic_kernel<<<unsigned((N + 7) / 8), 256, 0, s>>>(w, x, y, int(N), int(K), ncols);
    return cudaGetLastError();
}

}  // namespace

size_t matvec_workspace_bytes(int64_t K, int ncols) { return prep_bytes_for(K, ncols); }

bool matvec_fast_path_ok(const void *w, int64_t K) {
    return K % 512 == 0 && (reinterpret_cast<uintptr_t>(w) & 15u) == 0;
}

int matvec_run(const uint8_t *w, const float *x, float *y, int64_t N, int64_t K, int ncols,
               void *ws, size_t ws_bytes, cudaStream_t s) {
    if (!matvec_fast_path_ok(w, K)) return cuda_status(launch_generic(w, x, y, N, K, ncols, s));
    if (ws_bytes < prep_bytes_for(K, ncols)) return Q2_0_EINVAL;
    unsigned long long *err = error_word_ptr();
    if (!err) return Q2_0_ECUDA;
    uint8_t *prep = static_cast<uint8_t *>(ws);
    MvPrepJob pj{x, prep, int(K)};
    cudaError_t e = launch_prep(pj, nullptr, 1, ncols, s);
    if (e != cudaSuccess) return Q2_0_ECUDA;
    MvJob J;
    if (!make_job(J, w, prep, y, N, K)) return Q2_0_ECUDA;
    MvParams prm{nullptr, nullptr, nullptr, ncols, n_stages_for(ncols), err};
    const int grid = std::max(1, std::min(J.n_tiles, sm_count()));
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
    q2::MvJob *d_jobs = nullptr;
    q2::MvItem *d_items = nullptr;
    int *d_cta_begin = nullptr;
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
            total += prep_bytes_for(descs[fast[j]].K, ncols);
        }
        std::vector<MvJob> jobs(P->n_fast);
        std::vector<MvPrepJob> pjobs(P->n_fast);
        if (cudaMalloc(&P->d_prep, total) != cudaSuccess) st = Q2_0_ECUDA;
        for (int j = 0; j < P->n_fast && st == Q2_0_OK; ++j) {
            const q2_0_mv_desc &d = descs[fast[j]];
            if (!make_job(jobs[j], static_cast<const uint8_t *>(d.w), P->d_prep + off[j], d.y, d.N,
                          d.K))
                st = Q2_0_ECUDA;
            pjobs[j] = MvPrepJob{d.x, P->d_prep + off[j], int(d.K)};
        }
        // Longest-processing-time-first schedule of (job, tile) items over one CTA
        // per SM; cost of an item = rows in the tile x K.
        std::vector<MvItem> items;
        std::vector<double> cost;
        for (int j = 0; j < P->n_fast; ++j)
            for (int t = 0; t < jobs[j].n_tiles; ++t) {
                items.push_back(MvItem{j, t});
                const int rows = std::min(kTileRows, jobs[j].N - t * kTileRows);
                cost.push_back(double(rows) * jobs[j].nb);
            }
        std::vector<int> order(items.size());
        for (size_t k = 0; k < order.size(); ++k) order[k] = int(k);
        std::stable_sort(order.begin(), order.end(),
                         [&](int a, int b) { return cost[a] > cost[b]; });
        const int grid = std::max(1, std::min<int>(sm_count(), int(items.size())));
        using Load = std::pair<double, int>;
        std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
        for (int c = 0; c < grid; ++c) heap.push(Load(0.0, c));
        std::vector<std::vector<MvItem>> per_cta(grid);
        for (int k : order) {
            Load l = heap.top();
            heap.pop();
            per_cta[l.second].push_back(items[k]);
            heap.push(Load(l.first + cost[k], l.second));
        }
        std::vector<MvItem> flat;
        std::vector<int> begin(grid + 1, 0);
        for (int c = 0; c < grid; ++c) {
            begin[c] = int(flat.size());
            flat.insert(flat.end(), per_cta[c].begin(), per_cta[c].end());
        }
        begin[grid] = int(flat.size());
        P->grid = grid;
        if (st == Q2_0_OK &&
            (cudaMalloc(&P->d_jobs, sizeof(MvJob) * jobs.size()) != cudaSuccess ||
             cudaMalloc(&P->d_items, sizeof(MvItem) * flat.size()) != cudaSuccess ||
             cudaMalloc(&P->d_cta_begin, sizeof(int) * begin.size()) != cudaSuccess ||
             cudaMalloc(&P->d_prep_jobs, sizeof(MvPrepJob) * pjobs.size()) != cudaSuccess))
            st = Q2_0_ECUDA;
        if (st == Q2_0_OK &&
            (cudaMemcpy(P->d_jobs, jobs.data(), sizeof(MvJob) * jobs.size(),
                        cudaMemcpyHostToDevice) != cudaSuccess ||
             cudaMemcpy(P->d_items, flat.data(), sizeof(MvItem) * flat.size(),
                        cudaMemcpyHostToDevice) != cudaSuccess ||
             cudaMemcpy(P->d_cta_begin, begin.data(), sizeof(int) * begin.size(),
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
        if (launch_prep(none, P->d_prep_jobs, P->n_fast, P->ncols, s) != cudaSuccess)
            return Q2_0_ECUDA;
        MvJob dummy;
        std::memset(&dummy, 0, sizeof(dummy));
        MvParams prm{P->d_jobs, P->d_items, P->d_cta_begin, P->ncols, n_stages_for(P->ncols),
                     P->err};
        if (launch_tc(dummy, prm, P->grid, s) != cudaSuccess) return Q2_0_ECUDA;
    }
    for (const q2_0_mv_desc &d : P->generic)
        if (launch_generic(static_cast<const uint8_t *>(d.w), d.x, d.y, d.N, d.K, P->ncols, s) !=
            cudaSuccess)
            return Q2_0_ECUDA;
    return Q2_0_OK;
}

}  // namespace q2
