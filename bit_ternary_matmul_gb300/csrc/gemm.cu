// Q2_0 prefill GEMM on the 5th-generation tensor cores (tcgen05, sm_103a):
//   Y[m][n] = sum_k W[n][k] X[m][k]   (M tokens, N weight rows).
//
// Source: "WebGPU: add Q2_0 support" (bisque.today write-up of llama.cpp
// PR 30914), shader paragraph — the tiled matrix multiply unpacks each thread's
// 16 codes into shared memory as half precision before the product. Here the
// unpacked operand is (q - 1) * d in fp16, which is exact for every code and
// every fp16 d with |2d| <= 65504, so the scale needs no separate pass.
//
// Data flow of one CTA (persistent over output units of 256 weight rows x 128
// tokens; K in 64-wide slabs, one Q2_0 block per row per slab):
//   warp 0   TMA producer: the packed W box (256 rows x 144 B = 8 slabs) into a
//            2-deep ring; per slab the X_hi (and X_lo) tile [128 x 64] fp16 with
//            128-byte swizzle into a 4-deep ring.
//   warp 1   TMEM allocation (all 512 columns) and the MMA issuer (one thread):
//            per slab, for each of the two 128-row weight tiles, 4 K=16 steps
//            for hi and lo: tcgen05.mma kind::f16 M=128 N=128 with the A operand
//            (expanded weights) in TMEM and B (X) in shared memory; the fp32
//            accumulators are TMEM columns 0..255. tcgen05.commit frees the slab.
//   warps 2-9   expansion: thread r decodes weight row r's block of the slab
//            into 64 fp16 values (q - 1) * d and writes them to the slab's TMEM
//            A slot with one tcgen05.st (32 columns of its lane).
//   warps 10-17 epilogue: tcgen05.ld of the accumulators, F32 stores, then the
//            accumulators are released to the MMA issuer for the next unit.
// Two weight tiles share every X tile, so shared memory carries 96 bytes per
// clock of MMA work instead of the whole bandwidth a single 128 x 128 tile
// would need; the weights never pass through shared memory once expanded.
//
#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "q2_0_device.cuh"
#include "q2_0_tcgen05.cuh"
#include "q2_0_internal.h"

namespace q2 {

namespace {

constexpr int kBM = 128;            // weight rows per MMA tile (MMA M)
constexpr int kWT = 2;              // weight tiles per CTA unit (256 rows)
constexpr int kBN = 128;            // tokens per unit (MMA N)
constexpr int kSlabK = 64;          // one Q2_0 block
constexpr int kStages = 4;          // X ring and TMEM A-slot ring depth
constexpr int kWStages = 2;         // packed-W ring depth (8 slabs each)
constexpr int kExpandWarps = 8;     // one thread per weight row of the unit
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kExpandWarps + kEpiWarps) * 32;  // 576
constexpr int kXTileBytes = kBN * kSlabK * 2;     // 16 KB per part
constexpr int kWBoxBytes = kWT * kBM * 144;       // 36 KB
constexpr int kTmemCols = 512;                    // 256 accumulator + 256 A-slot columns
constexpr int kAccCol = 0;                        // tile t accumulator at t * 128
constexpr int kASlotCol = 256;                    // slot s, tile t at 256 + (2s + t) * 32
constexpr int kMaxGrid = 160;                     // stream-K CTAs (>= SMs of a GB300)
constexpr int kPartialBytes = kBN * kWT * kBM * 4;  // one fp32 unit tile

constexpr int kTagGemm = 200;

// One product of a launch: Y = W X^T with its own tensor maps and its place in
// the launch's slab order. A q2_0_mul_mat call is a launch of one product; a
// plan (q2_0_mm_plan_*) pools several, e.g. the projections that share one X.
struct GemmJob {  // 64-byte aligned through its CUtensorMap members
    CUtensorMap w_map;     // uint8 [N][K/64*18], box {144, 256}
    CUtensorMap xh_map;    // fp16 [M][K], box {64, 128}, 128B swizzle
    CUtensorMap xl_map;
    float *y;              // [M][N]
    const int *row_shift;  // [M]: X row m entered the MMA as X * 2^row_shift[m]
    long long slab0;       // the product's first slab in the launch's slab order
    int M, N, K;
    int n_mtiles;          // units = (N / 256 rounded up) x n_mtiles (M / 128 rounded up)
};

struct GemmArgs {
    GemmJob single;         // the product of a single call
    const GemmJob *jobs;    // a plan's products in device memory, slab0 ascending; or null
    int n_jobs;
    int split;              // 1: hi + lo, 0: hi only
    long long total_slabs;  // sum over the products of units * K / 64: the stream-K space
    float *partials;        // 2 slots per CTA of kBN x (kWT * kBM) fp32
    unsigned long long *err;
};

// Where global slab g lies: its product, unit, slab within the unit and the
// unit's first global slab. Products are concatenated in the slab order, each
// unit-major (a unit's K slabs consecutive).
struct SlabPos {
    const GemmJob *job;
    int u, kb, n_slabs;
    long long ustart;
};
__device__ __forceinline__ SlabPos locate(const GemmArgs &a, long long g) {
    const GemmJob *J = &a.single;
    if (a.jobs) {
        int j = 0;
        while (j + 1 < a.n_jobs && a.jobs[j + 1].slab0 <= g) ++j;
        J = a.jobs + j;
    }
    SlabPos p;
    p.job = J;
    p.n_slabs = J->K / kSlabK;
    const long long local = g - J->slab0;
    p.u = int(local / p.n_slabs);
    p.kb = int(local % p.n_slabs);
    p.ustart = J->slab0 + (long long)p.u * p.n_slabs;
    return p;
}

// Stream-K: CTA c owns global slabs [T*c/G, T*(c+1)/G) of the unit-major slab
// order. A unit whose slabs span several CTAs is summed afterwards by
// gemm_reduce_kernel from the CTAs' partial tiles, in K order.
__host__ __device__ inline long long sk_begin(int c, long long T, int G) {
    return (T * c) / G;
}
__host__ __device__ inline int sk_owner(long long g, long long T, int G) {
    return int(((g + 1) * G + T - 1) / T) - 1;  // max c with sk_begin(c) <= g
}
// End slab (exclusive, within the unit) of a segment starting at slab kb with
// rem slabs left in the CTA's range.
__host__ __device__ inline int seg_end(int n_slabs, int kb, long long rem) {
    return rem < (long long)(n_slabs - kb) ? kb + int(rem) : n_slabs;
}

// Instruction descriptor, kind::f16: D f32, A and B f16, both K-major, N, M.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n) {
    return (1u << 4) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

// ---------------------------------------------------------------------------
// Prepass: X [M][K] (F32, or F16 whose values are already exact fp16) -> fp16
// hi (and lo) [M][K] in the permuted K order, each row scaled by a power of
// two first. Row m with M_m = max |x| = f * 2^e (f in [0.5, 1)) is multiplied
// by 2^s, s = 15 - e, so that its largest element lies in [2^14, 2^15): hi
// never overflows fp16, and hi + lo hold each element to 2^-22 of its value
// plus 2^-39 of the row maximum. F16 rows are only scaled
// up (s >= 0), which keeps them exact. The scaling is exact and undone on the
// f32 result (y = acc * 2^-s). One CTA per row and grid row y per activation
// matrix of the launch; X 16-byte aligned.
// ---------------------------------------------------------------------------
constexpr int kMaxPrepX = 8;
struct GemmPrepSet {  // the distinct activation matrices of one prep launch
    const void *x[kMaxPrepX];
    __half *xh[kMaxPrepX];
    __half *xl[kMaxPrepX];  // null unless split
    int *row_shift[kMaxPrepX];
    int M[kMaxPrepX];
    int K[kMaxPrepX];
    int split;
};

__device__ __forceinline__ void load16(const float *p, float (&v)[16]) {
    const float4 *src = reinterpret_cast<const float4 *>(p);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 f = src[q];
        v[4 * q] = f.x;
        v[4 * q + 1] = f.y;
        v[4 * q + 2] = f.z;
        v[4 * q + 3] = f.w;
    }
}
__device__ __forceinline__ void load16(const __half *p, float (&v)[16]) {
    const uint4 *src = reinterpret_cast<const uint4 *>(p);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const uint4 u = src[q];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[k]));
            v[8 * q + 2 * k] = f.x;
            v[8 * q + 2 * k + 1] = f.y;
        }
    }
}

// v * 2^e for |e| <= 252 with two exact power-of-two factors (each a normal f32).
__device__ __forceinline__ float mul_pow2(float v, int e) {
    const int e1 = e / 2, e2 = e - e1;
    return v * __int_as_float((127 + e1) << 23) * __int_as_float((127 + e2) << 23);
}

constexpr int kPrepThreads = 128;
constexpr int kPrepCache = 3;

// One CTA per row: the row maximum by a block reduction, then the conversion.
template <typename XT>
__global__ void __launch_bounds__(kPrepThreads) gemm_prep_kernel(
    const __grid_constant__ GemmPrepSet ps) {
    // The GEMM kernel that follows may start its prologue and weight loads now;
    // it waits for this grid before reading X.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int e = blockIdx.y, m = blockIdx.x;
    if (m >= ps.M[e]) return;  // grid x covers the set's largest M
    const XT *__restrict__ x = static_cast<const XT *>(ps.x[e]);
    __half *__restrict__ xh = ps.xh[e];
    __half *__restrict__ xl = ps.xl[e];
    int *__restrict__ row_shift = ps.row_shift[e];
    const int K = ps.K[e], split = ps.split;
    const int tid = threadIdx.x, lane = tid & 31;
    const XT *xr = x + size_t(m) * K;
    const int groups = K / 16;
    // the first kPrepCache groups of 16 per thread stay in registers between
    // the maximum and the conversion (all of a row up to K = 6144)
    float cache[kPrepCache][16];
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < kPrepCache; ++c) {
        const int gi = tid + c * kPrepThreads;
        if (gi < groups) {
            load16(xr + gi * 16, cache[c]);
#pragma unroll
            for (int t = 0; t < 16; ++t) amax = fmaxf(amax, fabsf(cache[c][t]));
        }
    }
    for (int gi = tid + kPrepCache * kPrepThreads; gi < groups; gi += kPrepThreads) {
        float v[16];
        load16(xr + gi * 16, v);
#pragma unroll
        for (int t = 0; t < 16; ++t) amax = fmaxf(amax, fabsf(v[t]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    __shared__ float red[kPrepThreads / 32];
    if (lane == 0) red[tid >> 5] = amax;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kPrepThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    int sh = 0;
    if (amax > 0.0f && amax <= 3.402823466e38f) {
        int e;
        frexpf(amax, &e);
        sh = 15 - e;
        if (sizeof(XT) == 2 && sh < 0) sh = 0;
    }
    if (tid == 0) row_shift[m] = sh;
    __half *hr = xh + size_t(m) * K;
    __half *lr = split ? xl + size_t(m) * K : nullptr;
    auto convert = [&](int gi, const float (&v)[16]) {
        uint32_t hw[8], lw[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const float a0 = mul_pow2(v[t], sh), a1 = mul_pow2(v[t + 8], sh);
            const __half h0 = __float2half_rn(a0);
            const __half h1 = __float2half_rn(a1);
            hw[t] = uint32_t(__half_as_ushort(h0)) | (uint32_t(__half_as_ushort(h1)) << 16);
            const __half l0 = __float2half_rn(a0 - __half2float(h0));
            const __half l1 = __float2half_rn(a1 - __half2float(h1));
            lw[t] = uint32_t(__half_as_ushort(l0)) | (uint32_t(__half_as_ushort(l1)) << 16);
        }
        uint4 *dh = reinterpret_cast<uint4 *>(hr + gi * 16);
        dh[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        dh[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
        if (split) {
            uint4 *dl = reinterpret_cast<uint4 *>(lr + gi * 16);
            dl[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            dl[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
        }
    };
#pragma unroll
    for (int c = 0; c < kPrepCache; ++c) {
        const int gi = tid + c * kPrepThreads;
        if (gi < groups) convert(gi, cache[c]);
    }
    for (int gi = tid + kPrepCache * kPrepThreads; gi < groups; gi += kPrepThreads) {
        float v[16];
        load16(xr + gi * 16, v);
        convert(gi, v);
    }
}

// ---------------------------------------------------------------------------
// tcgen05 GEMM kernel
// ---------------------------------------------------------------------------
// Two fp16 values (q - 1) * d for k-slots (2j, 2j+1) of the permuted order: the
// codes of elements t and t+8 of a word (t = j % 8) with the magic exponent
// 0x6400 give 1024 + q in each half; subtract 1025, multiply by d (exact).
__device__ __forceinline__ uint32_t expand_pair(uint32_t word, int t, __half2 d2) {
    const uint32_t bits = ((word >> (2 * t)) & 0x00030003u) | 0x64006400u;
    __half2 v = *reinterpret_cast<const __half2 *>(&bits);
    v = __hmul2(__hsub2(v, __floats2half2_rn(1025.0f, 1025.0f)), d2);
    return *reinterpret_cast<uint32_t *>(&v);
}

__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmArgs a) {
    // The stream-K reduction that follows may be scheduled now; it waits for
    // this grid to finish before it reads any partial tile.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled X tiles
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *xh_s = smem;                                   // kStages x 16 KB
    uint8_t *xl_s = xh_s + kStages * kXTileBytes;           // kStages x 16 KB
    uint8_t *w_s = xl_s + kStages * kXTileBytes;            // kWStages x 36 KB
    uint64_t *bars = reinterpret_cast<uint64_t *>(w_s + kWStages * kWBoxBytes);
    uint64_t *x_full = bars;                 // [kStages]
    uint64_t *a_full = x_full + kStages;     // [kStages]
    uint64_t *slot_free = a_full + kStages;  // [kStages]
    uint64_t *w_full = slot_free + kStages;  // [kWStages]
    uint64_t *w_free = w_full + kWStages;    // [kWStages]
    uint64_t *acc_full = w_free + kWStages;  // [1]
    uint64_t *acc_empty = acc_full + 1;      // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + 1);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long g_begin = sk_begin(blockIdx.x, a.total_slabs, gridDim.x);
    const long long g_end = sk_begin(blockIdx.x + 1, a.total_slabs, gridDim.x);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&a_full[i], kExpandWarps);
            mbar_init(&slot_free[i], 1);
        }
        for (int i = 0; i < kWStages; ++i) {
            mbar_init(&w_full[i], 1);
            mbar_init(&w_free[i], kExpandWarps);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, kEpiWarps);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // Unit u of a product -> (row pair, token tile) with the token tile fastest,
    // so CTAs running together share weight rows in L2.
    auto unit_coords = [&](const SlabPos &p, int &n0, int &m0) {
        n0 = (p.u / p.job->n_mtiles) * (kWT * kBM);
        m0 = (p.u % p.job->n_mtiles) * kBN;
    };

    if (warp == 0) {
        // ---------------------------- TMA producer ----------------------------
        if (lane == 0) {
            const uint32_t x_bytes = kXTileBytes * (a.split ? 2 : 1);
            int st = 0, wst = 0;
            uint32_t ph = 0, wph = 0;
            bool ok = true, prep_done = false;
            for (long long g = g_begin; g < g_end && ok;) {
                const SlabPos p = locate(a, g);
                const int kb = p.kb;
                const int ke = seg_end(p.n_slabs, kb, g_end - g);
                g += ke - kb;
                int n0, m0;
                unit_coords(p, n0, m0);
                const GemmJob *J = p.job;
                for (int kk = kb; kk < ke; ++kk) {
                    if ((kk & 7) == 0 || kk == kb) {
                        if (!mbar_wait(&w_free[wst], wph ^ 1u, a.err, kTagGemm + 1)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&w_full[wst], kWBoxBytes);
                        tma_load_2d(w_s + wst * kWBoxBytes, &J->w_map, (kk >> 3) * 144, n0,
                                    &w_full[wst]);
                    }
                    if (!mbar_wait(&slot_free[st], ph ^ 1u, a.err, kTagGemm + 2)) {
                        ok = false;
                        break;
                    }
                    if (!prep_done) {  // X comes from the prepass
                        asm volatile("griddepcontrol.wait;" ::: "memory");
                        prep_done = true;
                    }
                    mbar_arrive_expect_tx(&x_full[st], x_bytes);
                    tma_load_2d(xh_s + st * kXTileBytes, &J->xh_map, kk * kSlabK, m0, &x_full[st]);
                    if (a.split)
                        tma_load_2d(xl_s + st * kXTileBytes, &J->xl_map, kk * kSlabK, m0,
                                    &x_full[st]);
                    if (++st == kStages) {
                        st = 0;
                        ph ^= 1u;
                    }
                    if ((kk & 7) == 7 || kk == ke - 1) {
                        if (++wst == kWStages) {
                            wst = 0;
                            wph ^= 1u;
                        }
                    }
                }
            }
            if (!ok) {
                *(volatile int *)abort_flag = 1;
                // Let the copies already issued land before the CTA exits (bounded).
                int s2 = st, p2 = int(ph);
                for (int k = 0; k < kStages; ++k) {
                    if (--s2 < 0) {
                        s2 = kStages - 1;
                        p2 ^= 1;
                    }
                    mbar_wait(&x_full[s2], uint32_t(p2), a.err, kTagGemm + 9);
                }
                int w2 = wst, q2p = int(wph);
                for (int k = 0; k < kWStages; ++k) {
                    if (--w2 < 0) {
                        w2 = kWStages - 1;
                        q2p ^= 1;
                    }
                    mbar_wait(&w_full[w2], uint32_t(q2p), a.err, kTagGemm + 10);
                }
            }
        }
    } else if (warp == 1) {
        // ----------------------------- MMA issuer -----------------------------
        // The whole warp runs the loop (addresses and descriptors stay
        // warp-uniform); the elected lane issues the MMAs and their commits.
        const uint32_t idesc = idesc_f16(kBM, kBN);
        const bool leader = elect_one();
        int st = 0;
        uint32_t ph = 0;
        bool ok = true;
        int nu = 0;
        for (long long g = g_begin; g < g_end && ok; ++nu) {
            const SlabPos p = locate(a, g);
            const int kb = p.kb;
            const int ke = seg_end(p.n_slabs, kb, g_end - g);
            g += ke - kb;
            if (nu > 0 &&
                !__all_sync(0xffffffffu,
                            mbar_wait(acc_empty, uint32_t((nu - 1) & 1), a.err, kTagGemm + 3))) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int kk = kb; kk < ke; ++kk) {
                const bool got = mbar_wait2(&x_full[st], ph, kTagGemm + 4, &a_full[st], ph,
                                            kTagGemm + 5, a.err, kWaitLimitNs);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t h_addr = smem_addr(xh_s + st * kXTileBytes);
                const uint32_t l_addr = smem_addr(xl_s + st * kXTileBytes);
                if (leader) {
                    // consecutive MMAs alternate between the two accumulators
#pragma unroll
                    for (int ks = 0; ks < kSlabK / 16; ++ks) {
                        const uint64_t hd = sw128_desc(h_addr + ks * 32);
                        const uint64_t ld = sw128_desc(l_addr + ks * 32);
#pragma unroll
                        for (int t = 0; t < kWT; ++t)
                            tc_mma_f16_ta(tmem_base + kAccCol + t * kBN,
                                          tmem_base + kASlotCol + (2 * st + t) * 32 + ks * 8, hd,
                                          idesc, (kk > kb || ks > 0) ? 1u : 0u);
                        if (a.split) {
#pragma unroll
                            for (int t = 0; t < kWT; ++t)
                                tc_mma_f16_ta(tmem_base + kAccCol + t * kBN,
                                              tmem_base + kASlotCol + (2 * st + t) * 32 + ks * 8,
                                              ld, idesc, 1u);
                        }
                    }
                    tc_commit(&slot_free[st]);
                }
                __syncwarp();
                if (++st == kStages) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            if (ok && leader) tc_commit(acc_full);
            __syncwarp();
        }
        if (!ok && leader) *(volatile int *)abort_flag = 1;
    } else if (warp < 2 + kExpandWarps) {
        // ------------------------------ expansion ------------------------------
        // Warp w may access TMEM lanes 32 * (w % 4) .. +31: quarter q = w % 4 of
        // weight tile t = (w - 2) / 4.
        const int q = warp & 3, t = (warp - 2) >> 2;
        const int row = t * kBM + q * 32 + lane;  // row within the 256-row unit
        const uint32_t lane_addr = uint32_t(q * 32) << 16;
        int st = 0, wst = 0;
        uint32_t ph = 0, wph = 0;
        bool ok = true;
        for (long long g = g_begin; g < g_end && ok;) {
            const SlabPos p = locate(a, g);
            const int kb = p.kb;
            const int ke = seg_end(p.n_slabs, kb, g_end - g);
            g += ke - kb;
            for (int kk = kb; kk < ke; ++kk) {
                const bool got =
                    (kk & 7) == 0 || kk == kb
                        ? mbar_wait2(&w_full[wst], wph, kTagGemm + 6, &slot_free[st], ph ^ 1u,
                                     kTagGemm + 7, a.err, kWaitLimitNs)
                        : mbar_wait(&slot_free[st], ph ^ 1u, a.err, kTagGemm + 7);
                if (!__all_sync(0xffffffffu, got)) {  // warp-uniform decision
                    ok = false;
                    break;
                }
                // row's block (kk & 7) in the packed box: 18 bytes at row*144 + 18*(kk&7)
                const int off = 18 * (kk & 7);
                const uint32_t *up = reinterpret_cast<const uint32_t *>(
                    w_s + wst * kWBoxBytes + row * 144 + (off & ~3));
                const uint32_t u0 = up[0], u1 = up[1], u2 = up[2], u3 = up[3], u4 = up[4];
                uint32_t dbits, wd[4];
                if ((off & 3) == 0) {  // even block: d in u0 low half, words straddle
                    dbits = u0 & 0xFFFFu;
                    wd[0] = __byte_perm(u0, u1, 0x5432);
                    wd[1] = __byte_perm(u1, u2, 0x5432);
                    wd[2] = __byte_perm(u2, u3, 0x5432);
                    wd[3] = __byte_perm(u3, u4, 0x5432);
                } else {  // odd block: d in u0 high half, words aligned
                    dbits = u0 >> 16;
                    wd[0] = u1;
                    wd[1] = u2;
                    wd[2] = u3;
                    wd[3] = u4;
                }
                const __half dh = __ushort_as_half(static_cast<unsigned short>(dbits));
                const __half2 d2 = __halves2half2(dh, dh);
                uint32_t r[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = expand_pair(wd[j >> 3], j & 7, d2);
                tmem_st32(tmem_base + lane_addr + kASlotCol + (2 * st + t) * 32, r);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                const bool box_done = (kk & 7) == 7 || kk == ke - 1;
                if (lane == 0) {
                    mbar_arrive(&a_full[st]);
                    if (box_done) mbar_arrive(&w_free[wst]);
                }
                if (box_done) {
                    if (++wst == kWStages) {
                        wst = 0;
                        wph ^= 1u;
                    }
                }
                if (++st == kStages) {
                    st = 0;
                    ph ^= 1u;
                }
            }
        }
    } else {
        // ------------------------------- epilogue -------------------------------
        // the row exponents come from the prepass (the producer waits for it
        // before loading X; the epilogue waits too before reading them)
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int q = warp & 3, t = (warp - 2 - kExpandWarps) >> 2;
        const uint32_t lane_addr = uint32_t(q * 32) << 16;
        const int rloc = t * kBM + q * 32 + lane;  // row within the unit
        // A warp whose wait timed out stops reading TMEM and writing.
        bool dead = false;
        int nu = 0;
        for (long long g = g_begin; g < g_end; ++nu) {
            const SlabPos p = locate(a, g);
            const int kb = p.kb;
            const int ke = seg_end(p.n_slabs, kb, g_end - g);
            g += ke - kb;
            int n0, m0;
            unit_coords(p, n0, m0);
            const int jM = p.job->M, jN = p.job->N;
            float *const jy = p.job->y;
            const int *const jshift = p.job->row_shift;
            if (!dead) {
                const bool got = mbar_wait(acc_full, uint32_t(nu & 1), a.err, kTagGemm + 8);
                dead = !__all_sync(0xffffffffu, got);
            }
            if (dead) continue;
            const bool whole = kb == 0 && ke == p.n_slabs;
            tc_fence_after();
            const int n = n0 + rloc;
            // partial tiles: slot 2c for a CTA's first segment, 2c + 1 for its last
            float *mine = a.partials +
                          size_t(2 * blockIdx.x + (g_begin >= p.ustart ? 0 : 1)) * (kPartialBytes / 4);
#pragma unroll 1
            for (int cb = 0; cb < kBN; cb += 32) {
                uint32_t v[32];
                tmem_ld32(tmem_base + lane_addr + kAccCol + t * kBN + cb, v);
                if (whole) {
                    // the 32 tokens' row exponents: one load per lane, shared by shuffles
                    const int sh = m0 + cb + lane < jM ? jshift[m0 + cb + lane] : 0;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int shj = __shfl_sync(0xffffffffu, sh, j);
                        const int m = m0 + cb + j;
                        if (n < jN && m < jM)
                            jy[size_t(m) * jN + n] = mul_pow2(__uint_as_float(v[j]), -shj);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        mine[(cb + j) * (kWT * kBM) + rloc] = __uint_as_float(v[j]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);  // accumulators free for the next segment
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Stream-K reduction: the units split across CTAs, summed from the partial
// tiles in K order (deterministic) and written to Y. grid = (kReduceSlices,
// GEMM grid): column c of the grid takes the unit in which CTA c's range
// begins, if that unit began in an earlier CTA's range and ends in c's (c is
// the unit's last contributor), so each split unit is summed exactly once;
// slice z takes 1/kReduceSlices of the unit's tile. Launched as a programmatic
// dependent of the GEMM: it waits for the GEMM grid before reading partials.
// ---------------------------------------------------------------------------
constexpr int kReduceSlices = 8;
constexpr int kReduceThreads = 256;

__global__ void __launch_bounds__(kReduceThreads) gemm_reduce_kernel(
    const __grid_constant__ GemmArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int G = int(gridDim.y), c = int(blockIdx.y);
    const long long total_slabs = a.total_slabs;
    const long long gb = sk_begin(c, total_slabs, G);
    const SlabPos p = locate(a, gb);
    const long long ustart = p.ustart;
    if (gb == ustart) return;  // c begins its first unit: not a split unit's finisher
    const int c_first = sk_owner(ustart, total_slabs, G);
    const int c_last = sk_owner(ustart + p.n_slabs - 1, total_slabs, G);
    if (c != c_last) return;
    const int M = p.job->M, N = p.job->N;
    float *const y = p.job->y;
    const int *const row_shift = p.job->row_shift;
    const float *const partials = a.partials;
    const int n0 = (p.u / p.job->n_mtiles) * (kWT * kBM);
    const int m0 = (p.u % p.job->n_mtiles) * kBN;
    constexpr int kRowVec = kWT * kBM / 4;          // float4 per token row
    constexpr int kTileVec = kBN * kRowVec;         // float4 per tile
    constexpr int kSliceVec = kTileVec / kReduceSlices;
    constexpr int kPer = kSliceVec / kReduceThreads;  // float4 per thread
    const bool vec_y = (N % 4) == 0 && (reinterpret_cast<uintptr_t>(y) & 15u) == 0;
    float4 acc[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int i_base = int(blockIdx.x) * kSliceVec + int(threadIdx.x);
    for (int cp = c_first; cp <= c_last; ++cp) {
        const float4 *piece = reinterpret_cast<const float4 *>(
            partials + size_t(2 * cp + (sk_begin(cp, total_slabs, G) >= ustart ? 0 : 1)) *
                           (kPartialBytes / 4));
        float4 v[kPer];
#pragma unroll
        for (int r = 0; r < kPer; ++r) v[r] = __ldcg(piece + i_base + r * kReduceThreads);
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
            acc[r].x += v[r].x;
            acc[r].y += v[r].y;
            acc[r].z += v[r].z;
            acc[r].w += v[r].w;
        }
    }
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
        const int i = i_base + r * kReduceThreads;
        const int m = m0 + i / kRowVec;
        const int nn = n0 + 4 * (i % kRowVec);
        if (m >= M) continue;
        float *yr = y + size_t(m) * N;
        const int sh = -row_shift[m];
        acc[r].x = mul_pow2(acc[r].x, sh);
        acc[r].y = mul_pow2(acc[r].y, sh);
        acc[r].z = mul_pow2(acc[r].z, sh);
        acc[r].w = mul_pow2(acc[r].w, sh);
        if (vec_y && nn + 3 < N) {
            *reinterpret_cast<float4 *>(yr + nn) = acc[r];
        } else {
            if (nn < N) yr[nn] = acc[r].x;
            if (nn + 1 < N) yr[nn + 1] = acc[r].y;
            if (nn + 2 < N) yr[nn + 2] = acc[r].z;
            if (nn + 3 < N) yr[nn + 3] = acc[r].w;
        }
    }
}

// ---------------------------------------------------------------------------
// Generic GEMM (any K % 64 == 0, any alignment): CUDA cores, f32.
// Block of 32 x 8 threads computes Y[m0..m0+8) x [n0..n0+32).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ld_x(const float *p) { return *p; }
__device__ __forceinline__ float ld_x(const __half *p) { return __half2float(*p); }

template <typename XT>
__global__ void __launch_bounds__(256) gemm_generic_kernel(const uint8_t *__restrict__ w,
                                                           const XT *__restrict__ x,
                                                           float *__restrict__ y, int M, int N,
                                                           int K) {
    const int n = blockIdx.x * 32 + threadIdx.x;
    const int m = blockIdx.y * 8 + threadIdx.y;
    if (n >= N || m >= M) return;
    const int nb = K / 64;
    float acc = 0.0f;
    for (int b = 0; b < nb; ++b) {
        const uint8_t *blk = w + (size_t(n) * nb + b) * 18;
        const float d = half_bits_to_float(uint32_t(blk[0]) | (uint32_t(blk[1]) << 8));
        float s = 0.0f;
        for (int wi = 0; wi < 4; ++wi) {
            const uint8_t *pw = blk + 2 + 4 * wi;
            const uint32_t word = uint32_t(pw[0]) | (uint32_t(pw[1]) << 8) |
                                  (uint32_t(pw[2]) << 16) | (uint32_t(pw[3]) << 24);
            const XT *xe = x + size_t(m) * K + b * 64 + wi * 16;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                s = fmaf(float(int((word >> (2 * i)) & 3u) - 1), ld_x(xe + i), s);
        }
        acc = fmaf(d, s, acc);
    }
    y[size_t(m) * N + n] = acc;
}

constexpr int gemm_smem_bytes() {
    return 1024 /* alignment slack */ + kStages * 2 * kXTileBytes + kWStages * kWBoxBytes +
           8 * (3 * kStages + 2 * kWStages + 2) + 32;
}

std::mutex g_mu;
bool g_attr[64];

cudaError_t ensure_attr() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_mu);
    if (dev < 64 && g_attr[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             gemm_smem_bytes());
    if (e == cudaSuccess && dev < 64) g_attr[dev] = true;
    return e;
}

bool tc_path_ok(const void *w, const void *x, int64_t K) {
    return K % 512 == 0 && (reinterpret_cast<uintptr_t>(w) & 15u) == 0 &&
           (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
}

}  // namespace

namespace {

struct GemmLayout {
    size_t part;      // bytes of X_hi (and of X_lo)
    size_t partials;  // offset of the partial tiles
    size_t shifts;    // offset of the per-row exponents (int [M])
    size_t total;
    int n_mtiles, grid;
    long long total_slabs;
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

int mtiles_of(int64_t M) { return int((M + kBN - 1) / kBN); }

// Slabs of one product: units (256 weight rows x 128 tokens) times K / 64.
long long slabs_of(int64_t M, int64_t N, int64_t K) {
    const long long units = (long long)((N + kWT * kBM - 1) / (kWT * kBM)) * mtiles_of(M);
    return units * (K / kSlabK);
}

// Stream-K grid: one CTA per SM (at most kMaxGrid), at least 8 slabs each.
int grid_of(long long total_slabs, int sms) {
    const long long by_work = std::max<long long>(1, total_slabs / 8);
    return int(std::min<long long>(std::min<long long>(sms > 0 ? sms : kMaxGrid, kMaxGrid), by_work));
}

// Workspace: [X_hi][X_lo (split)][2 partial tiles per stream-K CTA][row exponents].
GemmLayout gemm_layout(int64_t M, int64_t N, int64_t K, int prec, int sms) {
    GemmLayout L;
    L.part = align256(size_t(M) * K * 2);
    L.n_mtiles = mtiles_of(M);
    L.total_slabs = slabs_of(M, N, K);
    L.grid = grid_of(L.total_slabs, sms);
    L.partials = (prec == Q2_0_PREC_F16_SPLIT ? 2 : 1) * L.part;
    L.shifts = L.partials + size_t(2) * L.grid * kPartialBytes;
    L.total = L.shifts + align256(size_t(M) * 4);
    return L;
}

// A product's tensor maps and scalars: W [N][K/64*18] bytes, X_hi and X_lo fp16
// [M][K] (xl null for the hi-only precision).
bool make_gemm_job(GemmJob &J, const uint8_t *w, const __half *xh, const __half *xl, float *y,
                   const int *row_shift, int64_t M, int64_t N, int64_t K, long long slab0) {
    std::memset(&J, 0, sizeof(J));
    const uint64_t row_bytes = uint64_t(K / 64) * 18;
    if (!encode_tmap_2d(&J.w_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, row_bytes, uint64_t(N),
                        row_bytes, 144, kWT * kBM, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tmap_2d(&J.xh_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xh, uint64_t(K), uint64_t(M),
                        uint64_t(K) * 2, kSlabK, kBN, CU_TENSOR_MAP_SWIZZLE_128B))
        return false;
    if (xl && !encode_tmap_2d(&J.xl_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xl, uint64_t(K),
                              uint64_t(M), uint64_t(K) * 2, kSlabK, kBN,
                              CU_TENSOR_MAP_SWIZZLE_128B))
        return false;
    J.y = y;
    J.row_shift = row_shift;
    J.slab0 = slab0;
    J.M = int(M);
    J.N = int(N);
    J.K = int(K);
    J.n_mtiles = mtiles_of(M);
    return true;
}

template <typename XT>
cudaError_t launch_prep(const GemmPrepSet &ps, int n_x, int max_m, cudaStream_t s) {
    gemm_prep_kernel<XT><<<dim3(unsigned(max_m), unsigned(n_x)), kPrepThreads, 0, s>>>(ps);
    return cudaGetLastError();
}

// The tensor-core kernel and its stream-K reduction, each a programmatic
// dependent of the launch before it on the stream.
cudaError_t launch_gemm_pair(const GemmArgs &args, int grid, cudaStream_t s) {
    cudaError_t e = ensure_attr();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = gemm_smem_bytes();
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemm_tc_kernel, args);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(kReduceSlices, unsigned(grid));
    cfg.blockDim = dim3(kReduceThreads);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, gemm_reduce_kernel, args);
}

template <typename XT>
cudaError_t launch_generic(const uint8_t *w, const XT *x, float *y, int64_t N, int64_t K,
                           int64_t M, cudaStream_t s) {
    dim3 grid(unsigned((N + 31) / 32), unsigned((M + 7) / 8));
    gemm_generic_kernel<XT><<<grid, dim3(32, 8), 0, s>>>(w, x, y, int(M), int(N), int(K));
    return cudaGetLastError();
}

}  // namespace

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int prec) {
    // sized for the largest grid so the query needs no device
    return gemm_layout(M, N, K, prec, kMaxGrid).total;
}

int gemm_run(const uint8_t *w, const void *x, int xtype, float *y, int64_t N, int64_t K,
             int64_t M, int prec, void *ws, size_t ws_bytes, cudaStream_t s) {
    if (!tc_path_ok(w, x, K)) {
        const cudaError_t e =
            xtype == kXF16
                ? launch_generic(w, static_cast<const __half *>(x), y, N, K, M, s)
                : launch_generic(w, static_cast<const float *>(x), y, N, K, M, s);
        return cuda_status(e);
    }
    // F16 activations are exact fp16 operands: no lo part
    const int split = (prec == Q2_0_PREC_F16_SPLIT && xtype == kXF32) ? 1 : 0;
    if (ws_bytes < gemm_workspace_bytes(M, N, K, prec) || !ws) return Q2_0_EINVAL;
    unsigned long long *err = error_word_ptr();
    if (!err) return Q2_0_ECUDA;
    const GemmLayout L = gemm_layout(M, N, K, prec, sm_count());
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    __half *xh = reinterpret_cast<__half *>(wsb);
    __half *xl = split ? reinterpret_cast<__half *>(wsb + L.part) : nullptr;
    float *partials = reinterpret_cast<float *>(wsb + L.partials);
    int *row_shift = reinterpret_cast<int *>(wsb + L.shifts);
    GemmPrepSet ps;
    std::memset(&ps, 0, sizeof(ps));
    ps.x[0] = x;
    ps.xh[0] = xh;
    ps.xl[0] = xl;
    ps.row_shift[0] = row_shift;
    ps.M[0] = int(M);
    ps.K[0] = int(K);
    ps.split = split;
    const cudaError_t pe = xtype == kXF16 ? launch_prep<__half>(ps, 1, int(M), s)
                                          : launch_prep<float>(ps, 1, int(M), s);
    if (pe != cudaSuccess) return Q2_0_ECUDA;

    GemmArgs args;
    std::memset(&args, 0, sizeof(args));
    if (!make_gemm_job(args.single, w, xh, xl, y, row_shift, M, N, K, 0)) return Q2_0_ECUDA;
    args.jobs = nullptr;
    args.n_jobs = 1;
    args.split = split;
    args.total_slabs = L.total_slabs;
    args.partials = partials;
    args.err = err;
    return cuda_status(launch_gemm_pair(args, L.grid, s));
}

}  // namespace q2

// ---------------------------------------------------------------------------
// Grouped GEMM plans
// ---------------------------------------------------------------------------
struct q2_0_mm_plan {
    int device = 0;
    int grid = 0;
    int n_fast = 0;
    q2::GemmArgs args;                       // the tensor-core launch (jobs in device memory)
    q2::GemmJob *d_jobs = nullptr;
    uint8_t *d_mem = nullptr;                // X copies and row exponents, then partial tiles
    std::vector<q2::GemmPrepSet> prep;       // up to 8 distinct X per prep launch
    std::vector<int> prep_n, prep_max_m;
    std::vector<q2_0_mm_desc> generic;       // descriptors outside the TMA path
};

namespace q2 {

void mm_plan_destroy(q2_0_mm_plan *plan) {
    if (!plan) return;
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(plan->device);
    cudaFree(plan->d_jobs);
    cudaFree(plan->d_mem);
    cudaSetDevice(cur);
    delete plan;
}

int mm_plan_create(const q2_0_mm_desc *descs, int n, int prec, q2_0_mm_plan **out) {
    q2_0_mm_plan *P = new q2_0_mm_plan();
    cudaGetDevice(&P->device);
    std::memset(&P->args, 0, sizeof(P->args));
    P->args.err = error_word_ptr();
    if (!P->args.err) {
        delete P;
        return Q2_0_ECUDA;
    }
    const int split = prec == Q2_0_PREC_F16_SPLIT ? 1 : 0;
    std::vector<int> fast;
    for (int i = 0; i < n; ++i) {
        if (tc_path_ok(descs[i].w, descs[i].x, descs[i].K))
            fast.push_back(i);
        else
            P->generic.push_back(descs[i]);
    }
    P->n_fast = int(fast.size());
    if (P->n_fast == 0) {
        *out = P;
        return Q2_0_OK;
    }
    // Distinct activation matrices: products with the same (x, M, K) share the
    // prepass output. Memory per X: X_hi, X_lo (split), row exponents.
    struct XEnt {
        const float *x;
        int64_t M, K;
        size_t off_h, off_l, off_s;
    };
    std::vector<XEnt> xs;
    std::vector<int> x_of(P->n_fast);
    size_t total = 0;
    for (int j = 0; j < P->n_fast; ++j) {
        const q2_0_mm_desc &d = descs[fast[j]];
        int hit = -1;
        for (int e = 0; e < int(xs.size()); ++e)
            if (xs[e].x == d.x && xs[e].M == d.M && xs[e].K == d.K) hit = e;
        if (hit < 0) {
            XEnt e;
            e.x = d.x;
            e.M = d.M;
            e.K = d.K;
            const size_t part = align256(size_t(d.M) * d.K * 2);
            e.off_h = total;
            e.off_l = total + part;
            e.off_s = total + (split ? 2 : 1) * part;
            total = e.off_s + align256(size_t(d.M) * 4);
            hit = int(xs.size());
            xs.push_back(e);
        }
        x_of[j] = hit;
    }
    long long total_slabs = 0;
    std::vector<long long> slab0(P->n_fast);
    for (int j = 0; j < P->n_fast; ++j) {
        const q2_0_mm_desc &d = descs[fast[j]];
        slab0[j] = total_slabs;
        total_slabs += slabs_of(d.M, d.N, d.K);
    }
    P->grid = grid_of(total_slabs, sm_count());
    const size_t partials_off = total;
    total += size_t(2) * P->grid * kPartialBytes;
    int st = Q2_0_OK;
    if (cudaMalloc(&P->d_mem, total) != cudaSuccess ||
        cudaMalloc(&P->d_jobs, sizeof(GemmJob) * P->n_fast) != cudaSuccess)
        st = Q2_0_ECUDA;
    std::vector<GemmJob> jobs(P->n_fast);
    for (int j = 0; j < P->n_fast && st == Q2_0_OK; ++j) {
        const q2_0_mm_desc &d = descs[fast[j]];
        const XEnt &e = xs[x_of[j]];
        const __half *xh = reinterpret_cast<const __half *>(P->d_mem + e.off_h);
        const __half *xl = split ? reinterpret_cast<const __half *>(P->d_mem + e.off_l) : nullptr;
        const int *rs = reinterpret_cast<const int *>(P->d_mem + e.off_s);
        if (!make_gemm_job(jobs[j], static_cast<const uint8_t *>(d.w), xh, xl, d.y, rs, d.M, d.N,
                           d.K, slab0[j]))
            st = Q2_0_ECUDA;
    }
    if (st == Q2_0_OK && cudaMemcpy(P->d_jobs, jobs.data(), sizeof(GemmJob) * P->n_fast,
                                    cudaMemcpyHostToDevice) != cudaSuccess)
        st = Q2_0_ECUDA;
    if (st != Q2_0_OK) {
        mm_plan_destroy(P);
        return st;
    }
    for (int e0 = 0; e0 < int(xs.size()); e0 += kMaxPrepX) {
        GemmPrepSet ps;
        std::memset(&ps, 0, sizeof(ps));
        ps.split = split;
        int cnt = 0, max_m = 0;
        for (int e = e0; e < int(xs.size()) && cnt < kMaxPrepX; ++e, ++cnt) {
            ps.x[cnt] = xs[e].x;
            ps.xh[cnt] = reinterpret_cast<__half *>(P->d_mem + xs[e].off_h);
            ps.xl[cnt] = split ? reinterpret_cast<__half *>(P->d_mem + xs[e].off_l) : nullptr;
            ps.row_shift[cnt] = reinterpret_cast<int *>(P->d_mem + xs[e].off_s);
            ps.M[cnt] = int(xs[e].M);
            ps.K[cnt] = int(xs[e].K);
            max_m = std::max(max_m, int(xs[e].M));
        }
        P->prep.push_back(ps);
        P->prep_n.push_back(cnt);
        P->prep_max_m.push_back(max_m);
    }
    P->args.jobs = P->d_jobs;
    P->args.n_jobs = P->n_fast;
    P->args.split = split;
    P->args.total_slabs = total_slabs;
    P->args.partials = reinterpret_cast<float *>(P->d_mem + partials_off);
    *out = P;
    return Q2_0_OK;
}

int mm_plan_execute(const q2_0_mm_plan *P, cudaStream_t s) {
    for (size_t i = 0; i < P->prep.size(); ++i)
        if (launch_prep<float>(P->prep[i], P->prep_n[i], P->prep_max_m[i], s) != cudaSuccess)
            return Q2_0_ECUDA;
    if (P->n_fast > 0 && launch_gemm_pair(P->args, P->grid, s) != cudaSuccess) return Q2_0_ECUDA;
    for (const q2_0_mm_desc &d : P->generic)
        if (launch_generic(static_cast<const uint8_t *>(d.w), d.x, d.y, d.N, d.K, d.M, s) !=
            cudaSuccess)
            return Q2_0_ECUDA;
    return Q2_0_OK;
}

int mm_plan_launches(const q2_0_mm_plan *P) {
    return int(P->prep.size()) + (P->n_fast > 0 ? 2 : 0) + int(P->generic.size());
}

}  // namespace q2
