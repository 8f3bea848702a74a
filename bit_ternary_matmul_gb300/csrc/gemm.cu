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

struct GemmArgs {
    CUtensorMap w_map;   // uint8 [N][K/64*18], box {144, 256}
    CUtensorMap xh_map;  // fp16 [M][K], box {64, 128}, 128B swizzle
    CUtensorMap xl_map;
    float *y;
    int M, N, K;
    int split;  // 1: hi + lo, 0: hi only
    int n_units, n_mtiles;  // units = (N / 256 rounded up) x (M / 128 rounded up)
    long long total_slabs;  // n_units * K / 64: the stream-K iteration space
    float *partials;        // 2 slots per CTA of kBN x (kWT * kBM) fp32
    const int *row_shift;   // [M]: X row m entered the MMA as X * 2^row_shift[m]
    unsigned long long *err;
};

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
// never overflows fp16, and the lo parts of small elements stay above fp16's
// subnormal range down to 2^-29 of the row maximum. F16 rows are only scaled
// up (s >= 0), which keeps them exact. The scaling is exact and undone on the
// f32 result (y = acc * 2^-s). One CTA per row; X 16-byte aligned.
// ---------------------------------------------------------------------------
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
    const XT *__restrict__ x, __half *__restrict__ xh, __half *__restrict__ xl,
    int *__restrict__ row_shift, int M, int K, int split) {
    // The GEMM kernel that follows may start its prologue and weight loads now;
    // it waits for this grid before reading X.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int m = blockIdx.x;
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
    const int n_slabs = a.K / kSlabK;
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

    // Unit u -> (row pair, token tile) with the token tile fastest, so CTAs running
    // together share weight rows in L2.
    auto unit_coords = [&](int u, int &n0, int &m0) {
        n0 = (u / a.n_mtiles) * (kWT * kBM);
        m0 = (u % a.n_mtiles) * kBN;
    };

    if (warp == 0) {
        // ---------------------------- TMA producer ----------------------------
        if (lane == 0) {
            const uint32_t x_bytes = kXTileBytes * (a.split ? 2 : 1);
            int st = 0, wst = 0;
            uint32_t ph = 0, wph = 0;
            bool ok = true, prep_done = false;
            for (long long g = g_begin; g < g_end && ok;) {
                const int u = int(g / n_slabs), kb = int(g % n_slabs);
                const int ke = seg_end(n_slabs, kb, g_end - g);
                g += ke - kb;
                int n0, m0;
                unit_coords(u, n0, m0);
                for (int kk = kb; kk < ke; ++kk) {
                    if ((kk & 7) == 0 || kk == kb) {
                        if (!mbar_wait(&w_free[wst], wph ^ 1u, a.err, kTagGemm + 1)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&w_full[wst], kWBoxBytes);
                        tma_load_2d(w_s + wst * kWBoxBytes, &a.w_map, (kk >> 3) * 144, n0,
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
                    tma_load_2d(xh_s + st * kXTileBytes, &a.xh_map, kk * kSlabK, m0, &x_full[st]);
                    if (a.split)
                        tma_load_2d(xl_s + st * kXTileBytes, &a.xl_map, kk * kSlabK, m0,
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
            const int kb = int(g % n_slabs);
            const int ke = seg_end(n_slabs, kb, g_end - g);
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
            const int kb = int(g % n_slabs);
            const int ke = seg_end(n_slabs, kb, g_end - g);
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
            const int u = int(g / n_slabs), kb = int(g % n_slabs);
            const int ke = seg_end(n_slabs, kb, g_end - g);
            g += ke - kb;
            int n0, m0;
            unit_coords(u, n0, m0);
            if (!dead) {
                const bool got = mbar_wait(acc_full, uint32_t(nu & 1), a.err, kTagGemm + 8);
                dead = !__all_sync(0xffffffffu, got);
            }
            if (dead) continue;
            const bool whole = kb == 0 && ke == n_slabs;
            tc_fence_after();
            const int n = n0 + rloc;
            // partial tiles: slot 2c for a CTA's first segment, 2c + 1 for its last
            const long long ustart = (long long)u * n_slabs;
            float *mine = a.partials +
                          size_t(2 * blockIdx.x + (g_begin >= ustart ? 0 : 1)) * (kPartialBytes / 4);
#pragma unroll 1
            for (int cb = 0; cb < kBN; cb += 32) {
                uint32_t v[32];
                tmem_ld32(tmem_base + lane_addr + kAccCol + t * kBN + cb, v);
                if (whole) {
                    // the 32 tokens' row exponents: one load per lane, shared by shuffles
                    const int sh = m0 + cb + lane < a.M ? a.row_shift[m0 + cb + lane] : 0;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int shj = __shfl_sync(0xffffffffu, sh, j);
                        const int m = m0 + cb + j;
                        if (n < a.N && m < a.M)
                            a.y[size_t(m) * a.N + n] = mul_pow2(__uint_as_float(v[j]), -shj);
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
    const float *__restrict__ partials, const int *__restrict__ row_shift, float *__restrict__ y,
    int M, int N, int n_mtiles, int n_slabs, long long total_slabs) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int G = int(gridDim.y), c = int(blockIdx.y);
    const long long gb = sk_begin(c, total_slabs, G);
    const int u = int(gb / n_slabs);
    const long long ustart = (long long)u * n_slabs;
    if (gb == ustart) return;  // c begins its first unit: not a split unit's finisher
    const int c_first = sk_owner(ustart, total_slabs, G);
    const int c_last = sk_owner(ustart + n_slabs - 1, total_slabs, G);
    if (c != c_last) return;
    const int n0 = (u / n_mtiles) * (kWT * kBM);
    const int m0 = (u % n_mtiles) * kBN;
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
    int n_units, n_mtiles, grid;
    long long total_slabs;
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Workspace: [X_hi][X_lo (split)][2 partial tiles per stream-K CTA][row exponents].
// The grid is at most kMaxGrid CTAs, at least 8 slabs each.
GemmLayout gemm_layout(int64_t M, int64_t N, int64_t K, int prec, int sms) {
    GemmLayout L;
    L.part = align256(size_t(M) * K * 2);
    L.n_mtiles = int((M + kBN - 1) / kBN);
    L.n_units = int((N + kWT * kBM - 1) / (kWT * kBM)) * L.n_mtiles;
    L.total_slabs = (long long)L.n_units * (K / kSlabK);
    const long long by_work = std::max<long long>(1, L.total_slabs / 8);
    L.grid = int(std::min<long long>(std::min<long long>(sms > 0 ? sms : kMaxGrid, kMaxGrid), by_work));
    L.partials = (prec == Q2_0_PREC_F16_SPLIT ? 2 : 1) * L.part;
    L.shifts = L.partials + size_t(2) * L.grid * kPartialBytes;
    L.total = L.shifts + align256(size_t(M) * 4);
    return L;
}

}  // namespace

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int prec) {
    // sized for the largest grid so the query needs no device
    return gemm_layout(M, N, K, prec, kMaxGrid).total;
}

int gemm_run(const uint8_t *w, const void *x, int xtype, float *y, int64_t N, int64_t K,
             int64_t M, int prec, void *ws, size_t ws_bytes, cudaStream_t s) {
    if (!tc_path_ok(w, x, K)) {
        dim3 grid(unsigned((N + 31) / 32), unsigned((M + 7) / 8));
        if (xtype == kXF16)
            gemm_generic_kernel<__half><<<grid, dim3(32, 8), 0, s>>>(
                w, static_cast<const __half *>(x), y, int(M), int(N), int(K));
        else
            gemm_generic_kernel<float><<<grid, dim3(32, 8), 0, s>>>(
                w, static_cast<const float *>(x), y, int(M), int(N), int(K));
        return cuda_status(cudaGetLastError());
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
    if (xtype == kXF16)
        gemm_prep_kernel<__half><<<unsigned(M), kPrepThreads, 0, s>>>(
            static_cast<const __half *>(x), xh, xl, row_shift, int(M), int(K), split);
    else
        gemm_prep_kernel<float><<<unsigned(M), kPrepThreads, 0, s>>>(
            static_cast<const float *>(x), xh, xl, row_shift, int(M), int(K), split);
    if (cudaGetLastError() != cudaSuccess) return Q2_0_ECUDA;

    GemmArgs args;
    std::memset(&args, 0, sizeof(args));
    const uint64_t row_bytes = uint64_t(K / 64) * 18;
    if (!encode_tmap_2d(&args.w_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, row_bytes, uint64_t(N),
                        row_bytes, 144, kWT * kBM, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tmap_2d(&args.xh_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xh, uint64_t(K), uint64_t(M),
                        uint64_t(K) * 2, kSlabK, kBN, CU_TENSOR_MAP_SWIZZLE_128B))
        return Q2_0_ECUDA;
    if (split && !encode_tmap_2d(&args.xl_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xl, uint64_t(K),
                                 uint64_t(M), uint64_t(K) * 2, kSlabK, kBN,
                                 CU_TENSOR_MAP_SWIZZLE_128B))
        return Q2_0_ECUDA;
    args.y = y;
    args.M = int(M);
    args.N = int(N);
    args.K = int(K);
    args.split = split;
    args.err = err;
    args.n_mtiles = L.n_mtiles;
    args.n_units = L.n_units;
    args.total_slabs = L.total_slabs;
    args.partials = partials;
    args.row_shift = row_shift;
    if (ensure_attr() != cudaSuccess) return Q2_0_ECUDA;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(L.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = gemm_smem_bytes();
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, gemm_tc_kernel, args) != cudaSuccess) return Q2_0_ECUDA;
    // the stream-K reduction, as a programmatic dependent of the GEMM
    cfg.gridDim = dim3(kReduceSlices, L.grid);
    cfg.blockDim = dim3(kReduceThreads);
    cfg.dynamicSmemBytes = 0;
    if (cudaLaunchKernelEx(&cfg, gemm_reduce_kernel, static_cast<const float *>(partials),
                           static_cast<const int *>(row_shift), y, int(M), int(N), L.n_mtiles,
                           int(K / kSlabK), L.total_slabs) !=
        cudaSuccess)
        return Q2_0_ECUDA;
    return cuda_status(cudaGetLastError());
}

}  // namespace q2
