// Q2_0 prefill GEMM on the 5th-generation tensor cores (tcgen05, sm_103a):
//   Y[m][n] = sum_k W[n][k] X[m][k]   (M tokens, N weight rows).
//
// Source: "WebGPU: add Q2_0 support" (bisque.today write-up of llama.cpp
// PR 30914), shader paragraph — the tiled matrix multiply unpacks each thread's
// 16 codes into shared memory as half precision before the product. Here the
// unpacked operand is (q - 1) * d in fp16, which is exact for every code and
// every fp16 d with |2d| <= 65504, so the scale needs no separate pass.
//
// Data flow of one CTA (a 128-row x BN-token output tile, K in 64-wide slabs,
// one Q2_0 block per row per slab):
//   warp 0  TMA producer: packed W box (128 rows x 144 B = 8 slabs) into a
//           2-deep ring; per slab the X_hi (and X_lo) tile [BN x 64] fp16 with
//           128-byte swizzle into a kStages-deep ring.
//   warp 1  TMEM allocation and the MMA issuer (one thread): 4 K=16 steps per
//           slab, for hi and lo, tcgen05.mma kind::f16 M=128 N=BN, fp32
//           accumulator in TMEM; tcgen05.commit frees the slab's ring slot.
//   warps 2-5  expansion: thread r decodes row r's block of the slab into 64
//           fp16 and stores them into the A tile (K-major, 128-byte swizzle);
//           then the epilogue: tcgen05.ld of the accumulator, F32 stores.
//
// K order inside a 16-element word group is permuted to (0,8,1,9,...,7,15) on
// both operands, so that one mask of a code word yields the fp16 pair
// (element t, element t+8); the prepass writes X in that order.
//
// Activations: the prepass writes hi = fp16(x) and lo = fp16(x - hi); the
// split path issues both products into the same accumulator.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "q2_0_device.cuh"
#include "q2_0_internal.h"

namespace q2 {

namespace {

constexpr int kBM = 128;            // weight rows per tile (MMA M)
constexpr int kBN = 128;            // tokens per tile (MMA N)
constexpr int kSlabK = 64;          // one Q2_0 block
constexpr int kStages = 3;          // X / A ring depth
constexpr int kWStages = 2;         // packed-W ring depth (8 slabs each)
constexpr int kThreads = 192;       // 6 warps
constexpr int kATileBytes = kBM * kSlabK * 2;     // 16 KB
constexpr int kXTileBytes = kBN * kSlabK * 2;     // 16 KB per part
constexpr int kWBoxBytes = kBM * 144;             // 18 KB
constexpr int kTmemCols = kBN;                    // fp32 accumulator columns

constexpr int kTagGemm = 200;

struct GemmArgs {
    CUtensorMap w_map;   // uint8 [N][K/64*18], box {144, 128}
    CUtensorMap xh_map;  // fp16 [M][K], box {64, 128}, 128B swizzle
    CUtensorMap xl_map;
    float *y;
    int M, N, K;
    int split;  // 1: hi + lo, 0: hi only
    unsigned long long *err;
};

// ---------------------------------------------------------------------------
// tcgen05 / TMEM wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(smem_dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (SBO), version 1, leading-byte offset unused (1).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3FFFu);
    d |= uint64_t(1) << 16;
    d |= uint64_t(1024 >> 4) << 32;
    d |= uint64_t(1) << 46;
    d |= uint64_t(2) << 61;
    return d;
}

// Instruction descriptor, kind::f16: D f32, A and B f16, both K-major, N, M.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n) {
    return (1u << 4) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

// ---------------------------------------------------------------------------
// Prepass: X f32 [M][K] -> fp16 hi (and lo) [M][K] in the permuted K order.
// One thread per 16-element word group.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gemm_prep_kernel(const float *__restrict__ x,
                                                        __half *__restrict__ xh,
                                                        __half *__restrict__ xl, int64_t groups,
                                                        int split) {
    for (int64_t gidx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; gidx < groups;
         gidx += int64_t(gridDim.x) * blockDim.x) {
        const float4 *src = reinterpret_cast<const float4 *>(x + gidx * 16);
        float v[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 f = src[q];
            v[4 * q] = f.x;
            v[4 * q + 1] = f.y;
            v[4 * q + 2] = f.z;
            v[4 * q + 3] = f.w;
        }
        uint32_t hw[8], lw[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const __half h0 = __float2half_rn(v[t]);
            const __half h1 = __float2half_rn(v[t + 8]);
            hw[t] = uint32_t(__half_as_ushort(h0)) | (uint32_t(__half_as_ushort(h1)) << 16);
            const __half l0 = __float2half_rn(v[t] - __half2float(h0));
            const __half l1 = __float2half_rn(v[t + 8] - __half2float(h1));
            lw[t] = uint32_t(__half_as_ushort(l0)) | (uint32_t(__half_as_ushort(l1)) << 16);
        }
        uint4 *dh = reinterpret_cast<uint4 *>(xh + gidx * 16);
        dh[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        dh[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
        if (split) {
            uint4 *dl = reinterpret_cast<uint4 *>(xl + gidx * 16);
            dl[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            dl[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
        }
    }
}

// ---------------------------------------------------------------------------
// tcgen05 GEMM kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled tiles
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *xh_s = smem;                                   // kStages x 16 KB
    uint8_t *xl_s = xh_s + kStages * kXTileBytes;           // kStages x 16 KB
    uint8_t *a_s = xl_s + kStages * kXTileBytes;            // kStages x 16 KB
    uint8_t *w_s = a_s + kStages * kATileBytes;             // kWStages x 18 KB
    uint64_t *bars = reinterpret_cast<uint64_t *>(w_s + kWStages * kWBoxBytes);
    uint64_t *x_full = bars;                 // [kStages]
    uint64_t *a_full = x_full + kStages;     // [kStages]
    uint64_t *slot_free = a_full + kStages;  // [kStages]
    uint64_t *w_full = slot_free + kStages;  // [kWStages]
    uint64_t *w_free = w_full + kWStages;    // [kWStages]
    uint64_t *acc_full = w_free + kWStages;  // [1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * kBM;
    const int m0 = blockIdx.y * kBN;
    const int n_slabs = a.K / kSlabK;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&a_full[i], 128);
            mbar_init(&slot_free[i], 1);
        }
        for (int i = 0; i < kWStages; ++i) {
            mbar_init(&w_full[i], 1);
            mbar_init(&w_free[i], 128);
        }
        mbar_init(acc_full, 1);
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

    if (warp == 0) {
        // ---------------------------- TMA producer ----------------------------
        if (lane == 0) {
            const uint32_t x_bytes = kXTileBytes * (a.split ? 2 : 1);
            int st = 0, wst = 0;
            uint32_t ph = 0, wph = 0;
            for (int kk = 0; kk < n_slabs; ++kk) {
                if ((kk & 7) == 0) {
                    if (!mbar_wait(&w_free[wst], wph ^ 1u, a.err, kTagGemm + 1)) break;
                    mbar_arrive_expect_tx(&w_full[wst], kWBoxBytes);
                    tma_load_2d(w_s + wst * kWBoxBytes, &a.w_map, (kk >> 3) * 144, n0,
                                &w_full[wst]);
                }
                if (!mbar_wait(&slot_free[st], ph ^ 1u, a.err, kTagGemm + 2)) break;
                mbar_arrive_expect_tx(&x_full[st], x_bytes);
                tma_load_2d(xh_s + st * kXTileBytes, &a.xh_map, kk * kSlabK, m0, &x_full[st]);
                if (a.split)
                    tma_load_2d(xl_s + st * kXTileBytes, &a.xl_map, kk * kSlabK, m0, &x_full[st]);
                if (++st == kStages) {
                    st = 0;
                    ph ^= 1u;
                }
                if ((kk & 7) == 7 || kk == n_slabs - 1) {
                    if (++wst == kWStages) {
                        wst = 0;
                        wph ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ----------------------------- MMA issuer -----------------------------
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(kBM, kBN);
            int st = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int kk = 0; kk < n_slabs && ok; ++kk) {
                if (!mbar_wait(&x_full[st], ph, a.err, kTagGemm + 3) ||
                    !mbar_wait(&a_full[st], ph, a.err, kTagGemm + 4)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = smem_addr(a_s + st * kATileBytes);
                const uint32_t h_addr = smem_addr(xh_s + st * kXTileBytes);
                const uint32_t l_addr = smem_addr(xl_s + st * kXTileBytes);
#pragma unroll
                for (int ks = 0; ks < kSlabK / 16; ++ks) {
                    const uint64_t ad = sw128_desc(a_addr + ks * 32);
                    tc_mma_f16(tmem_base, ad, sw128_desc(h_addr + ks * 32), idesc,
                               (kk > 0 || ks > 0) ? 1u : 0u);
                    if (a.split) tc_mma_f16(tmem_base, ad, sw128_desc(l_addr + ks * 32), idesc, 1u);
                }
                tc_commit(&slot_free[st]);
                if (++st == kStages) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            if (ok) tc_commit(acc_full);
            else *(volatile int *)abort_flag = 1;
        }
    } else {
        // ------------------------ expansion, then epilogue ------------------------
        const int r = threadIdx.x - 64;  // 0..127: tile row
        int st = 0, wst = 0;
        uint32_t ph = 0, wph = 0;
        bool ok = true;
        for (int kk = 0; kk < n_slabs; ++kk) {
            bool got = true;
            if ((kk & 7) == 0) got = mbar_wait(&w_full[wst], wph, a.err, kTagGemm + 5);
            got = got && mbar_wait(&slot_free[st], ph ^ 1u, a.err, kTagGemm + 6);
            if (!__all_sync(0xffffffffu, got)) {  // warp-uniform decision
                ok = false;
                break;
            }
            // row r's block (kk & 7) in the packed box: 18 bytes at r*144 + 18*(kk&7)
            const int bb = kk & 7;
            const uint8_t *rowp = w_s + wst * kWBoxBytes + r * 144;
            const int off = 18 * bb;
            const uint32_t *u = reinterpret_cast<const uint32_t *>(rowp + (off & ~3));
            const uint32_t u0 = u[0], u1 = u[1], u2 = u[2], u3 = u[3], u4 = u[4];
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
            const __half2 k1025 = __floats2half2_rn(1025.0f, 1025.0f);
            uint8_t *arow = a_s + st * kATileBytes + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {  // 16-byte chunk j = k-slots 8j..8j+7
                const uint32_t word = wd[j >> 1];
                uint32_t h[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int t = 4 * (j & 1) + q;  // pair (element t, element t+8)
                    const uint32_t bits = ((word >> (2 * t)) & 0x00030003u) | 0x64006400u;
                    __half2 v = *reinterpret_cast<const __half2 *>(&bits);
                    v = __hmul2(__hsub2(v, k1025), d2);
                    h[q] = *reinterpret_cast<uint32_t *>(&v);
                }
                *reinterpret_cast<uint4 *>(arow + ((j ^ (r & 7)) << 4)) =
                    make_uint4(h[0], h[1], h[2], h[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&a_full[st]);
            if (bb == 7 || kk == n_slabs - 1) {
                mbar_arrive(&w_free[wst]);
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
        // epilogue: wait for the accumulator, read TMEM lanes of this warp's quarter
        const bool acc_ready = ok && mbar_wait(acc_full, 0, a.err, kTagGemm + 7);
        if (__all_sync(0xffffffffu, acc_ready)) {
            tc_fence_after();
            const int quarter = warp & 3;
            const int n = n0 + quarter * 32 + lane;
            const uint32_t lane_base = tmem_base + (uint32_t(quarter * 32) << 16);
#pragma unroll 1
            for (int cb = 0; cb < kBN; cb += 32) {
                uint32_t v[32];
                tmem_ld32(lane_base + cb, v);
                if (n < a.N) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int m = m0 + cb + j;
                        if (m < a.M) a.y[size_t(m) * a.N + n] = __uint_as_float(v[j]);
                    }
                }
            }
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
// Generic GEMM (any K % 64 == 0, any alignment): CUDA cores, f32.
// Block of 32 x 8 threads computes Y[m0..m0+8) x [n0..n0+32).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gemm_generic_kernel(const uint8_t *__restrict__ w,
                                                           const float *__restrict__ x,
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
            const float *xe = x + size_t(m) * K + b * 64 + wi * 16;
#pragma unroll
            for (int i = 0; i < 16; ++i) s = fmaf(float(int((word >> (2 * i)) & 3u) - 1), xe[i], s);
        }
        acc = fmaf(d, s, acc);
    }
    y[size_t(m) * N + n] = acc;
}

constexpr int gemm_smem_bytes() {
    return 1024 /* alignment slack */ + kStages * (2 * kXTileBytes + kATileBytes) +
           kWStages * kWBoxBytes + 8 * (3 * kStages + 2 * kWStages + 1) + 16;
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

bool tc_path_ok(const void *w, const float *x, int64_t K) {
    return K % 512 == 0 && (reinterpret_cast<uintptr_t>(w) & 15u) == 0 &&
           (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
}

}  // namespace

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int prec) {
    (void)N;
    const size_t part = (size_t(M) * K * 2 + 255) & ~size_t(255);
    return prec == Q2_0_PREC_F16_SPLIT ? 2 * part : part;
}

int gemm_run(const uint8_t *w, const float *x, float *y, int64_t N, int64_t K, int64_t M, int prec,
             void *ws, size_t ws_bytes, cudaStream_t s) {
    if (!tc_path_ok(w, x, K)) {
        dim3 grid(unsigned((N + 31) / 32), unsigned((M + 7) / 8));
        gemm_generic_kernel<<<grid, dim3(32, 8), 0, s>>>(w, x, y, int(M), int(N), int(K));
        return cuda_status(cudaGetLastError());
    }
    const int split = prec == Q2_0_PREC_F16_SPLIT ? 1 : 0;
    if (ws_bytes < gemm_workspace_bytes(M, N, K, prec) || !ws) return Q2_0_EINVAL;
    unsigned long long *err = error_word_ptr();
    if (!err) return Q2_0_ECUDA;
    __half *xh = static_cast<__half *>(ws);
    const size_t part = (size_t(M) * K * 2 + 255) & ~size_t(255);
    __half *xl = split ? reinterpret_cast<__half *>(static_cast<uint8_t *>(ws) + part) : nullptr;
    const int64_t groups = M * K / 16;
    int64_t pgrid = std::min<int64_t>((groups + 255) / 256, int64_t(sm_count()) * 8);
    gemm_prep_kernel<<<unsigned(std::max<int64_t>(pgrid, 1)), 256, 0, s>>>(x, xh, xl, groups, split);
    if (cudaGetLastError() != cudaSuccess) return Q2_0_ECUDA;

    GemmArgs args;
    std::memset(&args, 0, sizeof(args));
    const uint64_t row_bytes = uint64_t(K / 64) * 18;
    if (!encode_tmap_2d(&args.w_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, row_bytes, uint64_t(N),
                        row_bytes, 144, kBM, CU_TENSOR_MAP_SWIZZLE_NONE) ||
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
    if (ensure_attr() != cudaSuccess) return Q2_0_ECUDA;
    dim3 grid(unsigned((N + kBM - 1) / kBM), unsigned((M + kBN - 1) / kBN));
    gemm_tc_kernel<<<grid, kThreads, gemm_smem_bytes(), s>>>(args);
    return cuda_status(cudaGetLastError());
}

}  // namespace q2
