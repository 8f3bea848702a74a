// Q2_0 decode mat-vec: Y[c][n] = sum_k W[n][k] X[c][k] for ncols = 1..8.
//
// Source: "WebGPU: add Q2_0 support" (bisque.today write-up of llama.cpp
// PR 30914), mat-vec kernel excerpt: four threads share a 64-weight block, each
// owning one 32-bit word of 16 codes; codes are shifted out of the word two
// bits at a time, (q - 1) multiplies the activation, and the scale d is applied
// once per block sum. This file keeps the per-word decode and the single
// application of d per block, and moves the multiply-accumulate onto the
// 5th-generation tensor cores (tcgen05.mma, accumulators in tensor memory):
//
//   ncols 1, 2    mv_t4_kernel: codes as packed e2m1 (q / 2, two logic ops per
//                 16 weights), activations as 16 block-scaled e2m1 pieces per
//                 column, kind::mxf4 with K = 64 = one block per MMA; the "- 1"
//                 is an exact per-block correction (see the fp4 section);
//   ncols 3..8    mv_s8_kernel<NC>: codes as signed e4m3 (q - 1, one byte-permute
//                 lookup per 4 weights), activations as 5 block-scaled e4m3
//                 pieces per column, kind::f8f6f4 with K = 32;
//   other shapes  mv_generic_kernel: CUDA cores, f32 (K % 512 != 0 or W not
//                 16-byte aligned).
//
// Both tensor-core kernels are persistent, one CTA per SM of 12 warps (16 with
// two epilogue warps per lane quarter: the fp4 kernel at two columns, the e4m3
// kernel), over 128-row tiles of one matrix or of a plan's many matrices; a
// pipeline stage is
// one 2-D TMA box of 128 rows x 144 bytes (8 blocks = 512 weights per row) plus
// the stage's activation image (bulk copy), in an 8-deep shared-memory ring.
// Warps 0 and 2 stream the even and odd stages, warps 3 and 1 issue the MMAs
// of the even and odd stages, warps 4-7 expand the codes of a stage into tensor memory (one warp
// per 32-lane quarter: a warp reaches only the lanes of its quarter) and warps
// 8-11 combine the accumulators, apply d and write y. Activations are F32 or
// F16 (the prep kernels and the generic kernel read either; F16 values are
// converted exactly).
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

constexpr int kChunkBlocks = 8;                  // blocks per stage
constexpr int kChunkBytes = kChunkBlocks * 18;   // 144 bytes of a row per stage
constexpr int kTcRows = 128;                     // rows per tile (MMA M)
constexpr int kRawBytes = kTcRows * kChunkBytes; // 18432: one stage's TMA box
constexpr int kPrepHeader = 1024;                // activation images start 1024-aligned
constexpr int kPrepThreads = 128;
constexpr int kTcThreads = 12 * 32;
// Warp roles of both tensor-core kernels (see the file comment). Two producers
// (warps 0 and 2) take the even and odd stages: issuing a stage's copies slows
// the other warps of the producer's SM sub-partition, and the stage period is
// set by the slowest expansion warp, so the issue work is split over two
// sub-partitions.
constexpr int kProdWarp = 2;
constexpr int kProdWarp2 = 0;
constexpr int kMmaWarp = 3;    // even stages; allocates TMEM
constexpr int kMmaWarp2 = 1;   // odd stages
constexpr int kExpWarp0 = 4;   // warps 4-7
constexpr int kExpWarps = 4;
constexpr int kEpiWarp0 = 8;   // warps 8-11
constexpr int kEpiWarps = 4;
// Dynamic shared memory a CTA may use: the opt-in maximum less the static part.
constexpr int kSmemOptIn = 232448;

struct MvPrepJob {
    const void *x;   // [ncols][K], F32 or F16 (the prep kernel's template argument)
    uint8_t *prep;   // prepared activation images
    int K;
    // fp4 prep only, launched without a job list: grid row j prepares the vector
    // at x + j * x_stride into prep + j * prep_stride (bytes)
    long long x_stride;
    long long prep_stride;
};

struct MvJob {  // 64-byte aligned through its CUtensorMap member
    CUtensorMap tmap;  // W as uint8 [N][K/64*18], box {144, 128}
    const uint8_t *prep;
    float *y;
    int N;
    int nb;        // K / 64
    int n_chunks;  // K / 512
    int n_tiles;   // ceil(N / 128)
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

// A plan CTA's share of the schedule in one record, so that a CTA learns its
// work and its first item with a single load.
struct MvFirst {
    int item_base;  // the CTA's first entry in items
    int n_items;
    int n_stages;   // stages (512-column chunks) of its items
    int job0;       // its first item: job, tile, and the job's fields the producer
    int tile0;      // needs, so that the first copies wait on no further load
    int n_chunks0;
    int n0;
    const uint8_t *prep0;
    float *y0;
};

struct MvParams {
    const MvJob *jobs;        // nullptr: the single job passed by value
    const MvItem *items;      // per-CTA work lists (schedule), when jobs != nullptr
    const MvFirst *first;     // [gridDim.x] each CTA's share of the schedule, plan only
    int ncols;
    unsigned long long *err;
    MvMoe moe;
    int layout;               // fp4 kernel only: kLayBlocks, kLaySplit or kLayG128
    // fp4 kernel, test hook (q2_0_test_inject_stall): when stall_stage > 0 the
    // producers stop before stage stall_stage - 1, so the consumers' waits on it
    // run out after wait_ns (0: the default limit)
    int stall_stage;
    unsigned long long wait_ns;
};

// Where the epilogue writes the tile a ring stage belongs to; the producer fills
// one per slot before the slot's barrier arrive.
struct StageMeta {
    float *y;              // nullptr: the tile is not written (an expert id out of range)
    int row0;              // first row of the tile
    int n_rows;            // rows of the matrix (also the column stride of y)
    int flags;             // kLastOfTile
    int pad;
};
constexpr int kLastOfTile = 2;

// v * 2^e for |e| <= 252 with two exact power-of-two factors (each a normal f32).
__device__ __forceinline__ float mul_pow2(float v, int e) {
    const int e1 = e / 2, e2 = e - e1;
    return v * __int_as_float((127 + e1) << 23) * __int_as_float((127 + e2) << 23);
}

// 2^k as a float for k <= 127: subnormal below -126, zero below -149.
__device__ __forceinline__ float pow2f(int k) {
    return k >= -126 ? __int_as_float((127 + k) << 23)
                     : k >= -149 ? __int_as_float(1 << (149 + k)) : 0.0f;
}

// Eight f32 values rounded to e2m1 (round to nearest, ties to even; the
// values here never reach the saturation bound 6), packed as nibbles: value i
// in bits 4i .. 4i + 3.
__device__ __forceinline__ uint32_t e2m1x8_rn(const float (&w)[8]) {
    uint32_t r;
    asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
        "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
        : "=r"(r)
        : "f"(w[0]), "f"(w[1]), "f"(w[2]), "f"(w[3]), "f"(w[4]), "f"(w[5]), "f"(w[6]), "f"(w[7]));
    return r;
}

// The e2m1 values of nibbles 2k (lo) and 2k + 1 (hi) of a packed word, exactly.
__device__ __forceinline__ void e2m1x2_values(uint32_t word, int k, float &lo, float &hi) {
    uint32_t h2;
    asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
        "mov.b32 {q0, q1, q2, q3}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, q0;\n\t}"
        : "=r"(h2)
        : "r"(word >> (8 * k)));
    asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
}

// Activation element load: F32 as is, F16 (IEEE binary16) converted exactly.
__device__ __forceinline__ float ld_x(const float *p) { return *p; }
__device__ __forceinline__ float ld_x(const __half *p) { return __half2float(*p); }

// fp16 scale at a shared-memory address, as f32.
__device__ __forceinline__ float lds_half_as_float(const uint8_t *p) {
    return __half2float(*reinterpret_cast<const __half *>(p));
}

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Byte offset of element (row n, K byte kc) of one stage's activation image of
// `rows` rows: K-major rows of 128 bytes in atoms of 8 rows (1024 B); the
// 16-byte chunk index is XOR-ed with the row within the atom (128-byte
// swizzle); the K extent is split into atom columns of 128 bytes, each holding
// all rows (rows * 128 bytes).
__host__ __device__ constexpr int img_offset(int rows, int n, int kc) {
    return (kc >> 7) * (rows * 128) + (n >> 3) * 1024 + (n & 7) * 128 +
           ((((kc & 127) >> 4) ^ (n & 7)) << 4) + (kc & 15);
}

// The 18 bytes of block 4G + bi of a row's stage slice as four code words,
// from the 72-byte half G loaded as u[0..17]: even blocks start 2 bytes into a
// 4-byte word (d first), so their words straddle two aligned words.
__device__ __forceinline__ uint32_t block_word(const uint32_t (&u)[18], int bi, int c) {
    if (bi == 0) return __byte_perm(u[c], u[c + 1], 0x5432);
    if (bi == 1) return u[5 + c];
    if (bi == 2) return __byte_perm(u[9 + c], u[10 + c], 0x5432);
    return u[14 + c];
}

// ---------------------------------------------------------------------------
// tcgen05 mat-vec on packed fp4 (ncols 1 and 2)
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
constexpr int kT4N = 16;                               // MMA N: one B row per piece
constexpr int kT4Stages = 8;
// per block of a stage: float {2^(e - 1), H, M, L}
constexpr int kT4BlockRec = 4;
constexpr int kT4BetaBytes = kChunkBlocks * kT4BlockRec * 4;  // 128
constexpr int kT4ABufs = 3;
constexpr int kT4ACol = 256;                           // A buffers at 256 + 64 i
constexpr int kT4ScaleCol = 448;  // scales A 448..451, B 452..455 (448..463 all hold 1.0)
// mbarriers: full / empty per stage, a_full / a_empty per A buffer, d_full /
// d_empty per D buffer, a drain per MMA issuer, and the two-column kernel's
// tile-end hand-offs (4 + 4, placed in every layout)
constexpr int kT4Barriers = 2 * kT4Stages + 2 * kT4ABufs + 2 * 2 + 2 + 8;
// a stage's activation data (image, then block records) is one bulk copy; in
// shared memory its slots stay 1024-aligned for the swizzled image
constexpr int kT4ActSlot = 5120;
constexpr int kT4Smem = 1024 /* alignment slack */ + kT4Stages * (kT4ActSlot + kRawBytes) +
                        kT4Barriers * 8;
static_assert(kT4Pieces == kT4N, "one B row per piece");
constexpr int kTagT4Full = 111;
constexpr int kTagT4Empty = 112;
constexpr int kTagT4AFull = 113;
constexpr int kTagT4DFull = 114;
constexpr int kTagT4DEmpty = 115;
constexpr int kTagT4Pair = 116;

// Weight layouts the fp4 kernel streams: 18-byte blocks of 64 weights, the
// split layout (codes and scales in separate arrays), and group-128 (34-byte
// blocks of 128 weights under one scale). A group-128 stage is 1024 weights of
// a row: one 272-byte box per row (eight blocks), two 64-column A buffers, and
// eight accumulator regions, one per 128-weight block, each the sum of two
// K = 64 MMAs; the activations are scaled per 128 elements to match, so every
// region is still exact. Every other quantity is the 64-weight layout's.
constexpr int kLayBlocks = 0;
constexpr int kLaySplit = 1;
constexpr int kLayG128 = 2;
constexpr int kG128Bytes = 34;
constexpr int kG128RowBytes = kChunkBlocks * kG128Bytes;  // 272

// NC: activation columns (1, or 2 for the 64-weight layout). Column j's pieces
// are B rows 16 j .. 16 j + 15, and each region has one record per column.
template <int L, int NC = 1>
struct T4Lay {
    static constexpr int kStageK = L == kLayG128 ? 1024 : 512;  // weights of a row per stage
    static constexpr int kAPer = kStageK / 512;                 // 64-column A buffers per stage
    static constexpr int kRaw = L == kLayG128 ? kTcRows * kG128RowBytes : kRawBytes;
    static constexpr int kN = kT4N * NC;                        // MMA N: B rows
    static constexpr int kImg = kN * kStageK / 2;               // e2m1 B image of a stage
    static constexpr int kAct = kImg + kT4BetaBytes * NC;       // image, then the region records
    static constexpr int kActSlot = (kAct + 1023) / 1024 * 1024;
    static constexpr int kStages = L == kLayG128 ? 4 : kT4Stages;
    // as kT4Barriers (the two-column hand-offs are counted for every layout)
    static constexpr int kBarriers = 2 * kStages + 2 * kT4ABufs + 2 * 2 + 2 + 8;
    static constexpr int kSmem = 1024 /* alignment slack */ + kStages * (kActSlot + kRaw) +
                                 kBarriers * 8;
    static constexpr int kEpi = kEpiWarps * NC;   // epilogue warps
    static constexpr int kThreads = kTcThreads + (NC - 1) * kEpiWarps * 32;
};
static_assert(T4Lay<kLayBlocks>::kActSlot == kT4ActSlot && T4Lay<kLayBlocks>::kSmem == kT4Smem,
              "the 64-weight layout keeps its stage geometry");
static_assert(T4Lay<kLayG128>::kStages % 2 == 0 && T4Lay<kLayG128>::kSmem <= kSmemOptIn,
              "group-128 ring: even depth (two producers), within the shared-memory limit");
static_assert(T4Lay<kLayBlocks, 2>::kSmem <= kSmemOptIn - 4096,
              "two-column ring (and the static hand-off buffer) within the shared-memory limit");
static_assert(T4Lay<kLayBlocks>::kThreads == kTcThreads && T4Lay<kLaySplit>::kThreads == kTcThreads &&
                  T4Lay<kLayG128>::kThreads == kTcThreads && T4Lay<kLayBlocks, 2>::kThreads == 16 * 32,
              "fp4 kernel block sizes: 12 warps, 16 with two epilogue warps per lane quarter");

size_t t4_prep_bytes(int64_t K, int ncols = 1) {
    const size_t n_chunks = size_t(K / 512);
    size_t b = kPrepHeader +
               n_chunks * (ncols == 2 ? T4Lay<kLayBlocks, 2>::kAct : T4Lay<kLayBlocks>::kAct);
    return (b + 255) & ~size_t(255);
}

size_t g4_prep_bytes(int64_t K) {
    const size_t n_chunks = size_t(K / 1024);
    size_t b = kPrepHeader + n_chunks * T4Lay<kLayG128>::kAct;
    return (b + 255) & ~size_t(255);
}

// kind::mxf4 instruction descriptor: A and B e2m1 (1), N, scales ue8m0, M.
__host__ __device__ constexpr uint32_t idesc_mxf4(int m, int n) {
    return (1u << 7) | (1u << 10) | (uint32_t(n >> 3) << 17) | (1u << 23) |
           (uint32_t(m >> 4) << 24);
}

// Preparation: grid (1, n_jobs, z), kPrepThreads threads. Item (block b,
// word c, parity h): the 8 elements 16c + 2j + h (j = 0..7) of block b, one
// 32-bit word of the B image per piece (K positions 64 (b % 8) + 16c + 8h + j,
// nibble j). The 8 items of a block are 8 consecutive lanes: they share the
// block maximum and sum the all-ones groups H, M, L by shuffles (every partial
// sum is exact).
// kG128: blocks of 128 elements (the group-128 layout's scale blocks), 16 items
// each; word c of block b falls in the 64-element half c / 4, which the image
// holds as the K positions 64 (2 (b % 8) + c / 4) + 16 (c % 4) + 8h + j of the
// 1024-element stage. The sums stay exact: 128 elements add one bit to every
// group, which still spans fewer than 24 bits.
template <typename XT, bool kG128>
__global__ void __launch_bounds__(kPrepThreads) t4_prep_kernel(
    const __grid_constant__ MvPrepJob single, const MvPrepJob *__restrict__ jobs,
    const int2 *__restrict__ ctas, int ncols) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Launched as a programmatic dependent of the kernel before it on the stream
    // (a mat-vec that may still read this buffer, or the producer of x): wait
    // for that grid before reading x or writing the prep buffer.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // a plan's CTA list: CTA y takes items ctas[y].y .. +127 of job ctas[y].x
    const int2 cta = ctas ? ctas[blockIdx.y] : make_int2(int(blockIdx.y), 0);
    const int idx0 = ctas ? cta.y : int(blockIdx.z) * kPrepThreads;
    const int idx_step = ctas ? (1 << 30) : int(gridDim.z) * kPrepThreads;
    MvPrepJob J = jobs ? jobs[cta.x] : single;
    if (!jobs) {  // a strided batch of vectors, one per grid row
        J.x = static_cast<const uint8_t *>(single.x) + size_t(blockIdx.y) * single.x_stride;
        J.prep = single.prep + size_t(blockIdx.y) * single.prep_stride;
    }
    using Lt = T4Lay<kG128 ? kLayG128 : kLayBlocks>;
    constexpr int kBE = kG128 ? 128 : 64;  // elements per scale block
    constexpr int kIPB = kBE / 8;          // items (lanes) per block
    const int K = J.K;
    // grid x: the activation column j (pieces in B rows 16 j .., one record per
    // region and column)
    const int j = int(blockIdx.x);
    const XT *xj = static_cast<const XT *>(J.x) + size_t(j) * K;
    const int nb = K / kBE;
    const int rows = kT4N * ncols;
    const int img_bytes = rows * Lt::kStageK / 2;
    const int act_bytes = img_bytes + kT4BetaBytes * ncols;
    uint8_t *act = J.prep + kPrepHeader;  // per stage: image, then region records
    const int lane = threadIdx.x & 31;
    // the block's kIPB threads
    const unsigned grp = kG128 ? 0xFFFFu << (lane & 16) : 0xFFu << (lane & 24);
    // kIPB items per block and nb blocks: whole warps share a block range, so the
    // shuffles below always run with all lanes of a block present
    for (int idx = idx0 + int(threadIdx.x); idx < nb * kIPB; idx += idx_step) {
        const int b = idx / kIPB, c = (idx >> 1) & (kIPB / 2 - 1), h = idx & 1;
        const XT *xe = xj + b * kBE + c * 16 + h;
        float v[8];
        float m = 0.0f;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            v[jj] = ld_x(xe + 2 * jj);
            m = fmaxf(m, fabsf(v[jj]));
        }
#pragma unroll
        for (int o = 1; o < kIPB; o <<= 1) m = fmaxf(m, __shfl_xor_sync(grp, m, o));
        // v = x * 2^(2 - e), max |v| over the block in [2, 4); all-zero (or
        // non-finite) blocks keep e = 0
        int e = 0;
        if (m > 0.0f && m <= 3.402823466e38f) frexpf(m, &e);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) v[jj] = mul_pow2(v[jj], 2 - e);
        uint8_t *bimg = act + size_t(b >> 3) * act_bytes;
        // byte of the item's first K position in the stage image
        const int kbyte = kG128 ? 32 * (2 * (b & 7) + (c >> 2)) + 8 * (c & 3) + 4 * h
                                : 32 * (b & 7) + 8 * c + 4 * h;
        float grp_sum[3] = {0.0f, 0.0f, 0.0f};  // this item's share of H, M, L
        // Piece p of element jj is e2m1(w), w = r_p * 4^p the scaled residual
        // (w = v for p = 0), rounded to nearest even by the conversion; then
        // w <- 4 (w - piece), exact: |w| < 4 at p = 0 (grid spacing 1 on [2, 4],
        // 1/2 below) and |w| <= 2 after it, so every residual is a multiple of
        // the grid's spacing far inside f32's precision.
#pragma unroll
        for (int p = 0; p < kT4Pieces; ++p) {
            const uint32_t word = e2m1x8_rn(v);
            *reinterpret_cast<uint32_t *>(bimg + img_offset(rows, kT4N * j + p, kbyte)) = word;
            float psum = 0.0f;  // sum of the item's 8 pieces (exact)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float lo, hi;
                e2m1x2_values(word, k, lo, hi);
                v[2 * k] = fmaf(v[2 * k], 4.0f, -4.0f * lo);
                v[2 * k + 1] = fmaf(v[2 * k + 1], 4.0f, -4.0f * hi);
                psum += lo + hi;
            }
            // sum of piece / 2, weighted by 4^-p, into its group
            const int gi = p < 6 ? 0 : p < 12 ? 1 : 2;
            grp_sum[gi] = fmaf(psum * 0.5f, __int_as_float((127 - 2 * p) << 23), grp_sum[gi]);
        }
#pragma unroll
        for (int gi = 0; gi < 3; ++gi)
#pragma unroll
            for (int o = 1; o < kIPB; o <<= 1) grp_sum[gi] += __shfl_xor_sync(grp, grp_sum[gi], o);
        if ((idx & (kIPB - 1)) == 0)
            *reinterpret_cast<float4 *>(bimg + img_bytes + ((b & 7) * ncols + j) * kT4BlockRec * 4) =
                make_float4(pow2f(e - 1), grp_sum[0], grp_sum[1], grp_sum[2]);
    }
}

constexpr int kT4SplitCodeBytes = kTcRows * 128;  // 16 KB of codes, then 2 KB of scales
static_assert(kT4SplitCodeBytes + kTcRows * 16 == kRawBytes, "split stage = block stage bytes");

// kLay: the weight layout. kLaySplit: codes [N][K/64][16] and scales [N][K/64];
// the stage's code box is 128 bytes x 128 rows with 128-byte swizzle and its
// scale box 16 bytes x 128 rows, together the same 18 KB as the block box of the
// 18-byte layout. kLayG128: 34-byte blocks of 128; the stage's box is 272 bytes
// (eight blocks) x 128 rows, read through a 16-bit view of the rows because a
// box holds at most 256 elements a dimension.
// At most 128 registers a thread (384 x 128 = 48K of the SM's 64K), so a CTA of
// the next prep kernel (256 threads x 64 registers) can be resident beside it
// and the programmatic launch overlaps the two.
template <int kLay, int kNc = 1>
__global__ void __maxnreg__(kNc == 1 ? 128 : 112)
    mv_t4_kernel(const __grid_constant__ MvJob single, const MvParams p) {
    using Lt = T4Lay<kLay, kNc>;
    static_assert(kNc == 1 || (kNc == 2 && kLay == kLayBlocks), "two columns: 64-weight blocks");
    constexpr bool kSplit = kLay == kLaySplit;
    constexpr bool kG = kLay == kLayG128;
    constexpr int kRowBytes = kG ? kG128RowBytes : kChunkBytes;  // a row's bytes in a stage
    // The next prep launch on the stream may become resident now; it waits for
    // this grid before it touches any buffer this kernel reads.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *act_ring = smem;                                   // Lt::kStages activation slots
    uint8_t *raw_ring = act_ring + Lt::kStages * Lt::kActSlot;  // Lt::kStages weight boxes
    uint64_t *full = reinterpret_cast<uint64_t *>(raw_ring + Lt::kStages * Lt::kRaw);
    uint64_t *empty = full + Lt::kStages;
    uint64_t *a_full = empty + Lt::kStages;
    uint64_t *a_empty = a_full + kT4ABufs;
    uint64_t *d_full = a_empty + kT4ABufs;
    uint64_t *d_empty = d_full + 2;
    uint64_t *drain = d_empty + 2;  // [2] one per MMA issuer: its final commit
    uint64_t *tile_w1 = drain + 2;  // two columns, [4] per quarter: warp 12+q's tile sums are in s_pair
    uint64_t *tile_w0 = tile_w1 + 4;  // [4] per quarter: warp 8+q has read them
    __shared__ float s_pair[kNc == 2 ? 4 * 32 * 4 : 1];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    // per ring slot, written by the producer before the slot's barrier arrive:
    // where the epilogue writes the tile that the stage belongs to
    __shared__ StageMeta s_meta[Lt::kStages];

    const uint64_t wl = p.wait_ns ? p.wait_ns : kWaitLimitNs;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // a plan CTA's share of the schedule (one load); the first item's tensor map early
    const MvFirst fst = p.jobs ? p.first[blockIdx.x] : MvFirst{};
    if (warp == kProdWarp && lane == 0 && p.jobs && fst.n_items > 0)
        prefetch_tensormap(&p.jobs[fst.job0].tmap);

    if (threadIdx.x == 0) {
        for (int i = 0; i < Lt::kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], Lt::kEpi);
        }
        if (kNc == 2)
            for (int i = 0; i < 4; ++i) {
                mbar_init(&tile_w1[i], 1);
                mbar_init(&tile_w0[i], 1);
            }
        for (int i = 0; i < kT4ABufs; ++i) {
            mbar_init(&a_full[i], kExpWarps);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], kEpiWarps);
        }
        for (int i = 0; i < 2; ++i) mbar_init(&drain[i], 1);
        s_abort = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&s_tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    int n_items, item_base = 0;
    if (p.jobs) {
        item_base = fst.item_base;
        n_items = fst.n_items;
    } else {
        // one matrix: its tiles; expert mat-vec: (output vector, tile) pairs
        const int total = p.moe.ids ? p.moe.n_vec * single.n_tiles : single.n_tiles;
        n_items = blockIdx.x < unsigned(total) ? (total - 1 - int(blockIdx.x)) / int(gridDim.x) + 1
                                               : 0;
    }
    auto item_at = [&](int i, const MvJob *&J, int &tile) {
        if (p.jobs) {
            if (i == 0) {  // from the CTA's record
                J = &p.jobs[fst.job0];
                tile = fst.tile0;
            } else {
                const MvItem it = p.items[item_base + i];
                J = &p.jobs[it.job];
                tile = it.tile;
            }
        } else {
            J = &single;
            tile = int(blockIdx.x) + i * int(gridDim.x);
        }
    };
    // stages of this CTA (every role but the producer runs a flat stage loop)
    const int n_stages = p.jobs ? fst.n_stages : n_items * single.n_chunks;
    auto stage_parity = [](int s) { return uint32_t(s / Lt::kStages) & 1u; };
    // A buffers in order of use: unit u = s * Lt::kAPer + h is part h of stage s
    auto a_buf = [](int u) { return u % kT4ABufs; };
    auto a_use = [](int u) { return uint32_t(u / kT4ABufs) & 1u; };
    auto a_col = [](int u) { return uint32_t(kT4ACol + (u % kT4ABufs) * 64); };
    auto d_col = [](int s) { return uint32_t((s & 1) * 128); };

    if (warp == kProdWarp || warp == kProdWarp2) {
        // ------------------------------ producers ------------------------------
        // warp 0 issues the even stages, warp 2 the odd ones; both walk every item
        const int pmine = warp == kProdWarp2 ? 0 : 1;
        if (lane == 0) {
            int s = 0, last = -1;
            bool ok = true, prep_ready = false;
            for (int i = 0; i < n_items && ok; ++i) {
                const MvJob *J;
                int tile;
                item_at(i, J, tile);
                // a plan's first item: the fields come with the CTA's record
                const bool rec = p.jobs && i == 0;
                const uint8_t *prep = rec ? fst.prep0 : J->prep;
                float *y_out = rec ? fst.y0 : J->y;
                const int n_rows = rec ? fst.n0 : J->N;
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
                const uint8_t *act = prep + kPrepHeader;
                const int nch = rec ? fst.n_chunks0 : J->n_chunks;
                for (int ch = 0; ch < nch; ++ch, ++s) {
                    if ((s & 1) != pmine) continue;
                    if (p.stall_stage && s >= p.stall_stage - 1) {  // test hook
                        ok = false;
                        break;
                    }
                    const int st = s % Lt::kStages;
                    if (!mbar_wait(&empty[st], stage_parity(s) ^ 1u, p.err, kTagT4Empty, true, wl) ||
                        *(volatile int *)&s_abort) {
                        ok = false;
                        s_abort = 1;
                        break;
                    }
                    StageMeta &m = s_meta[st];
                    m.y = y_out;
                    m.row0 = tile * kTcRows;
                    m.n_rows = n_rows;
                    m.flags = ch == nch - 1 ? kLastOfTile : 0;
                    mbar_arrive_expect_tx(&full[st], Lt::kRaw + Lt::kAct);
                    if (kSplit) {
                        tma_load_2d(raw_ring + st * Lt::kRaw, &J->tmap, ch * 128,
                                    row_base + tile * kTcRows, &full[st]);
                        tma_load_2d(raw_ring + st * Lt::kRaw + kT4SplitCodeBytes, &J->tmap_d,
                                    ch * 16, row_base + tile * kTcRows, &full[st]);
                    } else if (kG) {  // 16-bit elements: x = 136 ch (272 bytes, 16-aligned)
                        tma_load_2d(raw_ring + st * Lt::kRaw, &J->tmap, ch * (kG128RowBytes / 2),
                                    row_base + tile * kTcRows, &full[st]);
                    } else {
                        tma_load_2d(raw_ring + st * Lt::kRaw, &J->tmap, ch * kChunkBytes,
                                    row_base + tile * kTcRows, &full[st]);
                    }
                    if (!prep_ready) {
                        grid_dependency_wait();  // the B images come from the prep kernel
                        prep_ready = true;
                    }
                    bulk_g2s(act_ring + st * Lt::kActSlot, act + size_t(ch) * Lt::kAct,
                             Lt::kAct, &full[st]);
                    last = s;
                }
            }
            if (!ok) {
                // let this producer's copies in flight land (bounded) before the CTA exits
                for (int t = last; t >= 0 && t > last - Lt::kStages; t -= 2)
                    mbar_wait(&full[t % Lt::kStages], stage_parity(t), p.err, kTagT4Full, false, wl);
            }
        }
    } else if (warp == kMmaWarp || warp == kMmaWarp2) {
        // ------------------------------ MMA issuers ------------------------------
        // even / odd stages; the whole warp runs the loop and waits (so it stays
        // converged), the elected lane issues (one K = 64 MMA per block) and commits
        constexpr uint32_t idesc = idesc_mxf4(kTcRows, Lt::kN);
        const bool leader = elect_one();
        const int mine = warp == kMmaWarp ? 0 : 1;
        const uint64_t desc0 = sw128_desc(smem_addr(act_ring));
        const uint32_t sfa = tmem + kT4ScaleCol, sfb = tmem + kT4ScaleCol + 4;
        int last = -1;
        if constexpr (kNc == 2) {
            // One issuer (warp kMmaWarp) takes every stage. A stage fills both
            // accumulator buffers in turn, blocks 0-3 into buffer 0 and 4-7 into
            // buffer 1 (each block 32 columns: 16 pieces of 2 columns), so each
            // buffer's waits come in stage order.
            for (int s = mine == 0 ? 0 : n_stages; s < n_stages; ++s) {
                const int st = s % Lt::kStages;
                const uint64_t dst = desc0 + uint64_t((st * Lt::kActSlot) >> 4);
                const uint32_t dpar = uint32_t(s & 1) ^ 1u;  // buffer released by stage s - 1
                bool ok = true;
#pragma unroll
                for (int ss = 0; ss < 2; ++ss) {
                    const bool got =
                        ss == 0 ? mbar_wait3(&full[st], stage_parity(s), kTagT4Full, &a_full[a_buf(s)],
                                             a_use(s), kTagT4AFull, &d_empty[0], dpar, kTagT4DEmpty,
                                             p.err, wl, &s_abort)
                                : mbar_wait(&d_empty[1], dpar, p.err, kTagT4DEmpty, false, wl) &&
                                      !*(volatile int *)&s_abort;
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    last = s;
                    if (leader) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int sb = 4 * ss + i;
                            tc_mma_mxf4_ta(tmem + ss * 128 + i * Lt::kN, tmem + a_col(s) + sb * 8,
                                           dst + uint64_t(((sb >> 2) * (Lt::kN * 128) + (sb & 3) * 32) >> 4),
                                           idesc, sfa, sfb, 0u);
                        }
                        tc_commit(&d_full[ss]);
                    }
                    __syncwarp();
                }
                if (!ok) {
                    s_abort = 1;
                    break;
                }
                if (leader) tc_commit(&a_empty[a_buf(s)]);
                __syncwarp();
            }
        } else {
            for (int s = mine; s < n_stages; s += 2) {
                const int st = s % Lt::kStages;
                const uint32_t d_base = tmem + d_col(s);
                const uint64_t dst = desc0 + uint64_t((st * Lt::kActSlot) >> 4);
                bool ok = true;
#pragma unroll
                for (int h = 0; h < Lt::kAPer; ++h) {
                    const int u = s * Lt::kAPer + h;
                    const bool got =
                        h > 0 ? mbar_wait(&a_full[a_buf(u)], a_use(u), p.err, kTagT4AFull, false, wl) &&
                                    !*(volatile int *)&s_abort
                              : mbar_wait3(&full[st], stage_parity(s), kTagT4Full, &d_empty[s & 1],
                                           (uint32_t(s >> 1) & 1u) ^ 1u, kTagT4DEmpty,
                                           &a_full[a_buf(u)], a_use(u), kTagT4AFull, p.err, wl,
                                           &s_abort);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    last = s;
                    const uint32_t a_base = tmem + a_col(u);
                    if (leader) {
                        // the A buffer's eight 64-element sub-blocks sb of the stage;
                        // region = the block that owns d: sb itself, or for
                        // group-128 block sb / 2 (its second half accumulates)
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int sb = 8 * h + i;
                            const int region = kG ? sb >> 1 : sb;
                            tc_mma_mxf4_ta(d_base + region * kT4N, a_base + i * 8,
                                           dst + uint64_t(((sb >> 2) * 2048 + (sb & 3) * 32) >> 4),
                                           idesc, sfa, sfb, kG ? uint32_t(sb & 1) : 0u);
                        }
                        tc_commit(&a_empty[a_buf(u)]);
                    }
                    __syncwarp();
                }
                if (!ok) {
                    s_abort = 1;
                    break;
                }
                if (leader) tc_commit(&d_full[s & 1]);
                __syncwarp();
            }
        }
        // TMEM is freed only after this issuer's MMAs completed: one more commit
        // tracks all of them
        if (last >= 0) {
            if (leader) tc_commit(&drain[mine]);
            __syncwarp();
            if (leader) mbar_wait(&drain[mine], 0u, p.err, kTagT4DFull, false, wl);
            __syncwarp();
        }
    } else if (warp >= kExpWarp0 && warp < kExpWarp0 + kExpWarps) {
        // ------------------------------ expansion ------------------------------
        // warp w: TMEM lane quarter w % 4 (rows 32 (w % 4) ..), all 8 blocks
        const int qd = warp & 3;
        const int row = 32 * qd + lane;
        const uint32_t lane_base = uint32_t(32 * qd) << 16;
        {  // scale factors 1.0 (ue8m0 127) for this quarter's lanes, columns 448-463
            const uint32_t one = 0x7F7F7F7Fu;
#pragma unroll
            for (int c = 0; c < 16; c += 4) tmem_st4(tmem + lane_base + kT4ScaleCol + c, one, one, one, one);
        }
        bool ok = true;
        // The next stage's barriers are tested (without blocking) while this
        // stage's codes are expanded; when both had completed, the next stage
        // starts without a wait. An incomplete one takes the bounded wait.
        bool ready = false;
        for (int s = 0; s < n_stages && ok; ++s) {
            const int st = s % Lt::kStages;
            // one 64-column A buffer per 512 weights of the stage (two for group-128)
#pragma unroll 1
            for (int h = 0; h < Lt::kAPer; ++h) {
                const int u = s * Lt::kAPer + h;
                bool got = h == 0 && __all_sync(0xffffffffu, ready);
                if (!got)
                    got = h > 0 ? mbar_wait(&a_empty[a_buf(u)], a_use(u) ^ 1u, p.err, kTagT4AFull,
                                            false, wl) &&
                                      !*(volatile int *)&s_abort
                                : mbar_wait2(&full[st], stage_parity(s), kTagT4Full,
                                             &a_empty[a_buf(u)], a_use(u) ^ 1u, kTagT4AFull, p.err,
                                             wl, &s_abort);
                if (!__all_sync(0xffffffffu, got)) {
                    s_abort = 1;
                    ok = false;
                    break;
                }
                tc_fence_after();
                // This A buffer's code words, both 32-column halves G, loaded first.
                // Blocks layout: half G is bytes 72 G .. 72 G + 71 of the row's stage
                // slice, 9 8-byte words; even blocks start 2 bytes into a 4-byte word
                // (d first). Group-128: half h of the stage is blocks 4h .. 4h + 3
                // (136 bytes from an 8-byte boundary); its half G is 9 8-byte words
                // from byte 64 G (8-byte loads: 2-way bank conflicts at the 272-byte
                // row stride). Split layout: four 16-byte chunks per half, chunk 4G+bi
                // at (4G+bi) ^ (row % 8) under the 128-byte swizzle.
                uint32_t w32[2][18];
#pragma unroll
                for (int G = 0; G < 2; ++G) {
                    if constexpr (kSplit) {
                        const uint8_t *rp = raw_ring + st * Lt::kRaw + row * 128;
#pragma unroll
                        for (int bi = 0; bi < 4; ++bi) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(
                                rp + (((4 * G + bi) ^ (row & 7)) << 4));
                            w32[G][4 * bi + 0] = v.x;
                            w32[G][4 * bi + 1] = v.y;
                            w32[G][4 * bi + 2] = v.z;
                            w32[G][4 * bi + 3] = v.w;
                        }
                    } else {
                        const uint8_t *rp =
                            kG ? raw_ring + st * Lt::kRaw + row * kG128RowBytes + h * 136 + G * 64
                               : raw_ring + st * Lt::kRaw + row * kChunkBytes + G * 72;
#pragma unroll
                        for (int k = 0; k < 9; ++k) {
                            const uint2 v = *reinterpret_cast<const uint2 *>(rp + 8 * k);
                            w32[G][2 * k] = v.x;
                            w32[G][2 * k + 1] = v.y;
                        }
                    }
                }
                if (h == Lt::kAPer - 1) {  // the next stage's barriers, tested now
                    const int s1 = s + 1, u1 = s1 * Lt::kAPer;
                    const bool r1 = mbar_test_wait(&full[s1 % Lt::kStages], stage_parity(s1));
                    const bool r2 = mbar_test_wait(&a_empty[a_buf(u1)], a_use(u1) ^ 1u);
                    ready = s1 < n_stages && r1 && r2;
                }
#pragma unroll
                for (int G = 0; G < 2; ++G) {  // 32 columns of the A buffer per store
                    uint32_t a[32];
                    const uint32_t(&w)[18] = w32[G];
                    if constexpr (kG) {
                        // this store: blocks 2G and 2G + 1 (sub-blocks 4G .. 4G + 3 of
                        // the A buffer). Block 2G + b2 starts at byte 34 b2 + 4 G of the
                        // words: its codes are word wi at byte 34 b2 + 4 G + 2 + 4 wi,
                        // 2 bytes into a 32-bit word for b2 = 0 and aligned for b2 = 1.
#pragma unroll
                        for (int b2 = 0; b2 < 2; ++b2) {
#pragma unroll
                            for (int wi = 0; wi < 8; ++wi) {
                                const uint32_t cw =
                                    b2 ? w[9 + G + wi] : __byte_perm(w[G + wi], w[G + wi + 1], 0x5432);
                                // sub-block 2 b2 + wi / 4 of this store, word wi % 4
                                const int o = 8 * (2 * b2 + (wi >> 2)) + 2 * (wi & 3);
                                a[o] = cw & 0x33333333u;
                                a[o + 1] = (cw >> 2) & 0x33333333u;
                            }
                        }
                    } else if constexpr (kSplit) {
#pragma unroll
                        for (int bi = 0; bi < 4; ++bi) {
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                a[8 * bi + 2 * c + 0] = w[4 * bi + c] & 0x33333333u;
                                a[8 * bi + 2 * c + 1] = (w[4 * bi + c] >> 2) & 0x33333333u;
                            }
                        }
                    } else {
#pragma unroll
                        for (int bi = 0; bi < 4; ++bi) {
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const uint32_t cw = block_word(w, bi, c);
                                a[8 * bi + 2 * c + 0] = cw & 0x33333333u;
                                a[8 * bi + 2 * c + 1] = (cw >> 2) & 0x33333333u;
                            }
                        }
                    }
                    tmem_st32(tmem + lane_base + a_col(u) + 32 * G, a);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[a_buf(u)]);
            }
        }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + Lt::kEpi) {
        // ------------------------------ epilogue ------------------------------
        // warp w: TMEM lane quarter w % 4, all 8 blocks of each stage; it writes y
        // at the tile's last stage. Every wait is bounded; a warp whose wait
        // fails leaves the loop.
        const int qd = warp & 3;
        const int row = 32 * qd + lane;
        const uint32_t lane_base = uint32_t(32 * qd) << 16;
        if constexpr (kNc == 1) {
        float acc = 0.0f, comp = 0.0f;  // compensated sum of the stage sums
        for (int s = 0; s < n_stages; ++s) {
            const int st = s % Lt::kStages;
            const bool got = mbar_wait2(&full[st], stage_parity(s), kTagT4Full, &d_full[s & 1],
                                        uint32_t(s >> 1) & 1u, kTagT4DFull, p.err, wl, &s_abort);
            if (!__all_sync(0xffffffffu, got)) {
                s_abort = 1;
                break;
            }
            tc_fence_after();
            const StageMeta m = s_meta[st];
            const uint32_t d_base = tmem + lane_base + d_col(s);
            const uint8_t *rp = raw_ring + st * Lt::kRaw + row * kRowBytes;
            const float4 *brec =
                reinterpret_cast<const float4 *>(act_ring + st * Lt::kActSlot + Lt::kImg);
            float stage_sum = 0.0f;
            // regions (blocks of d) 4 hb .. 4 hb + 3: their 16 pieces each (64 registers)
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                uint32_t r[4][16];
#pragma unroll
                for (int bi = 0; bi < 4; ++bi) tmem_ld16(d_base + (4 * hb + bi) * kT4N, r[bi]);
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
                        kSplit ? lds_half_as_float(raw_ring + st * Lt::kRaw + kT4SplitCodeBytes +
                                                   row * 16 + 2 * b)
                               : lds_half_as_float(rp + (kG ? kG128Bytes : 18) * b);
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
            if (m.flags & kLastOfTile) {
                const int rr = m.row0 + row;
                if (m.y && rr < m.n_rows) m.y[rr] = acc + comp;
                acc = 0.0f;
                comp = 0.0f;
            }
        }
        } else {
        // Two columns: the stage's blocks 0-3 arrive in accumulator buffer 0 and
        // 4-7 in buffer 1, each block 32 columns (column jc's pieces at 16 jc ..).
        // Warp 8+q drains buffer 0 and warp 12+q buffer 1 of lane quarter q; at a
        // tile's end warp 12+q hands its sums to warp 8+q through s_pair, which
        // adds them and writes y.
        const int e = (warp - kEpiWarp0) >> 2;
        float *pair = s_pair + (qd * 32 + lane) * 4;
        float acc[2] = {0.0f, 0.0f}, comp[2] = {0.0f, 0.0f};
        int n_tile_ends = 0;
        for (int s = 0; s < n_stages; ++s) {
            const int st = s % Lt::kStages;
            const bool got = mbar_wait2(&full[st], stage_parity(s), kTagT4Full, &d_full[e],
                                        uint32_t(s & 1), kTagT4DFull, p.err, wl, &s_abort);
            if (!__all_sync(0xffffffffu, got)) {
                s_abort = 1;
                break;
            }
            tc_fence_after();
            const StageMeta m = s_meta[st];
            const uint8_t *rp = raw_ring + st * Lt::kRaw + row * kRowBytes;
            const float4 *brec =
                reinterpret_cast<const float4 *>(act_ring + st * Lt::kActSlot + Lt::kImg);
            const uint32_t d_base = tmem + lane_base + e * 128;
            float stage_sum[2] = {0.0f, 0.0f};
#pragma unroll
            for (int bi = 0; bi < 4; ++bi) {  // block 4 e + bi: 32 registers
                uint32_t r[32];
                tmem_ld32(d_base + bi * Lt::kN, r);
                tmem_wait_ld();
                if (bi == 3) {  // the buffer's accumulators are all in registers
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&d_empty[e]);
                }
                const int b = 4 * e + bi;
                const float d = lds_half_as_float(rp + 18 * b);
#pragma unroll
                for (int jc = 0; jc < 2; ++jc) {
                    auto C = [&](int pp) { return __uint_as_float(r[kT4N * jc + pp]); };
                    float gh = C(5) * 0x1p-10f, gm = C(11) * 0x1p-22f, gl = C(15) * 0x1p-30f;
#pragma unroll
                    for (int pp = 4; pp >= 0; --pp) gh = fmaf(C(pp), __int_as_float((127 - 2 * pp) << 23), gh);
#pragma unroll
                    for (int pp = 10; pp >= 6; --pp) gm = fmaf(C(pp), __int_as_float((127 - 2 * pp) << 23), gm);
#pragma unroll
                    for (int pp = 14; pp >= 12; --pp) gl = fmaf(C(pp), __int_as_float((127 - 2 * pp) << 23), gl);
                    const float4 br = brec[2 * b + jc];  // {2^(e - 1), H, M, L}
                    const float t = ((gh - br.y) + (gm - br.z)) + (gl - br.w);
                    stage_sum[jc] = fmaf(d, t * br.x, stage_sum[jc]);
                }
            }
            // both warps of a quarter release every stage once they have read its
            // records and d values
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
#pragma unroll
            for (int jc = 0; jc < 2; ++jc) {  // acc + comp += stage_sum (two-sum)
                const float sum = acc[jc] + stage_sum[jc];
                const float bb = sum - acc[jc];
                comp[jc] += (acc[jc] - (sum - bb)) + (stage_sum[jc] - bb);
                acc[jc] = sum;
            }
            if (m.flags & kLastOfTile) {
                const int t = n_tile_ends++;
                if (e == 1) {
                    // wait until warp 8+q has read the previous tile's sums
                    const bool free_pair =
                        t == 0 || mbar_wait(&tile_w0[qd], uint32_t(t - 1) & 1u, p.err, kTagT4Pair,
                                            false, wl);
                    if (!__all_sync(0xffffffffu, free_pair)) {
                        s_abort = 1;
                        break;
                    }
#pragma unroll
                    for (int jc = 0; jc < 2; ++jc) {
                        pair[2 * jc] = acc[jc];
                        pair[2 * jc + 1] = comp[jc];
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tile_w1[qd]);
                } else {
                    const bool have =
                        mbar_wait(&tile_w1[qd], uint32_t(t) & 1u, p.err, kTagT4Pair, false, wl);
                    if (!__all_sync(0xffffffffu, have)) {
                        s_abort = 1;
                        break;
                    }
                    const int rr = m.row0 + row;
#pragma unroll
                    for (int jc = 0; jc < 2; ++jc) {
                        const float o = pair[2 * jc];
                        const float sum = acc[jc] + o;
                        const float bb = sum - acc[jc];
                        const float err = (acc[jc] - (sum - bb)) + (o - bb);
                        const float yv = sum + (comp[jc] + pair[2 * jc + 1] + err);
                        if (m.y && rr < m.n_rows) m.y[size_t(jc) * m.n_rows + rr] = yv;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tile_w0[qd]);
                }
#pragma unroll
                for (int jc = 0; jc < 2; ++jc) acc[jc] = comp[jc] = 0.0f;
            }
        }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}


// ---------------------------------------------------------------------------
// tcgen05 mat-vec on signed e4m3 codes (ncols 3..8)
//
// Codes. The expansion warps turn each 2-bit code into the e4m3 value q - 1
// (-1, 0, 1, 2 are exact e4m3 values) with one byte-permute lookup per 4 codes:
// selecting byte q of the constant 0x403800B8 gives 0xB8 (-1), 0x00, 0x38 (+1)
// or 0x40 (+2). From a code word w, the selectors w, w >> 2, w >> 16 and
// w >> 18 (masked to their low two bits per nibble) give elements {0,2,4,6},
// {1,3,5,7}, {8,10,12,14} and {9,11,13,15}; tensor-memory column 4c + r of a
// block holds register r of word c, i.e. K byte 16c + 4r + j of the block is
// element 16c + 8 (r >> 1) + (r & 1) + 2j. A weight of code 1 is an exact zero
// operand: it contributes nothing however large its activation is.
//
// Activations, block by block and column by column. For block b of column j
// with M = max |x| over the block, M = f * 2^e (f in [0.5, 1)), the prep kernel
// forms v = x * 2^(8 - e) (max |v| in [128, 256)) and splits it into 5 e4m3
// pieces: piece p = e4m3(r_p * 16^p), r_0 = v, r_(p+1) = r_p - piece_p * 16^-p.
// e4m3 keeps 4 significant bits of each element's own magnitude, every
// subtraction is exact, and |r_5| <= 2^-20 |v| + 2^-26 (the last term from
// e4m3's subnormal step, i.e. 2^-33 of the block maximum). Piece p of column j
// is B row n = 5j + p; the MMA's N is 5 * ncols rounded up to 16.
//
// Per-block accumulators. d and the activation scale change every block, so
// each block has its own accumulator columns (N per block). The 512 tensor-
// memory columns hold two A buffers of 128 (a stage's 8 blocks x 64 e4m3 codes)
// and two accumulator buffers of 128; a stage's 8 blocks are issued in
// sub-stages of 128 / N blocks (8, 4 or 2), each committed to its own
// accumulator buffer, so the epilogue drains one sub-stage while the tensor
// core fills the other. The epilogue forms t_j = sum_p 16^-p C_(5j+p) per
// block and column and adds d * 2^(e - 8) * t_j; the stage sums are accumulated
// with a two-sum.
// ---------------------------------------------------------------------------
constexpr int kS8Pieces = 5;
constexpr int kS8RecBytes = 256;  // per stage: float scale[8 blocks][ncols]
__host__ __device__ constexpr int s8_n(int nc) { return (kS8Pieces * nc + 15) / 16 * 16; }
__host__ __device__ constexpr int s8_bs(int nc) { return 128 / s8_n(nc); }
__host__ __device__ constexpr int s8_subs(int nc) { return kChunkBlocks / s8_bs(nc); }
__host__ __device__ constexpr int s8_img_bytes(int nc) { return s8_n(nc) * kChunkBlocks * 64; }
// full/empty per stage, a_full/a_empty, d_full/d_empty, drain, and per lane
// quarter the two tile-end hand-offs between its epilogue warps
constexpr int kS8Barriers = 2 * 8 + 2 * 2 + 2 * 2 + 2 + 2 * 4;
// The fp4 kernel's roles with two epilogue warps per lane quarter (warps 8-11
// drain accumulator buffer 0, warps 12-15 buffer 1): 16 warps. With one
// accumulator sub-stage per stage (ncols 3) the expansion is the longest
// role, and it also gets two warps per lane quarter (warps 4-7 expand blocks
// 0-3 of a stage, warps 16-19 blocks 4-7): 20 warps at most 96 registers each.
constexpr int kS8EpiWarps = 8;
constexpr int kS8ExpWarp1 = 16;
__host__ __device__ constexpr bool s8_exp2(int nc) { return s8_n(nc) <= 16; }
__host__ __device__ constexpr int s8_threads(int nc) { return (s8_exp2(nc) ? 20 : 16) * 32; }
constexpr int kS8PairBytes = 4 * 32 * 2 * 8 * 4;  // tile-end exchange, ncols <= 8
// shared-memory slot of a stage's activation data (image, then block scales:
// one bulk copy), 1024-aligned for the swizzled image
__host__ __device__ constexpr int s8_act_slot(int nc) { return s8_img_bytes(nc) + 1024; }
// An even number of stages: each ring slot is then always filled by the same
// producer (stage parity), so no producer waits two barrier phases ahead.
__host__ __device__ constexpr int s8_stages(int nc) {
    return (kSmemOptIn - 2048 - kS8PairBytes - kS8Barriers * 8) / (kRawBytes + s8_act_slot(nc)) < 8
               ? (kSmemOptIn - 2048 - kS8PairBytes - kS8Barriers * 8) /
                     (kRawBytes + s8_act_slot(nc)) / 2 * 2
               : 8;
}
__host__ __device__ constexpr int s8_smem(int nc) {
    return 1024 /* alignment slack */ + s8_stages(nc) * (s8_act_slot(nc) + kRawBytes) +
           kS8Barriers * 8;
}
static_assert(s8_bs(2) == 8 && s8_bs(4) == 4 && s8_bs(8) == 2, "sub-stage sizes");
static_assert(s8_stages(8) >= 4 && s8_smem(8) <= kSmemOptIn - 1024, "shared memory");
static_assert(s8_stages(2) % 2 == 0 && s8_stages(4) % 2 == 0 && s8_stages(8) % 2 == 0 &&
                  kT4Stages % 2 == 0,
              "an even number of ring stages (two producers)");
constexpr int kS8ACol = 0;    // A buffers at 0 and 128
constexpr int kS8DCol = 256;  // accumulator buffers at 256 and 384
constexpr uint32_t kS8Lut = 0x403800B8u;  // e4m3 of q - 1 in byte q
constexpr int kTagS8Full = 121;
constexpr int kTagS8Empty = 122;
constexpr int kTagS8AFull = 123;
constexpr int kTagS8DFull = 124;
constexpr int kTagS8DEmpty = 125;
constexpr int kTagS8Pair = 126;

size_t s8_prep_bytes(int64_t K, int ncols) {
    const size_t n_chunks = size_t(K / 512);
    size_t b = kPrepHeader + n_chunks * (s8_img_bytes(ncols) + kS8RecBytes);
    return (b + 255) & ~size_t(255);
}

// kind::f8f6f4 instruction descriptor: D f32, A and B e4m3, both K-major, N, M.
__host__ __device__ constexpr uint32_t idesc_e4m3(int m, int n) {
    return (1u << 4) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

// Preparation: grid (ncols, n_jobs, z), kPrepThreads threads. Item (block b,
// word c, register r) of column j = blockIdx.x: the 4 elements
// 16c + 8 (r >> 1) + (r & 1) + 2i (i = 0..3) of block b, which sit at K bytes
// 64 (b % 8) + 16c + 4r + i of the stage; one 32-bit word of the image per
// piece. The 16 items of a block are 16 consecutive lanes; they share the
// block maximum by shuffles.
template <typename XT>
__global__ void __launch_bounds__(kPrepThreads) s8_prep_kernel(
    const __grid_constant__ MvPrepJob single, const MvPrepJob *__restrict__ jobs,
    const int2 *__restrict__ ctas, int ncols) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Launched as a programmatic dependent of the kernel before it on the stream
    // (a mat-vec that may still read this buffer, or the producer of x): wait
    // for that grid before reading x or writing the prep buffer.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // a plan's CTA list: CTA (j, y) takes items ctas[y].y .. +127 of job ctas[y].x
    const int2 cta = ctas ? ctas[blockIdx.y] : make_int2(int(blockIdx.y), 0);
    const int idx0 = ctas ? cta.y : int(blockIdx.z) * kPrepThreads;
    const int idx_step = ctas ? (1 << 30) : int(gridDim.z) * kPrepThreads;
    const MvPrepJob &J = jobs ? jobs[cta.x] : single;
    const int K = J.K;
    const int j = blockIdx.x;
    const XT *xj = static_cast<const XT *>(J.x) + size_t(j) * K;
    const int nb = K / 64;
    const int rows = s8_n(ncols);
    const size_t stage_bytes = size_t(s8_img_bytes(ncols)) + kS8RecBytes;
    const int lane = threadIdx.x & 31;
    const unsigned grp = 0xFFFFu << (lane & 16);  // the block's 16 threads
    // 16 items per block: whole half-warps share a block, so the shuffles below
    // always run with all 16 lanes of a block present
    for (int idx = idx0 + int(threadIdx.x); idx < nb * 16; idx += idx_step) {
        const int b = idx >> 4, c = (idx >> 2) & 3, r = idx & 3;
        const XT *xe = xj + b * 64 + 16 * c + 8 * (r >> 1) + (r & 1);
        float v[4];
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[i] = ld_x(xe + 2 * i);
            m = fmaxf(m, fabsf(v[i]));
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) m = fmaxf(m, __shfl_xor_sync(grp, m, o));
        // v = x * 2^(8 - e), max |v| over the block in [128, 256); all-zero (or
        // non-finite) blocks keep e = 0
        int e = 0;
        if (m > 0.0f && m <= 3.402823466e38f) frexpf(m, &e);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = mul_pow2(v[i], 8 - e);
        uint8_t *st_base = J.prep + kPrepHeader + size_t(b >> 3) * stage_bytes;
        const int kc = 64 * (b & 7) + 16 * c + 4 * r;
#pragma unroll
        for (int p = 0; p < kS8Pieces; ++p) {
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
            *reinterpret_cast<uint32_t *>(st_base + img_offset(rows, kS8Pieces * j + p, kc)) =
                uint32_t(lo) | (uint32_t(hi) << 16);
        }
        // column 0 clears the rows past the last column's pieces
        if (j == 0)
            for (int n = kS8Pieces * ncols; n < rows; ++n)
                *reinterpret_cast<uint32_t *>(st_base + img_offset(rows, n, kc)) = 0u;
        if ((idx & 15) == 0)
            reinterpret_cast<float *>(st_base + s8_img_bytes(ncols))[(b & 7) * ncols + j] =
                pow2f(e - 8);
    }
}

// NC: activation columns (2..8).
template <int NC>
__global__ void __launch_bounds__(s8_threads(NC), 1) mv_s8_kernel(const __grid_constant__ MvJob single,
                                              const MvParams p) {
    // The next prep launch on the stream may become resident now; it waits for
    // this grid before it touches any buffer this kernel reads.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int kN = s8_n(NC), kBS = s8_bs(NC), kSub = s8_subs(NC);
    constexpr int kImg = s8_img_bytes(NC), kStages = s8_stages(NC);
    constexpr int kRecCopy = kChunkBlocks * NC * 4;  // bytes of the stage's block scales
    constexpr int kGB = kN <= 16 ? 4 : kN <= 32 ? 2 : 1;  // blocks per tensor-memory wait
    static_assert(kBS % kGB == 0, "whole load groups per sub-stage");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    constexpr int kSlot = s8_act_slot(NC);
    uint8_t *act_ring = smem;                                 // kStages x kSlot (1024-aligned)
    uint8_t *raw_ring = act_ring + kStages * kSlot;           // kStages x 18 KB
    uint64_t *full = reinterpret_cast<uint64_t *>(raw_ring + kStages * kRawBytes);
    uint64_t *empty = full + 8;
    uint64_t *a_full = empty + 8;
    uint64_t *a_empty = a_full + 2;
    uint64_t *d_full = a_empty + 2;
    uint64_t *d_empty = d_full + 2;
    uint64_t *drain = d_empty + 2;  // [2] one per MMA issuer: its final commit
    uint64_t *tile_w1 = drain + 2;  // [4] per quarter: warp 12+q's tile sums are in s_pair
    uint64_t *tile_w0 = tile_w1 + 4;  // [4] per quarter: warp 8+q has read them
    __shared__ float s_pair[4][32][2 * NC];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ StageMeta s_meta[kStages];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // a plan CTA's share of the schedule (one load); the first item's tensor map early
    const MvFirst fst = p.jobs ? p.first[blockIdx.x] : MvFirst{};
    if (warp == kProdWarp && lane == 0 && p.jobs && fst.n_items > 0)
        prefetch_tensormap(&p.jobs[fst.job0].tmap);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kS8EpiWarps);  // both epilogue warps of each quarter
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&a_full[i], s8_exp2(NC) ? 2 * kExpWarps : kExpWarps);
            mbar_init(&a_empty[i], kSub >= 2 ? 2 : 1);  // one commit per issuer on the stage
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], kEpiWarps);  // the 4 warps that drain buffer i
            mbar_init(&drain[i], 1);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&tile_w1[i], 1);
            mbar_init(&tile_w0[i], 1);
        }
        s_abort = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&s_tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    int n_items, item_base = 0;
    if (p.jobs) {
        item_base = fst.item_base;
        n_items = fst.n_items;
    } else {
        n_items = blockIdx.x < unsigned(single.n_tiles)
                      ? (single.n_tiles - 1 - int(blockIdx.x)) / int(gridDim.x) + 1
                      : 0;
    }
    auto item_at = [&](int i, const MvJob *&J, int &tile) {
        if (p.jobs) {
            if (i == 0) {  // from the CTA's record
                J = &p.jobs[fst.job0];
                tile = fst.tile0;
            } else {
                const MvItem it = p.items[item_base + i];
                J = &p.jobs[it.job];
                tile = it.tile;
            }
        } else {
            J = &single;
            tile = int(blockIdx.x) + i * int(gridDim.x);
        }
    };
    const int n_stages = p.jobs ? fst.n_stages : n_items * single.n_chunks;
    auto stage_parity = [](int s) { return uint32_t(s / kStages) & 1u; };

    if (warp == kProdWarp || warp == kProdWarp2) {
        // ------------------------------ producers ------------------------------
        // warp 0 issues the even stages, warp 2 the odd ones; both walk every item
        const int pmine = warp == kProdWarp2 ? 0 : 1;
        if (lane == 0) {
            int s = 0, last = -1;
            bool ok = true, prep_ready = false;
            for (int i = 0; i < n_items && ok; ++i) {
                const MvJob *J;
                int tile;
                item_at(i, J, tile);
                // a plan's first item: the fields come with the CTA's record
                const bool rec = p.jobs && i == 0;
                const uint8_t *prep = (rec ? fst.prep0 : J->prep) + kPrepHeader;
                const int nch = rec ? fst.n_chunks0 : J->n_chunks;
                float *y_out = rec ? fst.y0 : J->y;
                const int n_rows = rec ? fst.n0 : J->N;
                for (int ch = 0; ch < nch; ++ch, ++s) {
                    if ((s & 1) != pmine) continue;
                    const int st = s % kStages;
                    if (!mbar_wait(&empty[st], stage_parity(s) ^ 1u, p.err, kTagS8Empty, true) ||
                        *(volatile int *)&s_abort) {
                        ok = false;
                        s_abort = 1;
                        break;
                    }
                    StageMeta &m = s_meta[st];
                    m.y = y_out;
                    m.row0 = tile * kTcRows;
                    m.n_rows = n_rows;
                    m.flags = ch == nch - 1 ? kLastOfTile : 0;
                    mbar_arrive_expect_tx(&full[st], kRawBytes + kImg + kRecCopy);
                    tma_load_2d(raw_ring + st * kRawBytes, &J->tmap, ch * kChunkBytes,
                                tile * kTcRows, &full[st]);
                    if (!prep_ready) {
                        grid_dependency_wait();  // the images come from the prep kernel
                        prep_ready = true;
                    }
                    bulk_g2s(act_ring + st * kSlot, prep + size_t(ch) * (kImg + kS8RecBytes),
                             kImg + kRecCopy, &full[st]);
                    last = s;
                }
            }
            if (!ok) {
                // let this producer's copies in flight land (bounded) before the CTA exits
                for (int t = last; t >= 0 && t > last - kStages; t -= 2)
                    mbar_wait(&full[t % kStages], stage_parity(t), p.err, kTagS8Full);
            }
        }
    } else if (warp == kMmaWarp || warp == kMmaWarp2) {
        // ------------------------------ MMA issuers ------------------------------
        // Issuer i takes the sub-stages g = i, i + 2, ... (g = s * kSub + ss) and
        // always fills accumulator buffer i, so each of its barrier waits is at
        // most one phase ahead of the barrier. The whole warp runs the loop and
        // waits (so it stays converged); the elected lane issues (two K = 32
        // MMAs per block) and commits the sub-stage to its buffer, and, after
        // its last sub-stage of a stage, the stage's A buffer (with kSub >= 2
        // both issuers work on every stage, and a_empty counts both commits).
        constexpr uint32_t idesc = idesc_e4m3(kTcRows, kN);
        const bool leader = elect_one();
        const int mine = warp == kMmaWarp ? 0 : 1;
        const uint64_t desc0 = sw128_desc(smem_addr(act_ring));
        const uint32_t d_base = tmem + kS8DCol + mine * 128;
        bool issued = false;
        for (int g = mine; g < n_stages * kSub; g += 2) {
            const int s = g / kSub, ss = g - s * kSub;
            const int st = s % kStages;
            const bool first = ss < 2, last_of_stage = ss + 2 >= kSub;
            const bool got =
                first ? mbar_wait3(&full[st], stage_parity(s), kTagS8Full, &a_full[s & 1],
                                   uint32_t(s >> 1) & 1u, kTagS8AFull, &d_empty[mine],
                                   (uint32_t(g >> 1) & 1u) ^ 1u, kTagS8DEmpty, p.err, kWaitLimitNs,
                                   &s_abort)
                      : mbar_wait(&d_empty[mine], (uint32_t(g >> 1) & 1u) ^ 1u, p.err, kTagS8DEmpty) &&
                            !*(volatile int *)&s_abort;
            if (!__all_sync(0xffffffffu, got)) {
                s_abort = 1;
                break;
            }
            tc_fence_after();
            const uint32_t a_base = tmem + kS8ACol + (s & 1) * 128;
            const uint64_t dst = desc0 + uint64_t((st * kSlot) >> 4);
            if (leader) {
#pragma unroll
                for (int bi = 0; bi < kBS; ++bi) {
                    const int b = ss * kBS + bi;
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        tc_mma_f8f6f4_ta(d_base + bi * kN, a_base + b * 16 + kk * 8,
                                         dst + uint64_t(((b >> 1) * (kN * 128) + (b & 1) * 64 +
                                                         kk * 32) >> 4),
                                         idesc, uint32_t(kk));
                }
                tc_commit(&d_full[mine]);
                if (last_of_stage) tc_commit(&a_empty[s & 1]);
            }
            __syncwarp();
            issued = true;
        }
        // TMEM is freed only after this issuer's MMAs completed: one more commit
        // tracks all of them
        if (issued) {
            if (leader) tc_commit(&drain[mine]);
            __syncwarp();
            if (leader) mbar_wait(&drain[mine], 0u, p.err, kTagS8DFull);
            __syncwarp();
        }
    } else if ((warp >= kExpWarp0 && warp < kExpWarp0 + kExpWarps) ||
               (s8_exp2(NC) && warp >= kS8ExpWarp1)) {
        // ------------------------------ expansion ------------------------------
        // warp w: TMEM lane quarter w % 4 (rows 32 (w % 4) ..): all 8 blocks, or with
        // two expansion warps per quarter blocks 4G..4G+3, G = 0 for warps 4-7 and 1
        // for warps 16-19
        const int qd = warp & 3;
        const int row = 32 * qd + lane;
        const uint32_t lane_base = uint32_t(32 * qd) << 16;
        for (int s = 0; s < n_stages; ++s) {
            const int st = s % kStages;
            const bool got = mbar_wait2(&full[st], stage_parity(s), kTagS8Full, &a_empty[s & 1],
                                        (uint32_t(s >> 1) & 1u) ^ 1u, kTagS8AFull, p.err,
                                        kWaitLimitNs, &s_abort);
            if (!__all_sync(0xffffffffu, got)) {
                s_abort = 1;
                break;
            }
            tc_fence_after();
            const int g_lo = s8_exp2(NC) ? (warp >= kS8ExpWarp1 ? 1 : 0) : 0;
            const int g_hi = s8_exp2(NC) ? g_lo + 1 : 2;
#pragma unroll
            for (int G = g_lo; G < g_hi; ++G) {
                const uint8_t *rp = raw_ring + st * kRawBytes + row * kChunkBytes + G * 72;
                uint32_t u[18];
#pragma unroll
                for (int k = 0; k < 9; ++k) {
                    const uint2 v = *reinterpret_cast<const uint2 *>(rp + 8 * k);
                    u[2 * k] = v.x;
                    u[2 * k + 1] = v.y;
                }
#pragma unroll
                for (int bp = 0; bp < 2; ++bp) {  // two blocks per tensor-memory store
                    uint32_t a[32];
#pragma unroll
                    for (int b2 = 0; b2 < 2; ++b2)
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            // even and odd codes, one per nibble; the byte permute
                            // reads only the selector's low 16 bits
                            const uint32_t w = block_word(u, 2 * bp + b2, c);
                            const uint32_t me = w & 0x33333333u, mo = (w >> 2) & 0x33333333u;
                            a[16 * b2 + 4 * c + 0] = __byte_perm(kS8Lut, 0u, me);
                            a[16 * b2 + 4 * c + 1] = __byte_perm(kS8Lut, 0u, mo);
                            a[16 * b2 + 4 * c + 2] = __byte_perm(kS8Lut, 0u, me >> 16);
                            a[16 * b2 + 4 * c + 3] = __byte_perm(kS8Lut, 0u, mo >> 16);
                        }
                    tmem_st32(tmem + lane_base + kS8ACol + (s & 1) * 128 + (4 * G + 2 * bp) * 16, a);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[s & 1]);
        }
    } else if (warp >= kEpiWarp0 && warp < kS8ExpWarp1) {
        // ------------------------------ epilogue ------------------------------
        // warp w: TMEM lane quarter q = w % 4 and accumulator buffer e = (w - 8) / 4,
        // i.e. the sub-stages g = s * kSub + ss with g % 2 == e. Each of the two
        // warps of a quarter sums its own sub-stages; at a tile's last stage warp
        // 12+q hands its sums to warp 8+q through s_pair, which adds them and
        // writes y. Every wait is bounded; a warp whose wait fails leaves the loop.
        const int qd = warp & 3, e = (warp - kEpiWarp0) >> 2;
        const int row = 32 * qd + lane;
        const uint32_t lane_base = uint32_t(32 * qd) << 16;
        float acc[NC], comp[NC];
#pragma unroll
        for (int j = 0; j < NC; ++j) acc[j] = comp[j] = 0.0f;
        bool ok = true;
        int n_tile_ends = 0;
        for (int s = 0; s < n_stages && ok; ++s) {
            const int st = s % kStages;
            const bool got = !*(volatile int *)&s_abort &&
                             mbar_wait(&full[st], stage_parity(s), p.err, kTagS8Full);
            if (!__all_sync(0xffffffffu, got)) {
                s_abort = 1;
                break;
            }
            const StageMeta m = s_meta[st];
            const uint8_t *rp = raw_ring + st * kRawBytes + row * kChunkBytes;
            const float *sc = reinterpret_cast<const float *>(act_ring + st * kSlot + kImg);
            float ssum[NC];
#pragma unroll
            for (int j = 0; j < NC; ++j) ssum[j] = 0.0f;
#pragma unroll 1
            for (int ss = 0; ss < kSub; ++ss) {
                const int g = s * kSub + ss;
                if ((g & 1) != e) continue;
                const bool have = mbar_wait(&d_full[e], uint32_t(g >> 1) & 1u, p.err,
                                            kTagS8DFull) &&
                                  !*(volatile int *)&s_abort;
                if (!__all_sync(0xffffffffu, have)) {
                    s_abort = 1;
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_base = tmem + lane_base + kS8DCol + e * 128;
                // kGB blocks' accumulators (at most 64 registers) per tensor-memory wait
#pragma unroll 1
                for (int gb = 0; gb < kBS; gb += kGB) {
                    uint32_t r[kGB][kN];
#pragma unroll
                    for (int bi = 0; bi < kGB; ++bi)
#pragma unroll
                        for (int q16 = 0; q16 < kN / 16; ++q16)
                            tmem_ld16(d_base + (gb + bi) * kN + 16 * q16,
                                      *reinterpret_cast<uint32_t(*)[16]>(&r[bi][16 * q16]));
                    tmem_wait_ld();
                    if (gb + kGB == kBS) {  // the sub-stage's accumulators are all read
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&d_empty[e]);
                    }
#pragma unroll
                    for (int bi = 0; bi < kGB; ++bi) {
                        const int b = ss * kBS + gb + bi;
                        const float d = lds_half_as_float(rp + 18 * b);
#pragma unroll
                        for (int j = 0; j < NC; ++j) {
                            const uint32_t *c = &r[bi][kS8Pieces * j];
                            float t = __uint_as_float(c[4]) * 0x1p-16f;
                            t = fmaf(__uint_as_float(c[3]), 0x1p-12f, t);
                            t = fmaf(__uint_as_float(c[2]), 0x1p-8f, t);
                            t = fmaf(__uint_as_float(c[1]), 0x1p-4f, t);
                            t = t + __uint_as_float(c[0]);
                            ssum[j] = fmaf(d * sc[b * NC + j], t, ssum[j]);
                        }
                    }
                }
            }
            if (!ok) break;
            // every epilogue warp releases every stage once it has read the stage's
            // record and d values (kept even without a sub-stage of its own, so
            // the slot is not refilled before both warps of a quarter read it)
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
#pragma unroll
            for (int j = 0; j < NC; ++j) {  // acc + comp += ssum (two-sum)
                const float sum = acc[j] + ssum[j];
                const float bb = sum - acc[j];
                comp[j] += (acc[j] - (sum - bb)) + (ssum[j] - bb);
                acc[j] = sum;
            }
            if (m.flags & kLastOfTile) {
                const int t = n_tile_ends++;
                if (e == 1) {
                    // wait until warp 8+q has read the previous tile's sums
                    const bool free_pair =
                        t == 0 || mbar_wait(&tile_w0[qd], uint32_t(t - 1) & 1u, p.err, kTagS8Pair);
                    if (!__all_sync(0xffffffffu, free_pair)) {
                        s_abort = 1;
                        break;
                    }
#pragma unroll
                    for (int j = 0; j < NC; ++j) {
                        s_pair[qd][lane][2 * j] = acc[j];
                        s_pair[qd][lane][2 * j + 1] = comp[j];
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tile_w1[qd]);
                } else {
                    const bool have = mbar_wait(&tile_w1[qd], uint32_t(t) & 1u, p.err, kTagS8Pair);
                    if (!__all_sync(0xffffffffu, have)) {
                        s_abort = 1;
                        break;
                    }
                    const int rr = m.row0 + row;
#pragma unroll
                    for (int j = 0; j < NC; ++j) {
                        const float o = s_pair[qd][lane][2 * j];
                        const float sum = acc[j] + o;
                        const float bb = sum - acc[j];
                        const float err = (acc[j] - (sum - bb)) + (o - bb);
                        const float yv = sum + (comp[j] + s_pair[qd][lane][2 * j + 1] + err);
                        if (rr < m.n_rows) m.y[size_t(j) * m.n_rows + rr] = yv;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tile_w0[qd]);
                }
#pragma unroll
                for (int j = 0; j < NC; ++j) acc[j] = comp[j] = 0.0f;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
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
bool g_t4_attr_done[64];

// Test hook (q2_0_test_inject_stall): a one-shot stall for the next fp4 mat-vec
// launch on a device.
std::mutex g_stall_mu;
int g_stall_stage[64];
unsigned long long g_stall_wait_ns[64];

void take_stall(MvParams &prm) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return;
    std::lock_guard<std::mutex> lk(g_stall_mu);
    if (g_stall_stage[dev] > 0) {
        prm.stall_stage = g_stall_stage[dev];
        prm.wait_ns = g_stall_wait_ns[dev];
        g_stall_stage[dev] = 0;
    }
}
bool g_s8_attr_done[64][9];

cudaError_t ensure_t4_attr() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (dev < 64 && g_t4_attr_done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(mv_t4_kernel<kLayBlocks>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             T4Lay<kLayBlocks>::kSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mv_t4_kernel<kLaySplit>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 T4Lay<kLaySplit>::kSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mv_t4_kernel<kLayG128>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 T4Lay<kLayG128>::kSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mv_t4_kernel<kLayBlocks, 2>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 T4Lay<kLayBlocks, 2>::kSmem);
    if (e == cudaSuccess && dev < 64) g_t4_attr_done[dev] = true;
    return e;
}

template <int NC>
cudaError_t launch_s8_nc(cudaLaunchConfig_t &cfg, const MvJob &single, const MvParams &prm) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(g_attr_mu);
        if (!(dev < 64 && g_s8_attr_done[dev][NC])) {
            e = cudaFuncSetAttribute(mv_s8_kernel<NC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     s8_smem(NC));
            if (e != cudaSuccess) return e;
            if (dev < 64) g_s8_attr_done[dev][NC] = true;
        }
    }
    cfg.blockDim = dim3(s8_threads(NC));
    cfg.dynamicSmemBytes = s8_smem(NC);
    return cudaLaunchKernelEx(&cfg, mv_s8_kernel<NC>, single, prm);
}

// ncols 1 and 2 run the fp4 kernel, ncols 3..8 the signed-e4m3 one.
bool use_t4(int ncols) { return ncols <= 2; }

bool make_job(MvJob &J, const uint8_t *w, const uint8_t *prep, float *y, int64_t N, int64_t K) {
    std::memset(&J, 0, sizeof(J));
    const uint64_t row_bytes = uint64_t(K / 64) * 18;
    if (!encode_tmap_2d(&J.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, row_bytes, uint64_t(N), row_bytes,
                        kChunkBytes, kTcRows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return false;
    J.prep = prep;
    J.y = y;
    J.N = int(N);
    J.nb = int(K / 64);
    J.n_chunks = int(K / 512);
    J.n_tiles = int((N + kTcRows - 1) / kTcRows);
    return true;
}

// The prep kernels are launched as programmatic dependents of whatever precedes
// them on the stream: their launch overlaps that kernel's tail, and they wait
// for it (griddepcontrol.wait) before reading x or writing their buffers.
// max_k: the largest K among the jobs (sets the grid's z extent).
// ctas (plans): n_ctas entries (job, first item), 128 items each, instead of the
// grid (.., n_jobs, z) sized by the largest K.
template <typename XT>
cudaError_t launch_prep_t(const MvPrepJob &single, const MvPrepJob *jobs, int n_jobs, int ncols,
                          int64_t max_k, cudaStream_t s, bool g128, const int2 *ctas,
                          int n_ctas) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(kPrepThreads);
    const int64_t items = max_k / 64 * (use_t4(ncols) ? 8 : 16);
    const unsigned z =
        ctas ? 1u : unsigned(std::min<int64_t>((items + kPrepThreads - 1) / kPrepThreads, 65535));
    const unsigned gy = unsigned(ctas ? n_ctas : n_jobs);
    if (use_t4(ncols)) {
        cfg.gridDim = dim3(ncols, gy, z);
        return g128 ? cudaLaunchKernelEx(&cfg, t4_prep_kernel<XT, true>, single, jobs, ctas, 1)
                    : cudaLaunchKernelEx(&cfg, t4_prep_kernel<XT, false>, single, jobs, ctas, ncols);
    }
    cfg.gridDim = dim3(ncols, gy, z);
    return cudaLaunchKernelEx(&cfg, s8_prep_kernel<XT>, single, jobs, ctas, ncols);
}

// g128: the fp4 preparation in 128-element scale blocks (the group-128 layout)
cudaError_t launch_prep(const MvPrepJob &single, const MvPrepJob *jobs, int n_jobs, int ncols,
                        int64_t max_k, int xtype, cudaStream_t s, bool g128 = false,
                        const int2 *ctas = nullptr, int n_ctas = 0) {
    return xtype == kXF16
               ? launch_prep_t<__half>(single, jobs, n_jobs, ncols, max_k, s, g128, ctas, n_ctas)
               : launch_prep_t<float>(single, jobs, n_jobs, ncols, max_k, s, g128, ctas, n_ctas);
}

// The tensor-core kernel is launched as a programmatic dependent of the prep
// kernel: its prologue and first weight loads overlap the prep's tail; its
// producer waits for the prep grid before loading any activation image.
cudaError_t launch_tc(const MvJob &single, const MvParams &prm, int grid, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (use_t4(prm.ncols)) {
        e = ensure_t4_attr();
        if (e != cudaSuccess) return e;
        cfg.blockDim = dim3(prm.ncols == 2 ? T4Lay<kLayBlocks, 2>::kThreads : kTcThreads);
        MvParams prm2 = prm;
        take_stall(prm2);
        if (prm2.layout == kLaySplit) {
            cfg.dynamicSmemBytes = T4Lay<kLaySplit>::kSmem;
            e = cudaLaunchKernelEx(&cfg, mv_t4_kernel<kLaySplit>, single, prm2);
        } else if (prm2.layout == kLayG128) {
            cfg.dynamicSmemBytes = T4Lay<kLayG128>::kSmem;
            e = cudaLaunchKernelEx(&cfg, mv_t4_kernel<kLayG128>, single, prm2);
        } else if (prm2.ncols == 2) {
            cfg.dynamicSmemBytes = T4Lay<kLayBlocks, 2>::kSmem;
            e = cudaLaunchKernelEx(&cfg, mv_t4_kernel<kLayBlocks, 2>, single, prm2);
        } else {
            cfg.dynamicSmemBytes = T4Lay<kLayBlocks>::kSmem;
            e = cudaLaunchKernelEx(&cfg, mv_t4_kernel<kLayBlocks>, single, prm2);
        }
    } else {
        switch (prm.ncols) {
            case 3: e = launch_s8_nc<3>(cfg, single, prm); break;
            case 4: e = launch_s8_nc<4>(cfg, single, prm); break;
            case 5: e = launch_s8_nc<5>(cfg, single, prm); break;
            case 6: e = launch_s8_nc<6>(cfg, single, prm); break;
            case 7: e = launch_s8_nc<7>(cfg, single, prm); break;
            default: e = launch_s8_nc<8>(cfg, single, prm); break;
        }
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
    return use_t4(ncols) ? t4_prep_bytes(K, ncols) : s8_prep_bytes(K, ncols);
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
    if (!make_job(J, w, prep, y, N, K)) return Q2_0_ECUDA;
    MvParams prm{nullptr, nullptr, nullptr, ncols, err};
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
                        128, kTcRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&J.tmap_d, CU_TENSOR_MAP_DATA_TYPE_UINT8, dsc, nb * 2, uint64_t(N), nb * 2,
                        16, kTcRows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return Q2_0_ECUDA;
    J.prep = prep;
    J.y = y;
    J.N = int(N);
    J.nb = int(nb);
    J.n_chunks = int(K / 512);
    J.n_tiles = int((N + kTcRows - 1) / kTcRows);
    MvParams prm{nullptr, nullptr, nullptr, 1, err, MvMoe{}, kLaySplit};
    const int grid = std::max(1, std::min(J.n_tiles, sm_count()));
    return cuda_status(launch_tc(J, prm, grid, s));
}

size_t matvec_g128_workspace_bytes(int64_t K, int ncols) {
    return ncols == 1 && K % 1024 == 0 ? g4_prep_bytes(K) : 0;
}

int matvec_g128_run(const uint8_t *w, const float *x, float *y, int64_t N, int64_t K, int ncols,
                    void *ws, size_t ws_bytes, cudaStream_t s) {
    if (matvec_g128_workspace_bytes(K, ncols) == 0 || (reinterpret_cast<uintptr_t>(w) & 15u) != 0)
        return cuda_status(launch_g128_generic(w, x, y, N, K, ncols, s));
    if (ws_bytes < g4_prep_bytes(K)) return Q2_0_EINVAL;
    unsigned long long *err = error_word_ptr();
    if (!err) return Q2_0_ECUDA;
    uint8_t *prep = static_cast<uint8_t *>(ws);
    MvPrepJob pj{x, prep, int(K)};
    if (launch_prep(pj, nullptr, 1, 1, K, kXF32, s, true) != cudaSuccess) return Q2_0_ECUDA;
    MvJob J;
    std::memset(&J, 0, sizeof(J));
    // rows of K / 128 * 34 bytes seen as 16-bit elements: a box of 136 elements
    // (one stage, 272 bytes) x 128 rows
    const uint64_t row_bytes = uint64_t(K / 128) * kG128Bytes;
    if (!encode_tmap_2d(&J.tmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, w, row_bytes / 2, uint64_t(N),
                        row_bytes, kG128RowBytes / 2, kTcRows, CU_TENSOR_MAP_SWIZZLE_NONE))
        return Q2_0_ECUDA;
    J.prep = prep;
    J.y = y;
    J.N = int(N);
    J.nb = int(K / 128);
    J.n_chunks = int(K / 1024);
    J.n_tiles = int((N + kTcRows - 1) / kTcRows);
    MvParams prm{nullptr, nullptr, nullptr, 1, err, MvMoe{}, kLayG128};
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
    if (!make_job(J, w, prep, y, n_expert * N, K)) return Q2_0_ECUDA;
    J.N = int(N);
    J.n_tiles = int((N + kTcRows - 1) / kTcRows);
    MvParams prm{nullptr, nullptr, nullptr, 1, err,
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
    q2::MvFirst *d_first = nullptr;  // [grid] each CTA's share of the schedule
    q2::MvPrepJob *d_prep_jobs = nullptr;
    int2 *d_prep_ctas = nullptr;  // the prep kernel's CTAs: (job, first item)
    int n_prep_ctas = 0;
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
    cudaFree(plan->d_first);
    cudaFree(plan->d_prep_jobs);
    cudaFree(plan->d_prep_ctas);
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
                          d.K))
                st = Q2_0_ECUDA;
            pjobs[j] = MvPrepJob{d.x, P->d_prep + off[j], int(d.K)};
            P->max_k = std::max<int64_t>(P->max_k, d.K);
        }
        // the prep kernel's CTAs: 128 items (fp4: 8 elements, e4m3: 4 elements
        // of one column) of one job each, so that no CTA of a short row idles
        std::vector<int2> pctas;
        for (int j = 0; j < P->n_fast; ++j) {
            const int64_t n_it = use_t4(ncols) ? descs[fast[j]].K / 8 : descs[fast[j]].K / 4;
            for (int64_t i0 = 0; i0 < n_it; i0 += kPrepThreads) pctas.push_back(make_int2(j, int(i0)));
        }
        P->n_prep_ctas = int(pctas.size());
        if (st == Q2_0_OK && (pctas.size() > 65535 ||
                              cudaMalloc(&P->d_prep_ctas, sizeof(int2) * pctas.size()) != cudaSuccess ||
                              cudaMemcpy(P->d_prep_ctas, pctas.data(), sizeof(int2) * pctas.size(),
                                         cudaMemcpyHostToDevice) != cudaSuccess))
            st = pctas.size() > 65535 ? Q2_0_EINVAL : Q2_0_ECUDA;
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
        std::vector<MvFirst> first(grid, MvFirst{});
        for (int c = 0; c < grid; ++c) {
            MvFirst &f = first[c];
            f.item_base = begin[c];
            f.n_items = begin[c + 1] - begin[c];
            f.n_stages = stages[c];
            if (f.n_items > 0) {
                f.job0 = flat[begin[c]].job;
                f.tile0 = flat[begin[c]].tile;
                const MvJob &j0 = jobs[f.job0];
                f.n_chunks0 = j0.n_chunks;
                f.n0 = j0.N;
                f.prep0 = j0.prep;
                f.y0 = j0.y;
            }
        }
        if (st == Q2_0_OK &&
            (cudaMalloc(&P->d_jobs, sizeof(MvJob) * jobs.size()) != cudaSuccess ||
             cudaMalloc(&P->d_items, sizeof(MvItem) * flat.size()) != cudaSuccess ||
             cudaMalloc(&P->d_first, sizeof(MvFirst) * first.size()) != cudaSuccess ||
             cudaMalloc(&P->d_prep_jobs, sizeof(MvPrepJob) * pjobs.size()) != cudaSuccess))
            st = Q2_0_ECUDA;
        if (st == Q2_0_OK &&
            (cudaMemcpy(P->d_jobs, jobs.data(), sizeof(MvJob) * jobs.size(),
                        cudaMemcpyHostToDevice) != cudaSuccess ||
             cudaMemcpy(P->d_items, flat.data(), sizeof(MvItem) * flat.size(),
                        cudaMemcpyHostToDevice) != cudaSuccess ||
             cudaMemcpy(P->d_first, first.data(), sizeof(MvFirst) * first.size(),
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
        if (launch_prep(none, P->d_prep_jobs, P->n_fast, P->ncols, P->max_k, kXF32, s, false,
                        P->d_prep_ctas, P->n_prep_ctas) != cudaSuccess)
            return Q2_0_ECUDA;
        MvJob dummy;
        std::memset(&dummy, 0, sizeof(dummy));
        MvParams prm{P->d_jobs, P->d_items, P->d_first, P->ncols, P->err};
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

// Test hook: the next fp4 mat-vec launch (ncols = 1 on the tensor-core path) on
// the current device stops feeding its pipeline before the given stage, and
// every pipeline wait of that launch gives up after wait_limit_ns.
extern "C" int q2_0_test_inject_stall(int stage, uint64_t wait_limit_ns) {
    int dev = 0;
    if (stage < 0 || wait_limit_ns == 0 || wait_limit_ns > 10000000000ull) return Q2_0_EINVAL;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q2_0_ECUDA;
    if (dev < 0 || dev >= 64) return Q2_0_EUNSUPPORTED;
    std::lock_guard<std::mutex> lk(q2::g_stall_mu);
    q2::g_stall_stage[dev] = stage + 1;
    q2::g_stall_wait_ns[dev] = wait_limit_ns;
    return Q2_0_OK;
}
