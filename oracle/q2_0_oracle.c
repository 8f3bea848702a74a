/*
 * Q2_0 oracle — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of what the Q2_0 kernels compute. Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may load it;
 * the product library never does. It shares no code, header, table or constant
 * with the CUDA sources.
 *
 * Sources (web pages; cited by title and section):
 *   [WGPU]  "WebGPU: add Q2_0 support" (bisque.today write-up of llama.cpp
 *           PR 30914) — the block-format paragraph, the get-rows / tiled-matmul /
 *           mat-vec shader paragraph and the mat-vec kernel excerpt.
 *   [AISV]  "Llama.cpp umí dvoubitový Q2_0 i na kartách NVIDIA" (aisvetem.cz),
 *           sections "Osmnáct bajtů na čtyřiašedesát vah" (block layout, code
 *           table), "Šest procent, o která se vedl spor" (group-64 vs group-128)
 *           and "Na běžný model to není" (reference quantizer rule).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - words are little-endian u32; element 16*w+i is bits 2i..2i+1 of word w;
 *   - code 3 decodes by the same rule, to +2d;
 *   - the quantizer's decisions use the unrounded block max |w|; the stored
 *     scale is that max rounded to fp16 (round to nearest, ties to even);
 *     ties between two levels go away from zero; an all-zero block stores d=0
 *     and code 1 everywhere.
 *
 * Every function is reentrant; the only parallelism is an optional OpenMP loop
 * over independent output rows, which leaves each row's summation order as
 * written.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QO_WEIGHTS_PER_BLOCK 64 /* [AISV] "Osmnáct bajtů…": groups of 64 weights */
#define QO_BYTES_PER_BLOCK 18   /* 2-byte fp16 scale + 64 two-bit codes (16 bytes) */

int qo_weights_per_block(void) { return QO_WEIGHTS_PER_BLOCK; }
int qo_bytes_per_block(void) { return QO_BYTES_PER_BLOCK; }

int qo_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void qo_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---------------------------------------------------------------------------
 * IEEE 754 binary16, written from the format definition: 1 sign bit, 5 exponent
 * bits with bias 15, 10 fraction bits; exponent 0 holds zero and subnormals
 * (fraction * 2^-24), exponent 31 holds infinities and NaNs.
 * ------------------------------------------------------------------------- */
double qo_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp(1024.0 + (double)frac, expo - 25); /* (1 + frac/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Round a binary32 value to binary16, round-to-nearest, ties-to-even; values
 * whose magnitude rounds past the largest finite half (65504) become infinity. */
uint16_t qo_float_to_half_rn(float f) {
    double a = (double)f;
    uint16_t sign = 0;
    if (signbit(a)) {
        sign = 0x8000;
        a = -a;
    }
    if (isnan(a)) return (uint16_t)(sign | 0x7e00);
    if (isinf(a)) return (uint16_t)(sign | 0x7c00);
    if (a == 0.0) return sign;
    int e2;
    (void)frexp(a, &e2); /* a = m * 2^e2 with m in [0.5, 1): unbiased exponent e2-1 */
    int e = e2 - 1;
    if (e < -14) {
        /* subnormal range: units of 2^-24; the scaled value is exact in double */
        double units = ldexp(a, 24);
        double r = nearbyint(units); /* default rounding mode: nearest-even */
        /* r == 1024 lands exactly on the smallest normal, whose code is 0x0400 */
        return (uint16_t)(sign | (uint16_t)r);
    }
    double mant = ldexp(a, 10 - e); /* in [1024, 2048) */
    double r = nearbyint(mant);
    if (r == 2048.0) {
        r = 1024.0;
        e += 1;
    }
    if (e > 15) return (uint16_t)(sign | 0x7c00);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)((int)r - 1024));
}

/* ---------------------------------------------------------------------------
 * Block decode. [WGPU] format paragraph and [AISV] "Osmnáct bajtů…": the first
 * two bytes are the fp16 scale d; the other 16 bytes are four 32-bit words of
 * sixteen 2-bit codes; code q decodes to (q - 1) * d. The mat-vec excerpt of
 * [WGPU] reads word t at byte offset 2 + 4t and shifts code i out of bits 2i.
 * ------------------------------------------------------------------------- */
static uint32_t qo_word_le(const uint8_t *p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
           ((uint32_t)p[3] << 24);
}

uint16_t qo_block_scale_bits(const uint8_t *blk) {
    return (uint16_t)(blk[0] | (blk[1] << 8));
}

int qo_block_code(const uint8_t *blk, int e) {
    int w = e / 16, i = e % 16;
    uint32_t word = qo_word_le(blk + 2 + 4 * w);
    return (int)((word >> (2 * i)) & 3u);
}

/* out[e] = (q_e - 1) * d for e < 64, in fp64 (exact). */
void qo_decode_block(const uint8_t *blk, double *out) {
    double d = qo_half_to_double(qo_block_scale_bits(blk));
    for (int e = 0; e < QO_WEIGHTS_PER_BLOCK; ++e)
        out[e] = (double)(qo_block_code(blk, e) - 1) * d;
}

/* Codes of one block, one per element (0..3). */
void qo_block_codes(const uint8_t *blk, uint8_t *codes) {
    for (int e = 0; e < QO_WEIGHTS_PER_BLOCK; ++e) codes[e] = (uint8_t)qo_block_code(blk, e);
}

/* Dequantize rows [r0, r0+nr) of an N x K matrix into fp64, row-major. */
void qo_dequantize_rows(const uint8_t *w, int64_t K, int64_t r0, int64_t nr, double *out) {
    int64_t nb = K / QO_WEIGHTS_PER_BLOCK;
    for (int64_t r = 0; r < nr; ++r)
        for (int64_t b = 0; b < nb; ++b)
            qo_decode_block(w + ((r0 + r) * nb + b) * QO_BYTES_PER_BLOCK,
                            out + r * K + b * QO_WEIGHTS_PER_BLOCK);
}

/* ---------------------------------------------------------------------------
 * Dequantize-then-dot in fp64 (the plain definition of the product that the
 * mat-vec and the GEMM compute): for each activation column c and each listed
 * weight row n,
 *     y[c][n]   = sum_k W[n][k] * x[c][k]
 *     acc[c][n] = sum_k |W[n][k] * x[c][k]|   (the scale of the tolerance)
 * x is f32 [ncols][K] row-major; y and acc are fp64 [ncols][n_rows_listed].
 * Each product (q-1)*d*x is exact in fp64 (2 + 11 + 24 significant bits).
 * rows == NULL means all rows 0..N-1.
 * ------------------------------------------------------------------------- */
void qo_matmul_rows(const uint8_t *w, int64_t N, int64_t K, const float *x, int64_t ncols,
                    const int64_t *rows, int64_t n_rows, double *y, double *acc) {
    (void)N;
    int64_t nr = rows ? n_rows : N;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < nr; ++j) {
        int64_t n = rows ? rows[j] : j;
        double wrow[QO_WEIGHTS_PER_BLOCK];
        int64_t nb = K / QO_WEIGHTS_PER_BLOCK;
        for (int64_t c = 0; c < ncols; ++c) {
            double s = 0.0, a = 0.0;
            const float *xc = x + c * K;
            for (int64_t b = 0; b < nb; ++b) {
                qo_decode_block(w + (n * nb + b) * QO_BYTES_PER_BLOCK, wrow);
                for (int e = 0; e < QO_WEIGHTS_PER_BLOCK; ++e) {
                    double t = wrow[e] * (double)xc[b * QO_WEIGHTS_PER_BLOCK + e];
                    s += t;
                    a += fabs(t);
                }
            }
            y[c * nr + j] = s;
            if (acc) acc[c * nr + j] = a;
        }
    }
}

/* ---------------------------------------------------------------------------
 * Expert mat-vec (ggml mul_mat_id). [WGPU] limitations paragraph: the port
 * leaves out MUL_MAT_ID, the expert-routed matmul of mixture-of-experts layers.
 * as holds n_expert matrices of N x K one after another; ids is
 * [n_tokens][n_used]; x is [n_tokens][n_x][K] with n_x = 1 (one vector per
 * token, shared by its experts) or n_x = n_used (one vector per slot).
 *   y[t][i][j] = sum_k W_{ids[t][i]}[rows[j]][k] * x[t][n_x == 1 ? 0 : i][k]
 * in fp64, with acc = sum |W x| likewise; y and acc are [n_tokens*n_used][nr].
 * Each slot is the plain matmul above on the selected matrix. Returns the
 * number of ids outside [0, n_expert); their y and acc rows are left untouched.
 * ------------------------------------------------------------------------- */
int64_t qo_matmul_id(const uint8_t *as, int64_t n_expert, int64_t N, int64_t K, const float *x,
                     int64_t n_x, const int32_t *ids, int64_t n_used, int64_t n_tokens,
                     const int64_t *rows, int64_t n_rows, double *y, double *acc) {
    int64_t bad = 0;
    int64_t nr = rows ? n_rows : N;
    size_t expert_bytes = (size_t)N * (size_t)(K / QO_WEIGHTS_PER_BLOCK) * QO_BYTES_PER_BLOCK;
    for (int64_t t = 0; t < n_tokens; ++t) {
        for (int64_t i = 0; i < n_used; ++i) {
            int64_t v = t * n_used + i;
            int64_t e = ids[v];
            if (e < 0 || e >= n_expert) {
                ++bad;
                continue;
            }
            const float *xv = x + (t * n_x + (n_x == 1 ? 0 : i)) * K;
            qo_matmul_rows(as + (size_t)e * expert_bytes, N, K, xv, 1, rows, n_rows, y + v * nr,
                           acc ? acc + v * nr : NULL);
        }
    }
    return bad;
}

/* ---------------------------------------------------------------------------
 * Split (structure-of-arrays) layout. [KOPI] "Why the weight has to stay
 * quantized" splits a block format's scales from its quants into separate
 * arrays when loading; for Q2_0 that gives, for an N x K matrix with
 * nb = K/64 blocks per row:
 *   qs[n][b][16]  the 16 code bytes of block (n, b), row-major;
 *   d[n][b]       its 2-byte little-endian fp16 scale, row-major;
 * with d starting qs_bytes_padded = round_up(N*nb*16, 256) bytes after qs.
 * The split moves bytes only; soa_to_raw is its inverse.
 * ------------------------------------------------------------------------- */
int64_t qo_soa_bytes(int64_t N, int64_t K) {
    int64_t nb = K / QO_WEIGHTS_PER_BLOCK;
    int64_t qs = (N * nb * 16 + 255) / 256 * 256;
    int64_t d = (N * nb * 2 + 255) / 256 * 256;
    return qs + d;
}

void qo_raw_to_soa(const uint8_t *w, int64_t N, int64_t K, uint8_t *soa) {
    int64_t nb = K / QO_WEIGHTS_PER_BLOCK;
    int64_t nblk = N * nb;
    uint8_t *qs = soa;
    uint8_t *d = soa + (nblk * 16 + 255) / 256 * 256;
    for (int64_t i = 0; i < nblk; ++i) {
        const uint8_t *blk = w + i * QO_BYTES_PER_BLOCK;
        d[2 * i] = blk[0];
        d[2 * i + 1] = blk[1];
        memcpy(qs + 16 * i, blk + 2, 16);
    }
}

void qo_soa_to_raw(const uint8_t *soa, int64_t N, int64_t K, uint8_t *w) {
    int64_t nb = K / QO_WEIGHTS_PER_BLOCK;
    int64_t nblk = N * nb;
    const uint8_t *qs = soa;
    const uint8_t *d = soa + (nblk * 16 + 255) / 256 * 256;
    for (int64_t i = 0; i < nblk; ++i) {
        uint8_t *blk = w + i * QO_BYTES_PER_BLOCK;
        blk[0] = d[2 * i];
        blk[1] = d[2 * i + 1];
        memcpy(blk + 2, qs + 16 * i, 16);
    }
}

/* ---------------------------------------------------------------------------
 * get_rows. [WGPU] shader paragraph: the get-rows shader copies rows of a Q2_0
 * tensor out and writes 64 floats per block. out[r][k] = W[ids[r]][k] as f32;
 * (q-1)*d is exact in fp64 and representable in f32, so the cast is exact and
 * keeps IEEE signed zeros. Returns the number of ids outside [0, n_rows); their
 * output rows are left untouched.
 * ------------------------------------------------------------------------- */
int64_t qo_get_rows(const uint8_t *table, int64_t n_rows, int64_t K, const int32_t *ids,
                    int64_t n_ids, float *out) {
    int64_t bad = 0;
    int64_t nb = K / QO_WEIGHTS_PER_BLOCK;
    for (int64_t r = 0; r < n_ids; ++r) {
        int64_t id = ids[r];
        if (id < 0 || id >= n_rows) {
            ++bad;
            continue;
        }
        double blk[QO_WEIGHTS_PER_BLOCK];
        for (int64_t b = 0; b < nb; ++b) {
            qo_decode_block(table + (id * nb + b) * QO_BYTES_PER_BLOCK, blk);
            for (int e = 0; e < QO_WEIGHTS_PER_BLOCK; ++e)
                out[r * K + b * QO_WEIGHTS_PER_BLOCK + e] = (float)blk[e];
        }
    }
    return bad;
}

/* ---------------------------------------------------------------------------
 * Reference quantizer. [AISV] "Na běžný model to není": the reference
 * quantizer takes the block's largest absolute value as the scale and rounds
 * each weight to the nearest of the four levels (q-1)*scale, q = 0..3.
 * With |w| <= amax the candidates are -amax (q=0), 0 (q=1), +amax (q=2); the
 * midpoints are -amax/2 and +amax/2. The comparisons 2w >= amax and
 * 2w <= -amax are exact in fp64. Ties go away from zero. amax = 0 gives d = 0
 * and q = 1 for every weight. Code 3 is never produced.
 * ------------------------------------------------------------------------- */
void qo_quantize_block(const float *src, uint8_t *blk) {
    double amax = 0.0;
    for (int e = 0; e < QO_WEIGHTS_PER_BLOCK; ++e) {
        double a = fabs((double)src[e]);
        if (a > amax) amax = a;
    }
    uint16_t d = qo_float_to_half_rn((float)amax);
    memset(blk, 0, QO_BYTES_PER_BLOCK);
    blk[0] = (uint8_t)(d & 0xff);
    blk[1] = (uint8_t)(d >> 8);
    for (int e = 0; e < QO_WEIGHTS_PER_BLOCK; ++e) {
        double w2 = 2.0 * (double)src[e];
        int q;
        if (amax == 0.0) q = 1;
        else if (w2 >= amax) q = 2;
        else if (w2 <= -amax) q = 0;
        else q = 1;
        int wi = e / 16, i = e % 16;
        uint32_t word = qo_word_le(blk + 2 + 4 * wi);
        word |= (uint32_t)q << (2 * i);
        uint8_t *p = blk + 2 + 4 * wi;
        p[0] = (uint8_t)(word & 0xff);
        p[1] = (uint8_t)((word >> 8) & 0xff);
        p[2] = (uint8_t)((word >> 16) & 0xff);
        p[3] = (uint8_t)((word >> 24) & 0xff);
    }
}

void qo_quantize_rows(const float *src, int64_t nrows, int64_t K, uint8_t *dst) {
    int64_t nb = K / QO_WEIGHTS_PER_BLOCK;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; ++r)
        for (int64_t b = 0; b < nb; ++b)
            qo_quantize_block(src + r * K + b * QO_WEIGHTS_PER_BLOCK,
                              dst + (r * nb + b) * QO_BYTES_PER_BLOCK);
}

/* ---------------------------------------------------------------------------
 * Group-128 blocks. [AISV] "Šest procent, o která se vedl spor": the packing the
 * format's authors use for their own models has 128 weights per block, 34 bytes
 * (2.125 bits per weight); its closing section: files named Q2_0.gguf without
 * the _g64 suffix are that older packing. The pages give only the size. Reading
 * (parity unpinned by the pages beyond the size): the group-64 layout extended
 * to 128 weights — fp16 scale at +0, then eight little-endian 32-bit words;
 * element 16w+i is bits 2i..2i+1 of word w; code q decodes to (q - 1) * d.
 * ------------------------------------------------------------------------- */
#define QO_G128_WEIGHTS 128
#define QO_G128_BYTES 34

void qo_decode_block_g128(const uint8_t *blk, double *out) {
    double d = qo_half_to_double(qo_block_scale_bits(blk));
    for (int e = 0; e < QO_G128_WEIGHTS; ++e) {
        int w = e / 16, i = e % 16;
        uint32_t word = qo_word_le(blk + 2 + 4 * w);
        out[e] = (double)((int)((word >> (2 * i)) & 3u) - 1) * d;
    }
}

/* As qo_matmul_rows for an N x K group-128 matrix (K % 128 == 0). */
void qo_matmul_rows_g128(const uint8_t *w, int64_t N, int64_t K, const float *x, int64_t ncols,
                         const int64_t *rows, int64_t n_rows, double *y, double *acc) {
    int64_t nr = rows ? n_rows : N;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < nr; ++j) {
        int64_t n = rows ? rows[j] : j;
        double wrow[QO_G128_WEIGHTS];
        int64_t nb = K / QO_G128_WEIGHTS;
        for (int64_t c = 0; c < ncols; ++c) {
            double s = 0.0, a = 0.0;
            const float *xc = x + c * K;
            for (int64_t b = 0; b < nb; ++b) {
                qo_decode_block_g128(w + (n * nb + b) * QO_G128_BYTES, wrow);
                for (int e = 0; e < QO_G128_WEIGHTS; ++e) {
                    double t = wrow[e] * (double)xc[b * QO_G128_WEIGHTS + e];
                    s += t;
                    a += fabs(t);
                }
            }
            y[c * nr + j] = s;
            if (acc) acc[c * nr + j] = a;
        }
    }
}

/* As qo_get_rows for a group-128 table. */
int64_t qo_get_rows_g128(const uint8_t *table, int64_t n_rows, int64_t K, const int32_t *ids,
                         int64_t n_ids, float *out) {
    int64_t bad = 0;
    int64_t nb = K / QO_G128_WEIGHTS;
    for (int64_t r = 0; r < n_ids; ++r) {
        int64_t id = ids[r];
        if (id < 0 || id >= n_rows) {
            ++bad;
            continue;
        }
        double blk[QO_G128_WEIGHTS];
        for (int64_t b = 0; b < nb; ++b) {
            qo_decode_block_g128(table + (id * nb + b) * QO_G128_BYTES, blk);
            for (int e = 0; e < QO_G128_WEIGHTS; ++e)
                out[r * K + b * QO_G128_WEIGHTS + e] = (float)blk[e];
        }
    }
    return bad;
}

/* Packed size of an N x K matrix at a given group size, from the layout: one
 * fp16 scale (2 bytes) plus group/4 bytes of 2-bit codes per group. [AISV]
 * "Šest procent…": 34 bytes per 128 weights vs 18 per 64. */
int64_t qo_packed_bytes(int64_t N, int64_t K, int64_t group) {
    return N * (K / group) * (2 + group / 4);
}

/* Array forms of the two codec functions (for exhaustive checks). */
void qo_half_to_double_array(const uint16_t *h, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = qo_half_to_double(h[i]);
}

void qo_float_to_half_rn_array(const float *f, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = qo_float_to_half_rn(f[i]);
}
