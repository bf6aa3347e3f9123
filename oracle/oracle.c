/*
 * oracle.c -- plain, slow, obviously correct CPU oracle for the q4_K x q8_1
 * quantized GEMM (MMQ).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only tests/, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA path.  Build flags (see oracle/__init__.py): -O2 -fno-fast-math
 * -ffp-contract=off, OpenMP over output rows.
 *
 * Sources (web pages on the method):
 *  [r15]  "20 . r15 -- f32-accumulate mma probe (dead end) + rank-1 term2
 *          rescale", section 2.1 "Where the two-term rescale comes from"
 *          (q8_1 fields da/sa, q4_K fields d, dmin, sc, m, v; S_ij; the two
 *          terms; dsv = d*sc, dmv = -dmin*m) and section 2.3 (|S| bound
 *          32*127*15, per-sub-block get_scale_min_k4 semantics).
 *  [r16]  "21 . r16 -- Narrow kernel gets the rank-1 fold", section 2.1
 *          (the fold dma = da*sa; a re-association only).
 *
 * Readings where the pages are silent:
 *  - q8_1 scale da is f32 (the pages store f16); da = amax/127 with IEEE
 *    round-to-nearest division; q = clamp(roundf(x/da), -127, 127) with
 *    roundf = round half away from zero; when da == 0 every q is 0 and sa = 0.
 *  - q4_K byte layout: the customary 144-byte super-block (fp16 d, fp16
 *    dmin, 12 bytes of packed 6-bit sc/m, 128 bytes of nibbles), see
 *    oracle_unpack_q4K below.
 *  - C is overwritten (beta = 0), row-major [M][N], f32 rounded once from a
 *    double accumulation.
 *
 * Pins (tests/test_oracle_pins.py): closed forms for constant, zero, one-hot,
 * alternating and tie blocks; hand-set scale bytes; pack/unpack round trip;
 * S against numpy int64 einsum; worked single-block examples E1..E5; the
 * identity C == dot(dequant(A), dequant(B)) on brute-force tiny inputs.
 * Every function here has at least one pin; none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK 32          /* elements per q8_1 block and per q4_K sub-block */
#define QKK 256        /* elements per q4_K super-block                   */
#define Q4K_BYTES 144  /* bytes per q4_K super-block                      */

/* IEEE binary16 bits -> double, written out from the format definition
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits). */
static double half_to_double(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 31;
    const int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                /* subnormal: f * 2^-24   */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);    /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* ---------------------------------------------------------------------------
 * O1  q8_1 quantize ([r15] 2.1: every 32 activations get a scale da and the
 *     sum sa of their integer quants, both written by the quantize pass).
 *     Oracle layout: q [M][K] int8, da [M][K/32] f32, sa [M][K/32] int32.
 * ------------------------------------------------------------------------- */
void oracle_quantize_q8_1(const float* x, int64_t M, int64_t K,
                          int8_t* q, float* da, int32_t* sa) {
    const int64_t nb = K / QK;
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < M; i++) {
        for (int64_t b = 0; b < nb; b++) {
            const float* xb = x + i * K + b * QK;
            float amax = 0.0f;
            for (int k = 0; k < QK; k++) {
                const float a = fabsf(xb[k]);
                if (a > amax) amax = a;
            }
            const float d = amax / 127.0f;
            int32_t s = 0;
            for (int k = 0; k < QK; k++) {
                int qk = 0;
                if (d != 0.0f) {
                    const float r = roundf(xb[k] / d);
                    qk = (int)r;
                    if (qk > 127) qk = 127;
                    if (qk < -127) qk = -127;
                }
                q[i * K + b * QK + k] = (int8_t)qk;
                s += qk;
            }
            da[i * nb + b] = d;
            sa[i * nb + b] = s;
        }
    }
}

/* ---------------------------------------------------------------------------
 * O2  q4_K unpack of one super-block ([r15] 2.1: fp16 d and dmin per
 *     super-block; 6-bit sc and m per 32-element sub-block, decoded the way
 *     get_scale_min_k4 decodes them; v in [0,15]).  Customary 144-byte layout:
 *       bytes 0-1  d (fp16, little endian)     bytes 2-3  dmin (fp16)
 *       bytes 4-15 s[0..11]: for c < 4:  sc = s[c] & 63,  m = s[c+4] & 63
 *                            for c >= 4: sc = (s[c+4] & 15) | (s[c-4] >> 6) << 4
 *                                        m  = (s[c+4] >> 4) | (s[c]   >> 6) << 4
 *       bytes 16-143: element e = 64p + 32h + l (p = 0..3, h = 0..1,
 *                     l = 0..31) is nibble h (0 = low) of byte 16 + 32p + l.
 * ------------------------------------------------------------------------- */
static void unpack_superblock(const uint8_t* blk, double* d, double* dmin,
                              uint8_t sc[8], uint8_t m[8], uint8_t v[QKK]) {
    *d = half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
    *dmin = half_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
    const uint8_t* s = blk + 4;
    for (int c = 0; c < 8; c++) {
        if (c < 4) {
            sc[c] = s[c] & 63;
            m[c] = s[c + 4] & 63;
        } else {
            sc[c] = (uint8_t)((s[c + 4] & 15) | ((s[c - 4] >> 6) << 4));
            m[c] = (uint8_t)((s[c + 4] >> 4) | ((s[c] >> 6) << 4));
        }
    }
    const uint8_t* qb = blk + 16;
    for (int e = 0; e < QKK; e++) {
        const int p = e / 64, h = (e / 32) % 2, l = e % 32;
        const uint8_t byte = qb[32 * p + l];
        v[e] = h ? (byte >> 4) : (byte & 15);
    }
}

/* Whole-matrix unpack: blk [N][K/256][144] -> d, dmin [N][K/256] (double,
 * exact), sc, m [N][K/32], v [N][K]. */
void oracle_unpack_q4K(const uint8_t* blk, int64_t N, int64_t K,
                       double* d, double* dmin, uint8_t* sc, uint8_t* m,
                       uint8_t* v) {
    const int64_t nsb = K / QKK;
    for (int64_t j = 0; j < N; j++)
        for (int64_t b = 0; b < nsb; b++)
            unpack_superblock(blk + (j * nsb + b) * Q4K_BYTES,
                              d + j * nsb + b, dmin + j * nsb + b,
                              sc + j * (K / QK) + b * 8, m + j * (K / QK) + b * 8,
                              v + j * K + b * QKK);
}

/* Dequantized weight w_jk = d*sc*v - dmin*m ([r15] 2.1: the weight a q4_K
 * code stands for), in double, [N][K]. */
void oracle_dequant_q4K(const uint8_t* blk, int64_t N, int64_t K, double* w) {
    const int64_t nsb = K / QKK;
    int64_t j;
#pragma omp parallel for schedule(static)
    for (j = 0; j < N; j++) {
        double d, dmin;
        uint8_t sc[8], m[8], v[QKK];
        for (int64_t b = 0; b < nsb; b++) {
            unpack_superblock(blk + (j * nsb + b) * Q4K_BYTES, &d, &dmin, sc, m, v);
            for (int e = 0; e < QKK; e++) {
                const int c = e / QK;
                w[j * K + b * QKK + e] = d * sc[c] * v[e] - dmin * m[c];
            }
        }
    }
}

/* ---------------------------------------------------------------------------
 * O3  exact per-32-k block dots ([r15] 2.1: S_ij = sum_k a_int[i,k] * v[j,k]
 *     per chunk).  S [M][N][K/32] int32.
 * ------------------------------------------------------------------------- */
void oracle_block_dots(const int8_t* q, const uint8_t* blk, int64_t M,
                       int64_t N, int64_t K, int32_t* S) {
    const int64_t nsb = K / QKK, nb = K / QK;
    uint8_t* v = (uint8_t*)malloc((size_t)(N * K));
    double* dd = (double*)malloc((size_t)(N * nsb) * sizeof(double));
    double* dm = (double*)malloc((size_t)(N * nsb) * sizeof(double));
    uint8_t* sc = (uint8_t*)malloc((size_t)(N * nb));
    uint8_t* m = (uint8_t*)malloc((size_t)(N * nb));
    oracle_unpack_q4K(blk, N, K, dd, dm, sc, m, v);
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < M; i++)
        for (int64_t j = 0; j < N; j++)
            for (int64_t c = 0; c < nb; c++) {
                int32_t s = 0;
                for (int l = 0; l < QK; l++)
                    s += (int32_t)q[i * K + c * QK + l] * (int32_t)v[j * K + c * QK + l];
                S[(i * N + j) * nb + c] = s;
            }
    free(v); free(dd); free(dm); free(sc); free(m);
}

/* ---------------------------------------------------------------------------
 * O4  the GEMM, per output (i, j), chunk by chunk in k order ([r15] 2.1):
 *       C_ij = sum_c [ da_ic * dsv_jc * S_ijc + dmv_jc * (da_ic * sa_ic) ]
 *     with dsv = d*sc and dmv = -dmin*m, accumulated in double and rounded
 *     once to f32.
 * O5  the tolerance scale T_ij = sum_k |(da_ic * q_ik) * w_jk| in double.
 * Both for a list of n (row, col) pairs, so full-size runs can be sampled.
 * ------------------------------------------------------------------------- */
static void gemm_one(const int8_t* q, const float* da, const int32_t* sa,
                     const uint8_t* blk, int64_t N, int64_t K, int64_t i,
                     int64_t j, float* C, double* C64, double* T) {
    (void)N;
    const int64_t nsb = K / QKK, nb = K / QK;
    double acc = 0.0, tol = 0.0;
    double d, dmin;
    uint8_t sc[8], m[8], v[QKK];
    for (int64_t b = 0; b < nsb; b++) {
        unpack_superblock(blk + (j * nsb + b) * Q4K_BYTES, &d, &dmin, sc, m, v);
        for (int c8 = 0; c8 < 8; c8++) {
            const int64_t c = b * 8 + c8;
            int32_t S = 0;
            for (int l = 0; l < QK; l++)
                S += (int32_t)q[i * K + c * QK + l] * (int32_t)v[c8 * QK + l];
            const double dsv = d * (double)sc[c8];
            const double dmv = -(dmin * (double)m[c8]);
            const double a_d = (double)da[i * nb + c];
            const double a_s = (double)sa[i * nb + c];
            acc += a_d * dsv * (double)S + dmv * (a_d * a_s);
            if (T) {
                for (int l = 0; l < QK; l++) {
                    const double w = d * sc[c8] * v[c8 * QK + l] - dmin * m[c8];
                    tol += fabs((a_d * (double)q[i * K + c * QK + l]) * w);
                }
            }
        }
    }
    if (C) *C = (float)acc;
    if (C64) *C64 = acc;
    if (T) *T = tol;
}

void oracle_gemm_sampled(const int8_t* q, const float* da, const int32_t* sa,
                         const uint8_t* blk, int64_t M, int64_t N, int64_t K,
                         int64_t n, const int64_t* rows, const int64_t* cols,
                         float* C, double* C64, double* T) {
    (void)M;
    int64_t t;
#pragma omp parallel for schedule(dynamic, 16)
    for (t = 0; t < n; t++)
        gemm_one(q, da, sa, blk, N, K, rows[t], cols[t],
                 C ? C + t : NULL, C64 ? C64 + t : NULL, T ? T + t : NULL);
}

/* Full GEMM: C [M][N] f32 (and optionally C64, T [M][N] double). */
void oracle_gemm(const int8_t* q, const float* da, const int32_t* sa,
                 const uint8_t* blk, int64_t M, int64_t N, int64_t K,
                 float* C, double* C64, double* T) {
    int64_t i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < M; i++)
        for (int64_t j = 0; j < N; j++)
            gemm_one(q, da, sa, blk, N, K, i, j, C ? C + i * N + j : NULL,
                     C64 ? C64 + i * N + j : NULL, T ? T + i * N + j : NULL);
}

/* ---------------------------------------------------------------------------
 * O6  brute-force identity (tiny shapes): D_ij = sum_k (da_ic*q_ik) * w_jk in
 *     double, i.e. dot(dequant(A), dequant(B)) with no blockwise structure.
 * ------------------------------------------------------------------------- */
void oracle_dequant_dot(const int8_t* q, const float* da, const uint8_t* blk,
                        int64_t M, int64_t N, int64_t K, double* D) {
    const int64_t nb = K / QK;
    double* w = (double*)malloc((size_t)(N * K) * sizeof(double));
    oracle_dequant_q4K(blk, N, K, w);
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < M; i++)
        for (int64_t j = 0; j < N; j++) {
            double s = 0.0;
            for (int64_t k = 0; k < K; k++)
                s += ((double)da[i * nb + k / QK] * (double)q[i * K + k]) * w[j * K + k];
            D[i * N + j] = s;
        }
    free(w);
}
