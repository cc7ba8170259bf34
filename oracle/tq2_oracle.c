/*
 * CPU oracle for the TQ2_0_g128 ternary matmul.  TEST INFRASTRUCTURE ONLY:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library.  It shares no code, header, table or helper with the
 * CUDA library; it is a plain, slow, obviously-correct restatement of the
 * definition, in double precision.
 *
 * What it follows:
 *  - "oxibonsai-image 0.2.2 src/gpu.rs", module doc "Correctness contract":
 *    for row-major input[M,K], out-major weight blocks [N, K/128] and
 *    out[M,N], out[m,n] = sum_k input[m,k] * dequant(W)[n,k]  (an A.B^T
 *    contraction, no transpose of the operands).
 *  - same page, doc of `blocks_as_bytes` and test
 *    `block_is_thirty_four_bytes`: a block is 34 bytes, qs[32] then d:f16,
 *    no padding, little endian.
 *  - the code convention of the library (not printed on the pages): code c
 *    in {0,1,2} means weight c-1; weight j of a block sits in bits
 *    2*(j%4)..2*(j%4)+1 of qs[j/4].  Code 3 is never generated; this oracle
 *    decodes it arithmetically (c-1 = +2).
 *  - the optional residual is added after the contraction:
 *    out = x.W^T + residual (the "_residual" decode kernels listed on the
 *    "oxibonsai-kernels 0.1.5 src/gpu_backend/metal_graph/pipelines.rs" page
 *    have no TQ2 counterpart there; this is the plain reading).
 *  - the struct-of-arrays layout is this library's own definition (the pages
 *    only name an "SoA weight buffer"): the qs plane [N][K/4] bytes followed by
 *    the d plane [N][K/128] binary16 values; block (n,b) keeps its qs bytes at
 *    (n*(K/128)+b)*32 and its two d bytes at N*K/4 + (n*(K/128)+b)*2.
 *
 *  - the encoder (f32 weights -> blocks) is this library's reading, because
 *    the pages never show how the blocks are produced (they are read from a
 *    GGUF file): the absmean rule of ternary weights, with every step that
 *    decides a code fixed (see tq2o_quantize below).
 *
 * Everything is computed in IEEE double; the binary16 scale is decoded from
 * its bits by hand (no compiler half type).  Rows of the output are spread
 * over OpenMP threads when the build has OpenMP; the arithmetic per element is
 * the same plain loop over k either way.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define TQ2O_BLOCK_W 128
#define TQ2O_BLOCK_BYTES 34
#define TQ2O_QS_BYTES 32

/* IEEE 754 binary16 -> double, exactly: sign, 5-bit exponent (bias 15),
 * 10-bit fraction; exponent 0 is subnormal (no implicit 1), 31 is Inf/NaN. */
double tq2o_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* f * 2^-10 * 2^-14 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* The scale of one 34-byte block: bytes 32 (low) and 33 (high). */
static double block_scale(const uint8_t *blk) {
    uint16_t bits = (uint16_t)(blk[TQ2O_QS_BYTES] | ((uint16_t)blk[TQ2O_QS_BYTES + 1] << 8));
    return tq2o_half_to_double(bits);
}

/* Code of weight j (0..127) of one block, in {0,1,2,3}. */
static int block_code(const uint8_t *blk, int j) {
    return (blk[j / 4] >> (2 * (j % 4))) & 3;
}

int tq2o_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void tq2o_set_threads(int t) {
#ifdef _OPENMP
    if (t > 0) omp_set_num_threads(t);
#else
    (void)t;
#endif
}

/* Dequantised weight row n as doubles: w[k] = (code - 1) * d. */
static void dequant_row(const uint8_t *w_aos, int64_t n, int64_t k, double *w) {
    int64_t kb = k / TQ2O_BLOCK_W;
    for (int64_t b = 0; b < kb; ++b) {
        const uint8_t *blk = w_aos + (n * kb + b) * TQ2O_BLOCK_BYTES;
        double d = block_scale(blk);
        for (int j = 0; j < TQ2O_BLOCK_W; ++j) {
            w[b * TQ2O_BLOCK_W + j] = (double)(block_code(blk, j) - 1) * d;
        }
    }
}

/* Dense dequantised weight, double [N, K]. Returns 0, or -1 if k % 128. */
int tq2o_dequant(const uint8_t *w_aos, int64_t n, int64_t k, double *w) {
    if (k <= 0 || k % TQ2O_BLOCK_W) return -1;
    for (int64_t r = 0; r < n; ++r) dequant_row(w_aos, r, k, w + r * k);
    return 0;
}

/*
 * out[i, c] = sum_k x[rows[i], k] * dequant(W)[c, k]  (+ residual[rows[i], c])
 * absdot[i, c] = sum_k |x[rows[i], k] * dequant(W)[c, k]|
 * for i in [0, n_rows) and c in [0, n).  `rows` may be NULL (then rows[i]=i and
 * n_rows = m).  x is float32 [m, k] row-major, residual float32 [m, n] or NULL,
 * out and absdot double [n_rows, n] (absdot may be NULL).
 * Returns 0, or -1 if k is not a positive multiple of 128.
 */
int tq2o_matmul(const uint8_t *w_aos, const float *x, const float *residual,
                int64_t m, int64_t n, int64_t k, const int64_t *rows, int64_t n_rows,
                double *out, double *absdot) {
    if (k <= 0 || k % TQ2O_BLOCK_W) return -1;
    if (!rows) n_rows = m;
    int failed = 0;
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)k);
        if (!w) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
        for (int64_t c = 0; c < n; ++c) {
            if (!w) continue;
            dequant_row(w_aos, c, k, w);
            for (int64_t i = 0; i < n_rows; ++i) {
                int64_t r = rows ? rows[i] : i;
                const float *xr = x + r * k;
                double acc = 0.0, acc_abs = 0.0;
                for (int64_t kk = 0; kk < k; ++kk) {
                    double p = (double)xr[kk] * w[kk];
                    acc += p;
                    acc_abs += fabs(p);
                }
                if (residual) acc += (double)residual[r * n + c];
                out[i * n + c] = acc;
                if (absdot) absdot[i * n + c] = acc_abs;
            }
        }
        free(w);
    }
    return failed ? -2 : 0;
}

/* Bytes of one weight in either layout: N * (K/128) * 34. */
int64_t tq2o_weight_bytes(int64_t n, int64_t k) { return n * (k / TQ2O_BLOCK_W) * TQ2O_BLOCK_BYTES; }

/* AoS [N][K/128]{qs[32], d} -> SoA (qs plane [N][K/4], then d plane [N][K/128]). */
int tq2o_aos_to_soa(const uint8_t *aos, uint8_t *soa, int64_t n, int64_t k) {
    if (k <= 0 || k % TQ2O_BLOCK_W) return -1;
    int64_t nblk = n * (k / TQ2O_BLOCK_W);
    uint8_t *qs_plane = soa;
    uint8_t *d_plane = soa + nblk * TQ2O_QS_BYTES;
    for (int64_t i = 0; i < nblk; ++i) {
        const uint8_t *blk = aos + i * TQ2O_BLOCK_BYTES;
        for (int j = 0; j < TQ2O_QS_BYTES; ++j) qs_plane[i * TQ2O_QS_BYTES + j] = blk[j];
        d_plane[i * 2 + 0] = blk[TQ2O_QS_BYTES + 0];
        d_plane[i * 2 + 1] = blk[TQ2O_QS_BYTES + 1];
    }
    return 0;
}

/* Inverse of tq2o_aos_to_soa. */
int tq2o_soa_to_aos(const uint8_t *soa, uint8_t *aos, int64_t n, int64_t k) {
    if (k <= 0 || k % TQ2O_BLOCK_W) return -1;
    int64_t nblk = n * (k / TQ2O_BLOCK_W);
    const uint8_t *qs_plane = soa;
    const uint8_t *d_plane = soa + nblk * TQ2O_QS_BYTES;
    for (int64_t i = 0; i < nblk; ++i) {
        uint8_t *blk = aos + i * TQ2O_BLOCK_BYTES;
        for (int j = 0; j < TQ2O_QS_BYTES; ++j) blk[j] = qs_plane[i * TQ2O_QS_BYTES + j];
        blk[TQ2O_QS_BYTES + 0] = d_plane[i * 2 + 0];
        blk[TQ2O_QS_BYTES + 1] = d_plane[i * 2 + 1];
    }
    return 0;
}

/* double -> IEEE binary16 bits, round to nearest even, by hand: values at or
 * above 65520 (halfway past the largest finite 65504) become Inf; magnitudes at
 * or below 2^-25 become (signed) zero; subnormals keep the 2^-24 step. */
uint16_t tq2o_double_to_half(double v) {
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v)) return 0x7e00;
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: integer multiple of 2^-24 (1024 carries into the
         * smallest normal, which is the right encoding) */
        double f = nearbyint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)f);
    }
    int ex;
    frexp(a, &ex); /* a = m * 2^ex, m in [0.5, 1): the unbiased exponent is ex - 1 */
    int e = ex - 1;
    double r = nearbyint(ldexp(a, 10 - e)); /* in [1024, 2048] */
    if (r >= 2048.0) {
        r = 1024.0;
        e += 1;
    }
    if (e > 15) return (uint16_t)(sign | 0x7c00);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(r - 1024.0));
}

/* Encoder: f32 weights w[n][k] (row-major) -> AoS blocks [n][k/128] of 34
 * bytes.  For each 128-weight block (the absmean rule of ternary weights):
 *   gamma = (sum_{j=0..127} |w_j|) / 128, the sum in double in index order;
 *   d     = binary16(gamma), round to nearest even;
 *   q_j   = rint(w_j / (float)d) in binary32 (IEEE division, ties to even),
 *           clamped to [-1, 1]; code c_j = q_j + 1 (weight j at bits
 *           2*(j%4) of qs[j/4]).
 * A zero or non-finite d gives code 1 (weight 0) everywhere.  Returns -1 for
 * a k that is not a positive multiple of 128. */
int tq2o_quantize(const float *w, int64_t n, int64_t k, uint8_t *aos) {
    if (k <= 0 || k % TQ2O_BLOCK_W) return -1;
    const int64_t nb = k / TQ2O_BLOCK_W;
    int64_t r;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (r = 0; r < n; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *wb = w + r * k + b * TQ2O_BLOCK_W;
            double s = 0.0;
            for (int j = 0; j < TQ2O_BLOCK_W; ++j) s += fabs((double)wb[j]);
            const uint16_t dh = tq2o_double_to_half(s / 128.0);
            const double dd = tq2o_half_to_double(dh);
            const int live = dd > 0.0 && isfinite(dd);
            const float df = (float)dd; /* exact: a binary16 value */
            uint8_t *blk = aos + (r * nb + b) * TQ2O_BLOCK_BYTES;
            memset(blk, 0, TQ2O_QS_BYTES);
            for (int j = 0; j < TQ2O_BLOCK_W; ++j) {
                int c = 1;
                if (live) {
                    const float q = rintf(wb[j] / df);
                    c = q >= 1.0f ? 2 : (q <= -1.0f ? 0 : 1);
                }
                blk[j / 4] |= (uint8_t)(c << (2 * (j % 4)));
            }
            blk[TQ2O_QS_BYTES + 0] = (uint8_t)(dh & 0xff);
            blk[TQ2O_QS_BYTES + 1] = (uint8_t)(dh >> 8);
        }
    }
    return 0;
}
