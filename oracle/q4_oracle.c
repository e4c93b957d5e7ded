/*
 * q4_oracle.c -- plain, slow, obviously correct CPU oracle for the int4
 * weight-streaming GEMV / matmul and the dense f32 GEMV control.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  The CUDA
 * library shares no code, header, table or helper with it, and neither
 * imports the other.
 *
 * What it computes (restated from the pages, in this file's own words):
 *
 *   gerbil GPU-engine kernel reference (docs/gpu-engine/kernels.md),
 *   section "3. MatMulInt4":
 *     - "Computes": C[M,N] = A[M,K] * dequant(B_q), one output element is a
 *       plain dot product over K.
 *     - "INT4 Packing": a nibble at position pos of a packed word is
 *       (word >> 4*pos) & 0xF, so the lowest nibble is the first element.
 *     - "Dequantization": value = (nibble - zero[group]) * scale[group].
 *
 *   Refractometer page, sweep "b) q4 GEMV": the weights are in the
 *   MatMulNBits layout -- one row per output feature n, packed along K,
 *   groups of g consecutive k inside one row, fp16 scales and packed 4-bit
 *   zero points.
 *
 * Readings taken where the pages are silent or disagree (each is listed in
 * the design notes): the weight is [N][K] (row n = output feature); groups
 * run along K inside a row; scales are fp16 [N][K/g]; zero points are
 * 4-bit, two per byte with the even group in the low nibble, each row padded
 * to ceil((K/g)/2) bytes (the pad nibble is ignored); a missing zero-point
 * array means the symmetric variant with zero = 8.
 *
 * Arithmetic: a dequantised weight (q - z) * s is formed in binary32.  It is
 * exact: |q - z| <= 15 needs 4 bits and an fp16 scale has an 11-bit
 * significand, so the product fits in binary32's 24 bits.  Dot products are
 * accumulated in binary64 in plain k order and rounded once to binary32.
 * The tolerance bound sum_k |w_nk * x_mk| is accumulated in binary64 too.
 *
 * Plain C99, no threads, no vector intrinsics, no blocking or reordering.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* ---------------------------------------------------------------------- */
/* Number formats, from their IEEE 754 / bfloat16 definitions.            */
/* ---------------------------------------------------------------------- */

/* IEEE 754 binary16 -> value.  sign | 5-bit exponent (bias 15) | 10-bit
 * fraction.  Exponent 0 is subnormal: fraction * 2^-24.  Exponent 31 is
 * Inf/NaN.  Otherwise (1024 + fraction) * 2^(exponent - 25).  Every binary16
 * value is exactly representable in binary32, so the final cast is exact. */
float orc_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25);
    return (float)(sign ? -v : v);
}

/* bfloat16 is the upper half of a binary32 bit pattern. */
float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bfloat16, round to nearest, ties to even.  The dropped low 16
 * bits are compared with one half of the kept unit in the last place; on an
 * exact tie the kept pattern is rounded to the even one.  NaN stays a quiet
 * NaN. */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u; /* a carry into the exponent is the correct rounding */
    return (uint16_t)kept;
}

/* ---------------------------------------------------------------------- */
/* Layout accessors.                                                      */
/* ---------------------------------------------------------------------- */

/* Code q[n][k]: row n holds K/2 bytes; byte k/2 holds element k in its low
 * nibble when k is even and in its high nibble when k is odd. */
int orc_q4_code(const uint8_t *codes, int64_t K, int64_t n, int64_t k)
{
    uint8_t byte = codes[n * (K / 2) + k / 2];
    return (k % 2 == 0) ? (byte & 0x0f) : (byte >> 4);
}

/* Zero point z[n][b] for group b of row n.  Row n holds ceil(nb/2) bytes;
 * group b sits in byte b/2, low nibble for even b.  NULL: symmetric, 8. */
int orc_q4_zero(const uint8_t *zeros, int64_t nb, int64_t n, int64_t b)
{
    if (zeros == NULL)
        return 8;
    int64_t row_bytes = (nb + 1) / 2;
    uint8_t byte = zeros[n * row_bytes + b / 2];
    return (b % 2 == 0) ? (byte & 0x0f) : (byte >> 4);
}

/* Scale s[n][b] as a value. */
float orc_q4_scale(const uint16_t *scales, int64_t nb, int64_t n, int64_t b)
{
    return orc_f16_to_f32(scales[n * nb + b]);
}

/* ---------------------------------------------------------------------- */
/* The method.                                                            */
/* ---------------------------------------------------------------------- */

/* One dequantised weight: (q - z) * s in binary32 (exact, see header). */
float orc_q4_weight(const uint8_t *codes, const uint16_t *scales,
                    const uint8_t *zeros, int64_t K, int64_t g,
                    int64_t n, int64_t k)
{
    int64_t nb = K / g;
    int64_t b = k / g;
    int q = orc_q4_code(codes, K, n, k);
    int z = orc_q4_zero(zeros, nb, n, b);
    float s = orc_q4_scale(scales, nb, n, b);
    return (float)(q - z) * s;
}

/* W[n][k] = (q - z) * s for the whole matrix, row-major [N][K]. */
void orc_q4_dequant(const uint8_t *codes, const uint16_t *scales,
                    const uint8_t *zeros, int64_t N, int64_t K, int64_t g,
                    float *w)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = orc_q4_weight(codes, scales, zeros, K, g, n, k);
}

/* The bfloat16 tile a tensor-core path feeds its MMA with: each exact
 * binary32 weight rounded once to bfloat16 (nearest, ties to even). */
void orc_q4_dequant_bf16(const uint8_t *codes, const uint16_t *scales,
                         const uint8_t *zeros, int64_t N, int64_t K,
                         int64_t g, uint16_t *wb)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            wb[n * K + k] = orc_f32_to_bf16(
                orc_q4_weight(codes, scales, zeros, K, g, n, k));
}

/* y[m][n] = sum_k W[n][k] * x[m][k]   (x row-major [M][K], y [M][N]).
 * bound[m][n] = sum_k |W[n][k] * x[m][k]|, both accumulated in binary64 in
 * k order; y is rounded once to binary32.  bound may be NULL. */
void orc_q4_gemv(const uint8_t *codes, const uint16_t *scales,
                 const uint8_t *zeros, const float *x, int64_t M, int64_t N,
                 int64_t K, int64_t g, float *y, double *bound)
{
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double w = (double)orc_q4_weight(codes, scales, zeros, K, g, n, k);
                double p = w * (double)x[m * K + k];
                acc += p;
                mag += fabs(p);
            }
            y[m * N + n] = (float)acc;
            if (bound)
                bound[m * N + n] = mag;
        }
    }
}

/* The tensor-core-shaped matmul: C[m][n] = sum_k W[n][k] * A[m][k] with A
 * given as bfloat16 [M][K] (widened exactly to binary32), output binary32. */
void orc_q4_gemm(const uint8_t *codes, const uint16_t *scales,
                 const uint8_t *zeros, const uint16_t *a_bf16, int64_t M,
                 int64_t N, int64_t K, int64_t g, float *c, double *bound)
{
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double w = (double)orc_q4_weight(codes, scales, zeros, K, g, n, k);
                double p = w * (double)orc_bf16_to_f32(a_bf16[m * K + k]);
                acc += p;
                mag += fabs(p);
            }
            c[m * N + n] = (float)acc;
            if (bound)
                bound[m * N + n] = mag;
        }
    }
}

/* Dense control (cera wgpu_gemv_bench.rs, the F32 "control" row):
 * y[m][n] = sum_k W[n][k] * x[m][k], W row-major [N][K] binary32. */
void orc_f32_gemv(const float *W, const float *x, int64_t M, int64_t N,
                  int64_t K, float *y, double *bound)
{
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = (double)W[n * K + k] * (double)x[m * K + k];
                acc += p;
                mag += fabs(p);
            }
            y[m * N + n] = (float)acc;
            if (bound)
                bound[m * N + n] = mag;
        }
    }
}

/* ---------------------------------------------------------------------- */
/* The fused decode variants (the prologue and epilogue of a projection). */
/* ---------------------------------------------------------------------- */

/* gerbil GPU-engine kernel reference, section "4. RMSNorm", "Computes": each
 * row of the input is divided by its root mean square, rms(v) =
 * sqrt(mean(v^2) + eps), and multiplied elementwise by the weight vector.
 * xn[m][k] = x[m][k] / rms(x[m][:]) * gamma[k], all in binary64 (the sum of
 * squares in k order), nothing rounded. */
void orc_rmsnorm(const float *x, const float *gamma, double eps, int64_t M,
                 int64_t K, double *xn)
{
    for (int64_t m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double v = (double)x[m * K + k];
            ss += v * v;
        }
        double rms = sqrt(ss / (double)K + eps);
        for (int64_t k = 0; k < K; ++k)
            xn[m * K + k] = (double)x[m * K + k] / rms * (double)gamma[k];
    }
}

/* The GEMV of section "3. MatMulInt4" on a binary64 input (the normalised
 * activations of the fused variant): y[m][n] = sum_k W[n][k] * x[m][k] and
 * bound[m][n] = sum_k |W[n][k] * x[m][k]|, binary64 in k order, unrounded. */
void orc_q4_gemv_f64(const uint8_t *codes, const uint16_t *scales,
                     const uint8_t *zeros, const double *x, int64_t M,
                     int64_t N, int64_t K, int64_t g, double *y, double *bound)
{
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double w = (double)orc_q4_weight(codes, scales, zeros, K, g, n, k);
                double p = w * x[m * K + k];
                acc += p;
                mag += fabs(p);
            }
            y[m * N + n] = acc;
            bound[m * N + n] = mag;
        }
    }
}

/* Section "9. SiLU", "Computes": silu(v) = v / (1 + exp(-v)); its
 * optimisation notes name the SwiGLU combine, out = silu(gate) * up. */
double orc_silu(double v)
{
    return v / (1.0 + exp(-v));
}

void orc_swiglu(const double *gate, const double *up, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_silu(gate[i]) * up[i];
}

/* ---------------------------------------------------------------------- */
/* A second format: 32-element blocks of 18 bytes.                        */
/* ---------------------------------------------------------------------- */

/* cera wgpu_gemv_bench.rs, block geometry: Q4_0 holds 32 elements in 18 bytes.
 * Read here as: a binary16 scale d (bytes 0-1, little-endian), then 16 bytes of
 * 4-bit codes with element 2j in the low nibble of byte 2 + j and element 2j + 1
 * in the high nibble (the INT4 packing of the kernel reference page), zero point 8
 * (the symmetric convention).  A row of K elements is K/32 consecutive blocks.
 * w[n][k] = (q - 8) * d, exact in binary32 as for the MatMulNBits weights. */
float orc_q40_weight(const uint8_t *blocks, int64_t K, int64_t n, int64_t k)
{
    const uint8_t *blk = blocks + (n * (K / 32) + k / 32) * 18;
    uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
    int64_t e = k % 32;
    uint8_t byte = blk[2 + e / 2];
    int q = (e % 2 == 0) ? (byte & 0x0f) : (byte >> 4);
    return (float)(q - 8) * orc_f16_to_f32(dbits);
}

/* y[m][n] = sum_k W[n][k] * x[m][k] over Q4_0 weights; bound as for the GEMV. */
void orc_q40_gemv(const uint8_t *blocks, const float *x, int64_t M, int64_t N,
                  int64_t K, float *y, double *bound)
{
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = (double)orc_q40_weight(blocks, K, n, k) * (double)x[m * K + k];
                acc += p;
                mag += fabs(p);
            }
            y[m * N + n] = (float)acc;
            if (bound)
                bound[m * N + n] = mag;
        }
    }
}

/* ---------------------------------------------------------------------- */
/* A third format: 32-element blocks of 34 bytes.                         */
/* ---------------------------------------------------------------------- */

/* cera wgpu_gemv_bench.rs, block geometry: Q8_0 holds 32 elements in 34 bytes.
 * Read here as: a binary16 scale d (bytes 0-1, little-endian, as for Q4_0), then
 * 32 signed 8-bit codes in two's complement, element j of the block at byte 2 + j;
 * no zero point.  A row of K elements is K/32 consecutive blocks.
 * w[n][k] = q * d: |q| <= 128 (8 bits) times an 11-bit significand is exact in
 * binary32. */
float orc_q80_weight(const uint8_t *blocks, int64_t K, int64_t n, int64_t k)
{
    const uint8_t *blk = blocks + (n * (K / 32) + k / 32) * 34;
    uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
    int q = blk[2 + k % 32];
    if (q >= 128)
        q -= 256;
    return (float)q * orc_f16_to_f32(dbits);
}

/* y[m][n] = sum_k W[n][k] * x[m][k] over Q8_0 weights; bound as for the GEMV. */
void orc_q80_gemv(const uint8_t *blocks, const float *x, int64_t M, int64_t N,
                  int64_t K, float *y, double *bound)
{
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = (double)orc_q80_weight(blocks, K, n, k) * (double)x[m * K + k];
                acc += p;
                mag += fabs(p);
            }
            y[m * N + n] = (float)acc;
            if (bound)
                bound[m * N + n] = mag;
        }
    }
}

/* Read probe (webgpu-bench README, "read-bandwidth"; Refractometer
 * "a) bandwidth"): the sum of every binary32 element of a buffer, in
 * binary64.  The probe kernel's own partial sums are compared against it. */
double orc_sum_f32(const float *buf, int64_t n)
{
    double acc = 0.0;
    for (int64_t i = 0; i < n; ++i)
        acc += (double)buf[i];
    return acc;
}
