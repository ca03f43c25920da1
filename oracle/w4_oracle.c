/*
 * w4_oracle.c -- plain, slow CPU oracle for group-wise int4 weight-only
 * quantization and the mixed bf16 x int4 linear, and for the same affine
 * path at 2 and 8 bits.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this code:
 * only the test-suite, the smoke check and the CPU-baseline leg of the
 * benchmark load it.  It shares no code, header, table or constant with the
 * CUDA library; the only thing both sides share is the seeded input
 * generator, which holds none of the method's arithmetic.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC.
 * Rows are independent, so the row loops may run on several threads (OpenMP,
 * w4_ref_threads); each row is still computed sequentially in the order
 * written, so results do not depend on the thread count.
 * On x86-64 float arithmetic is IEEE binary32 with round-to-nearest-even, and
 * -ffp-contract=off forbids fusing a*b+c, so every float operation below is
 * exactly one correctly rounded IEEE operation.
 *
 * What the pages fix, and where:
 *  - weights below 8 bits are projected group-wise and affinely, with an
 *    offset ("zero point"):  Optimum Quanto, "Design overview / Tensors";
 *  - the integer mapping is plain rounding, torch.round(), which rounds half
 *    to even:  Optimum Quanto, "Design overview / Tensors";
 *  - the projection aims to avoid saturated and flushed values, so the whole
 *    [min, max] of a group maps onto the code range:  same section;
 *  - weights are grouped along their first axis (output features), i.e. the
 *    groups of W[N,K] run along K inside one output row:  Optimum Quanto,
 *    "Design overview / Modules" and "Pitfalls when quantizing activations";
 *  - group sizes 32 / 64 / 128:  torchao README "Quick start"; torchao guide
 *    section 3.1; TorchAO 0.14.0 release notes "Deprecations";
 *  - the matmul result is accumulated at higher precision than its inputs:
 *    Optimum Quanto, "Pitfalls when quantizing activations";
 *  - weights of 2, 4 and 8 bits:  Optimum Quanto, feature list ("int2, int4,
 *    int8 and float8 weights"); int8 weights in groups of 128:  torchao
 *    README, the diffusers example (Int8WeightOnlyConfig, PerGroup(128));
 *  - int8 activations quantized at run time beside int4 group-wise weights:
 *    torchao's Int8DynamicActivationInt4WeightConfig (README, guide); one
 *    symmetric scale per tensor:  Optimum Quanto, "Design overview / Modules".
 * The concrete formulas (scale = (max-min)/15 with an eps clamp,
 * q = clamp(rne((w-min)/scale), 0, 15), w' = q*scale + min) are the plainest
 * reading consistent with all of the above; the readings of points the pages
 * leave open (eps value, stored-scale coding, -0 ordering, nibble order) are
 * marked "reading" below.  At b bits the same steps run with L = 2^b - 1
 * levels in place of 15 (reading: the pages give the bit widths, not their
 * formulas; the affine path with the full code range is the plainest one),
 * and 8/b codes share a byte, the code of the lowest k in the lowest bits.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#include <omp.h>

/* reading: the pages say nothing about the clamp; 1e-6 (fp32) keeps the
 * clamp inactive for every non-constant group of realistic weights. */
#define REF_EPS 1e-6f

/* ---- bf16 <-> fp32 ---------------------------------------------------- */

/* A bf16 value is the top 16 bits of the fp32 value: exact widening. */
static float ref_bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round an fp32 value to the nearest bf16, ties to even.  The format is
 * sign-magnitude, so rounding the 32-bit pattern at bit 16 rounds the
 * magnitude; a carry out of the mantissa correctly bumps the exponent. */
static uint16_t ref_float_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u); /* keep NaN a (quiet) NaN */
    uint32_t upper = u >> 16;
    uint32_t rest = u & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)upper;
}

/* Total order used for the group min / max: the usual < on finite values,
 * and -0.0 below +0.0 (reading: the pages leave the choice between two equal
 * zeros open; this one makes the result independent of scan order). */
static int ref_less(float a, float b)
{
    if (a < b)
        return 1;
    if (a == 0.0f && b == 0.0f)
        return signbit(a) && !signbit(b);
    return 0;
}

static int ref_group_ok(int64_t N, int64_t K, int g)
{
    if (g != 32 && g != 64 && g != 128)
        return 0;
    if (N < 0 || K <= 0 || K % g != 0)
        return 0;
    return 1;
}

/* Code widths of the affine path: 2, 4 or 8 bits. */
static int ref_bits_ok(int bits)
{
    return bits == 2 || bits == 4 || bits == 8;
}

/* ---- quantize --------------------------------------------------------- */

/*
 * W[N,K] bf16 (row-major)  ->  Wq[N,K*b/8] packed codes, scales[N,K/g] bf16,
 * offsets[N,K/g] bf16, with L = 2^b - 1.  For each row n and each group j of
 * g consecutive k, in this order:
 *   1. mn, mx = min and max of the group (ref_less order);
 *   2. s32 = (mx - mn) / L, two IEEE fp32 operations;
 *   3. s32 = eps if s32 < eps;
 *   4. s = bf16(s32): the stored scale; the codes are computed with it
 *      (reading: coding with the stored scale keeps w' self-consistent);
 *   5. o = mn, stored as bf16 (exact, mn already is a bf16 value);
 *   6. q = clamp(round_half_even((w - o) / s), 0, L), fp32 subtract and
 *      divide, then rintf() in the default round-to-nearest-even mode;
 *   7. the 8/b codes k = (8/b) p .. (8/b) p + 8/b - 1 share byte p of the
 *      row, code k at bit b (k mod 8/b): at 4 bits even k in the low nibble
 *      (reading: the pages name packing formats but define none).
 * Returns 0, or -1 on an unsupported shape or width.
 */
int w4_ref_quantize_bits(const uint16_t *W, int64_t N, int64_t K, int g, int bits,
                         uint8_t *Wq, uint16_t *scales, uint16_t *offsets)
{
    if (!ref_group_ok(N, K, g) || !ref_bits_ok(bits))
        return -1;
    const int levels = (1 << bits) - 1;
    const int per_byte = 8 / bits;
    const int64_t row_bytes = K / per_byte;
    const int64_t groups = K / g;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t j = 0; j < groups; ++j) {
            const uint16_t *wg = W + n * K + j * g;
            float mn = ref_bf16_to_float(wg[0]);
            float mx = mn;
            for (int i = 1; i < g; ++i) {
                float v = ref_bf16_to_float(wg[i]);
                if (ref_less(v, mn))
                    mn = v;
                if (ref_less(mx, v))
                    mx = v;
            }
            float range = mx - mn;
            float s32 = range / (float)levels;
            if (s32 < REF_EPS)
                s32 = REF_EPS;
            uint16_t s_bits = ref_float_to_bf16(s32);
            uint16_t o_bits = ref_float_to_bf16(mn);
            float s = ref_bf16_to_float(s_bits);
            float o = ref_bf16_to_float(o_bits);
            scales[n * groups + j] = s_bits;
            offsets[n * groups + j] = o_bits;
            for (int i = 0; i < g; ++i) {
                float v = ref_bf16_to_float(wg[i]);
                float d = v - o;
                float t = d / s;
                float r = rintf(t);
                int q = (int)r;
                if (q < 0)
                    q = 0;
                if (q > levels)
                    q = levels;
                int64_t k = j * g + i;
                uint8_t *byte = Wq + n * row_bytes + k / per_byte;
                int shift = (int)(k % per_byte) * bits;
                if (shift == 0)
                    *byte = (uint8_t)q;
                else
                    *byte = (uint8_t)(*byte | (q << shift));
            }
        }
    }
    return 0;
}

/* The int4 case: two codes a byte, even k in the low nibble. */
int w4_ref_quantize(const uint16_t *W, int64_t N, int64_t K, int g,
                    uint8_t *Wq, uint16_t *scales, uint16_t *offsets)
{
    return w4_ref_quantize_bits(W, N, K, g, 4, Wq, scales, offsets);
}

/* ---- dequantize ------------------------------------------------------- */

/* One weight: w' = bf16( fp32(q) * s + o ), one fp32 multiply (exact: an
 * integer of at most 8 bits times an 8-bit significand), one fp32 add, then
 * rounding to bf16.  Optimum Quanto, "Pitfalls when quantizing activations":
 * the result of the quantized matmul is brought back to float. */
static uint16_t ref_dequant_one(const uint8_t *Wq, const uint16_t *scales,
                                const uint16_t *offsets, int64_t K, int g,
                                int bits, int64_t n, int64_t k)
{
    const int per_byte = 8 / bits;
    uint8_t byte = Wq[n * (K / per_byte) + k / per_byte];
    int q = (byte >> ((int)(k % per_byte) * bits)) & ((1 << bits) - 1);
    float s = ref_bf16_to_float(scales[n * (K / g) + k / g]);
    float o = ref_bf16_to_float(offsets[n * (K / g) + k / g]);
    float t = (float)q * s;
    float u = t + o;
    return ref_float_to_bf16(u);
}

int w4_ref_dequantize_bits(const uint8_t *Wq, const uint16_t *scales,
                           const uint16_t *offsets, int64_t N, int64_t K, int g,
                           int bits, uint16_t *W_out)
{
    if (!ref_group_ok(N, K, g) || !ref_bits_ok(bits))
        return -1;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            W_out[n * K + k] = ref_dequant_one(Wq, scales, offsets, K, g, bits, n, k);
    return 0;
}

int w4_ref_dequantize(const uint8_t *Wq, const uint16_t *scales,
                      const uint16_t *offsets, int64_t N, int64_t K, int g,
                      uint16_t *W_out)
{
    return w4_ref_dequantize_bits(Wq, scales, offsets, N, K, g, 4, W_out);
}

/* ---- linear ----------------------------------------------------------- */

/*
 * Y[m,n] = sum_k X[m,k] * W'[n,k] in fp64, with W' the bf16 dequantized
 * weights of w4_ref_dequantize: the reference value y_ref of the tolerance
 * |y - y_ref| <= 4e-3 |y_ref| + 1e-2 rms(y_ref).  Y is fp64 [M,N].
 */
int w4_ref_linear_bits(const uint16_t *X, int64_t M, int64_t K, const uint8_t *Wq,
                       const uint16_t *scales, const uint16_t *offsets, int64_t N,
                       int g, int bits, double *Y)
{
    if (!ref_group_ok(N, K, g) || !ref_bits_ok(bits) || M < 0)
        return -1;
    /* one dequantized row per thread */
    const int nt = omp_get_max_threads();
    double *wbuf = (double *)malloc((size_t)nt * (size_t)K * sizeof(double));
    if (wbuf == NULL)
        return -2;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        double *wrow = wbuf + (size_t)omp_get_thread_num() * (size_t)K;
        for (int64_t k = 0; k < K; ++k)
            wrow[k] = (double)ref_bf16_to_float(
                ref_dequant_one(Wq, scales, offsets, K, g, bits, n, k));
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)ref_bf16_to_float(X[m * K + k]) * wrow[k];
            Y[m * N + n] = acc;
        }
    }
    free(wbuf);
    return 0;
}

/*
 * The linear with the layer's bias: Y[m,n] = sum_k X[m,k] W'[n,k] + bias[n]
 * in fp64.  Optimum Quanto, "Design overview / Modules": the bias of a
 * quantized module is not quantized, so it enters in float (bf16 here, widened
 * exactly) on top of the product.
 */
int w4_ref_linear_bias_bits(const uint16_t *X, int64_t M, int64_t K, const uint8_t *Wq,
                            const uint16_t *scales, const uint16_t *offsets, int64_t N,
                            int g, int bits, const uint16_t *bias, double *Y)
{
    int rc = w4_ref_linear_bits(X, M, K, Wq, scales, offsets, N, g, bits, Y);
    if (rc != 0)
        return rc;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            Y[m * N + n] += (double)ref_bf16_to_float(bias[n]);
    return 0;
}

int w4_ref_linear(const uint16_t *X, int64_t M, int64_t K, const uint8_t *Wq,
                  const uint16_t *scales, const uint16_t *offsets, int64_t N,
                  int g, double *Y)
{
    return w4_ref_linear_bits(X, M, K, Wq, scales, offsets, N, g, 4, Y);
}

/* ---- int8 dynamic activations x int4 weights ------------------------- */

/*
 * Dynamic symmetric int8 quantization of the activations X[M,K] (bf16).
 * torchao README "Training / QAT" and torchao guide (QAT, edge deployment):
 * Int8DynamicActivationInt4WeightConfig quantizes the activations to int8 at
 * run time and the weights to int4 in groups.  Optimum Quanto, "Design
 * overview / Modules" and "Pitfalls when quantizing activations": activations
 * are quantized per tensor, with a symmetric range (the default [-1, 1]);
 * the integer mapping rounds half to even (torch.round, "Design overview /
 * Tensors").
 * Readings: "dynamic" means the scale comes from the tensor itself at run
 * time, s_x = a / 127 with a = max |x| (fp32 IEEE division), clamped below at
 * the weights' eps; the codes are q_x = clamp(rne(x / s_x), -127, 127), so the
 * largest magnitude codes to +-127 and zero to 0.  The torchao pages leave the
 * granularity open, so one scale per row of X (per token) is offered beside
 * Quanto's one scale per tensor.  x_scale gets 1 value (per tensor) or M.
 */
int w4_ref_quantize_activation_i8(const uint16_t *X, int64_t M, int64_t K, int per_token,
                                  int8_t *Xq, float *x_scale)
{
    if (M < 0 || K <= 0)
        return -1;
    const int64_t nscales = per_token ? M : (M > 0 ? 1 : 0);
    for (int64_t r = 0; r < nscales; ++r) {
        const int64_t m0 = per_token ? r : 0, m1 = per_token ? r + 1 : M;
        float a = 0.0f;
        for (int64_t m = m0; m < m1; ++m)
            for (int64_t k = 0; k < K; ++k) {
                float v = fabsf(ref_bf16_to_float(X[m * K + k]));
                if (v > a)
                    a = v;
            }
        float s = a / 127.0f;
        if (s < REF_EPS)
            s = REF_EPS;
        x_scale[r] = s;
        for (int64_t m = m0; m < m1; ++m)
            for (int64_t k = 0; k < K; ++k) {
                float t = ref_bf16_to_float(X[m * K + k]) / s;
                float q = rintf(t);
                if (q > 127.0f)
                    q = 127.0f;
                if (q < -127.0f)
                    q = -127.0f;
                Xq[m * K + k] = (int8_t)q;
            }
    }
    return 0;
}

/*
 * The linear on int8 activation codes and int4 weight codes:
 *   Y[m,n] = s_x(m) * sum_j ( s_j * I_j + o_j * S_j ) + bias[n]      (fp64)
 * with, over the k of group j, I_j = sum q_x[m,k] q[n,k] and S_j = sum q_x[m,k]
 * accumulated exactly in integers.  This is sum_k (s_x q_x)(q s_j + o_j): the
 * integer product of the codes, accumulated wider than its inputs and then
 * brought back to float with the activation scale and each group's scale and
 * offset, and the float bias added last (Optimum Quanto, "Pitfalls when
 * quantizing activations").  s_x(m) = x_scale[m] per token, x_scale[0] per
 * tensor.  bias may be NULL.  Weights: 4-bit codes, the layout of w4_ref_quantize.
 */
int w4_ref_linear_i8(const int8_t *Xq, const float *x_scale, int per_token, int64_t M, int64_t K,
                     const uint8_t *Wq, const uint16_t *scales, const uint16_t *offsets, int64_t N,
                     int g, const uint16_t *bias, double *Y)
{
    if (!ref_group_ok(N, K, g) || M < 0)
        return -1;
    const int64_t ng = K / g;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t j = 0; j < ng; ++j) {
                int64_t I = 0, S = 0;
                for (int64_t k = j * g; k < (j + 1) * g; ++k) {
                    int q = (Wq[n * (K / 2) + k / 2] >> ((int)(k % 2) * 4)) & 0xF;
                    I += (int64_t)Xq[m * K + k] * q;
                    S += (int64_t)Xq[m * K + k];
                }
                acc += (double)ref_bf16_to_float(scales[n * ng + j]) * (double)I
                     + (double)ref_bf16_to_float(offsets[n * ng + j]) * (double)S;
            }
            double y = (double)x_scale[per_token ? m : 0] * acc;
            if (bias != NULL)
                y += (double)ref_bf16_to_float(bias[n]);
            Y[m * N + n] = y;
        }
    return 0;
}

/* The clamp constant, exported so tests can state which reading they pin. */
float w4_ref_eps(void) { return REF_EPS; }

/* Threads of the row loops: n > 0 sets n, n <= 0 every core the host offers;
 * returns the number now in use. */
int w4_ref_threads(int n)
{
    omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
    return omp_get_max_threads();
}
