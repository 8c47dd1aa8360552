/*
 * nvfp4_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU statement of what the NVFP4 weight-only
 * SwiGLU FFN decode computes.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table
 * or constant generator with the CUDA library; it is the yardstick the CUDA
 * path is checked against, never a fallback for it.
 *
 * Sources (the Atlas inference engine's published Rust pages):
 *  - "spark_model/layers/dense_ffn.rs", module doc comment: the FFN is
 *    out = down_proj(act(gate_proj(x)) * up_proj(x)).
 *  - same page, doc comment of DenseFfnLayer::ensure_int8_weight: an NVFP4
 *    projection holds E2M1 codes two to a byte ([N, K/2], `weight`), an E4M3
 *    scale for every 16 K elements ([N, K/16], `weight_scale`) and a single
 *    FP32 scale for the tensor (`weight_scale_2`).
 *  - same page, DenseFfnLayer::forward (split-SiLU branch): gate and up are
 *    written as BF16 buffers, the act*up product overwrites gate as BF16, the
 *    down GEMV reads that BF16 vector.
 *  - same page, enum FfnActivation: SiLU or GELU gating.
 *  - "spark_model/weight_loader/qwen35_dense.rs", load_layers: BF16/FP32
 *    weights become NVFP4 through a global-absmax kernel followed by a
 *    quantize kernel; the fused-QKV comment there: the per-tensor scale2 is
 *    applied once per launch, outside the per-16 scales.
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *  - E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}, sign in bit 3; element 2j in
 *    the low nibble of byte j.
 *  - E4M3 is the "fn" variant: bias 7, subnormals m/8*2^-6, 0x7F/0xFF NaN,
 *    largest finite 448, no infinities.
 *  - Quantise: amax = max|W|; scale2 = amax/2688 (2688 = 6*448), 1 if amax==0;
 *    per 16-block s = E4M3(bamax/6/scale2); code = E2M1(w/(E4M3(s)*scale2)),
 *    all IEEE fp32 operations in that order.  Both converts round to nearest,
 *    ties to the even code, saturate at the largest finite value, keep the
 *    sign (so a negative value that rounds to zero is code 0x8).  A block with
 *    s == 0 gets code 0 with the element's sign.
 *  - GEMV: y = bf16(scale2 * sum_k x*e2m1*e4m3), the sum in double.
 *  - FFN: g = bf16(gemv_gate), u = bf16(gemv_up), h = bf16(act(g)*u),
 *    out = bf16(gemv_down(h)); SiLU(t) = t/(1+e^-t); GeLU is the tanh form.
 *    No clamp.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no fast-math, so
 * every float operation below is one correctly rounded IEEE operation).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------- element codecs ---------------- */

/* E2M1 magnitude for the three low code bits (sign is bit 3). */
static const double E2M1_MAGNITUDE[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_decode(uint8_t code)
{
    double m = E2M1_MAGNITUDE[code & 7];
    return (code & 8) ? -m : m;
}

/* E4M3 (fn variant): sign | 4-bit exponent, bias 7 | 3-bit mantissa. */
double orc_e4m3_decode(uint8_t b)
{
    int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/*
 * Nearest E2M1 code by exhaustive search over the 8 magnitudes: ties go to
 * the even code (mantissa bit 0 clear), |q| >= 6 saturates to 6, the sign bit
 * of q is kept.  q must not be NaN.
 */
uint8_t orc_e2m1_encode(float q)
{
    uint8_t sign = signbit(q) ? 8 : 0;
    double a = fabs((double)q);
    int best = 0;
    double best_d;
    if (a >= 6.0)
        return sign | 7;
    best_d = a; /* distance to magnitude 0 (code 0, even) */
    for (int c = 1; c < 8; ++c) {
        double d = fabs(a - E2M1_MAGNITUDE[c]);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return sign | (uint8_t)best;
}

/*
 * Nearest finite E4M3 byte by exhaustive search over the 127 non-negative
 * finite codes; ties to the even code, saturating at 448 (0x7E).  q must not
 * be NaN.
 */
uint8_t orc_e4m3_encode(float q)
{
    uint8_t sign = signbit(q) ? 0x80 : 0;
    double a = fabs((double)q);
    int best = 0;
    double best_d;
    if (a >= 448.0)
        return sign | 0x7E;
    best_d = a;
    for (int c = 1; c <= 0x7E; ++c) {
        double d = fabs(a - orc_e4m3_decode((uint8_t)c));
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return sign | (uint8_t)best;
}

/* ---------------- bf16 ---------------- */

double orc_bf16_decode(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/*
 * Round a double straight to the nearest bf16 (ties to even), without an
 * intermediate float (which could round twice).  bf16 keeps 8 significant
 * bits; its subnormal spacing is 2^-133; past the largest finite value the
 * result is infinity.
 */
uint16_t orc_bf16_from_double(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v), r;
    int e, ulp_exp;
    float f;
    uint32_t u;
    if (isnan(v))
        return 0x7FC0;
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    frexp(a, &e);           /* a = f * 2^e with f in [0.5, 1) */
    ulp_exp = e - 8;        /* spacing of the 8-bit significand grid */
    if (ulp_exp < -133)
        ulp_exp = -133;
    r = nearbyint(ldexp(a, -ulp_exp)); /* default mode: nearest, ties even */
    r = ldexp(r, ulp_exp);
    if (r > 3.3895313892515355e38) /* largest finite bf16 */
        return sign | 0x7F80;
    f = (float)r;           /* exact: r is a bf16 value */
    memcpy(&u, &f, 4);
    return sign | (uint16_t)(u >> 16);
}

/* ---------------- quantise (fp32 arithmetic, in this order) ---------------- */

static void quantize_rows(const float *w, int64_t N, int64_t K, uint8_t *codes,
                          uint8_t *scales, float *scale2_out)
{
    float amax = 0.0f, scale2;
    int64_t n;
    for (int64_t i = 0; i < N * K; ++i) {
        float a = fabsf(w[i]);
        if (a > amax)
            amax = a;
    }
    scale2 = (amax == 0.0f) ? 1.0f : amax / 2688.0f;
    *scale2_out = scale2;
#pragma omp parallel for schedule(static)
    for (n = 0; n < N; ++n) {
        for (int64_t b = 0; b < K / 16; ++b) {
            const float *blk = w + n * K + b * 16;
            float bamax = 0.0f, t, denom;
            uint8_t s;
            for (int j = 0; j < 16; ++j) {
                float a = fabsf(blk[j]);
                if (a > bamax)
                    bamax = a;
            }
            t = bamax / 6.0f;
            t = t / scale2;
            s = orc_e4m3_encode(t);
            scales[n * (K / 16) + b] = s;
            denom = (float)orc_e4m3_decode(s) * scale2;
            for (int j = 0; j < 16; ++j) {
                uint8_t c;
                if (s == 0) {
                    c = signbit(blk[j]) ? 8 : 0;
                } else {
                    float q = blk[j] / denom;
                    c = orc_e2m1_encode(q);
                }
                {
                    int64_t byte = n * (K / 2) + b * 8 + j / 2;
                    if ((j & 1) == 0)
                        codes[byte] = c;
                    else
                        codes[byte] |= (uint8_t)(c << 4);
                }
            }
        }
    }
}

/* W fp32 [N, K] row-major, K % 16 == 0.  codes [N, K/2], scales [N, K/16]. */
int orc_quantize_f32(const float *w, int64_t N, int64_t K, uint8_t *codes,
                     uint8_t *scales, float *scale2_out)
{
    if (K % 16 != 0 || N < 0 || K < 0)
        return 1;
    quantize_rows(w, N, K, codes, scales, scale2_out);
    return 0;
}

/* Same with a bf16 source: each bf16 value widens exactly to fp32 first. */
int orc_quantize_bf16(const uint16_t *w, int64_t N, int64_t K, uint8_t *codes,
                      uint8_t *scales, float *scale2_out)
{
    float *wf;
    if (K % 16 != 0 || N < 0 || K < 0)
        return 1;
    wf = (float *)malloc((size_t)(N * K > 0 ? N * K : 1) * sizeof(float));
    if (!wf)
        return 2;
    for (int64_t i = 0; i < N * K; ++i)
        wf[i] = (float)orc_bf16_decode(w[i]);
    quantize_rows(wf, N, K, codes, scales, scale2_out);
    free(wf);
    return 0;
}

/* Dequantised weight e2m1(code) * e4m3(scale) * scale2, in double. */
void orc_dequantize(const uint8_t *codes, const uint8_t *scales, float scale2,
                    int64_t N, int64_t K, double *out)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = codes[n * (K / 2) + k / 2];
            uint8_t c = (k & 1) ? (byte >> 4) : (byte & 15);
            out[n * K + k] = orc_e2m1_decode(c) *
                             orc_e4m3_decode(scales[n * (K / 16) + k / 16]) *
                             (double)scale2;
        }
}

/* ---------------- GEMV and FFN ---------------- */

/*
 * y[m, n] = scale2 * sum_k x[m, k] * e2m1(c[n, k]) * e4m3(s[n, k/16]) in
 * double, before the final bf16 rounding.  x is bf16 [M, K].
 */
void orc_gemv_f64(const uint16_t *x, int64_t M, int64_t K, const uint8_t *codes,
                  const uint8_t *scales, float scale2, int64_t N, double *y)
{
    int64_t n;
#pragma omp parallel for schedule(static)
    for (n = 0; n < N; ++n) {
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                uint8_t byte = codes[n * (K / 2) + k / 2];
                uint8_t c = (k & 1) ? (byte >> 4) : (byte & 15);
                acc += orc_bf16_decode(x[m * K + k]) * orc_e2m1_decode(c) *
                       orc_e4m3_decode(scales[n * (K / 16) + k / 16]);
            }
            y[m * N + n] = (double)scale2 * acc;
        }
    }
}

/* The GEMV with its bf16 output rounding: y bf16 [M, N]. */
void orc_gemv(const uint16_t *x, int64_t M, int64_t K, const uint8_t *codes,
              const uint8_t *scales, float scale2, int64_t N, uint16_t *y)
{
    double *t = (double *)malloc((size_t)(M * N > 0 ? M * N : 1) * sizeof(double));
    if (!t)
        return;
    orc_gemv_f64(x, M, K, codes, scales, scale2, N, t);
    for (int64_t i = 0; i < M * N; ++i)
        y[i] = orc_bf16_from_double(t[i]);
    free(t);
}

/* SiLU(t) = t * sigmoid(t) = t / (1 + e^-t). */
double orc_silu(double t)
{
    return t / (1.0 + exp(-t));
}

/*
 * GeLU, tanh form: 0.5 t (1 + tanh(z)), z = sqrt(2/pi) (t + 0.044715 t^3).
 * Evaluated as t / (1 + e^(-2z)), the same function (1 + tanh z =
 * 2 / (1 + e^(-2z))): for negative t the literal 1 + tanh z cancels to a few
 * ulps of 1 and loses all relative accuracy in the tail (about 3% at t = -7).
 */
double orc_gelu_tanh(double t)
{
    const double c = sqrt(2.0 / 3.14159265358979323846);
    const double z = c * (t + 0.044715 * t * t * t);
    return t / (1.0 + exp(-2.0 * z));
}

/*
 * Gate/up half of the FFN: h[m, i] = bf16(act(g) * u) with g, u the bf16
 * roundings of the two projections.  act: 0 = SiLU, 1 = GeLU (tanh).
 */
void orc_ffn_hidden(const uint16_t *x, int64_t M, int64_t H, int64_t I,
                    const uint8_t *gc, const uint8_t *gs, float g2,
                    const uint8_t *uc, const uint8_t *us, float u2, int act,
                    uint16_t *h)
{
    uint16_t *g = (uint16_t *)malloc((size_t)(M * I > 0 ? M * I : 1) * 2);
    uint16_t *u = (uint16_t *)malloc((size_t)(M * I > 0 ? M * I : 1) * 2);
    if (!g || !u) {
        free(g);
        free(u);
        return;
    }
    orc_gemv(x, M, H, gc, gs, g2, I, g);
    orc_gemv(x, M, H, uc, us, u2, I, u);
    for (int64_t i = 0; i < M * I; ++i) {
        double gv = orc_bf16_decode(g[i]), uv = orc_bf16_decode(u[i]);
        double a = (act == 0) ? orc_silu(gv) : orc_gelu_tanh(gv);
        h[i] = orc_bf16_from_double(a * uv);
    }
    free(g);
    free(u);
}

/* Full FFN: out bf16 [M, H] = bf16(down(h)). */
void orc_ffn(const uint16_t *x, int64_t M, int64_t H, int64_t I,
             const uint8_t *gc, const uint8_t *gs, float g2,
             const uint8_t *uc, const uint8_t *us, float u2,
             const uint8_t *dc, const uint8_t *ds, float d2, int act,
             uint16_t *out)
{
    uint16_t *h = (uint16_t *)malloc((size_t)(M * I > 0 ? M * I : 1) * 2);
    if (!h)
        return;
    orc_ffn_hidden(x, M, H, I, gc, gs, g2, uc, us, u2, act, h);
    orc_gemv(h, M, I, dc, ds, d2, H, out);
    free(h);
}

/* ---------------- block-scaled FP8 (w8a16) ---------------- */

/*
 * The dense-FFN page's native FP8 arm ("spark_model/layers/dense_ffn.rs",
 * DenseFfnWeightsFp8 and the FP8 dispatch of DenseFfnLayer::forward: a dual
 * gate/up GEMV, then the activation-consuming down GEMV; the weight loader's
 * proj_is_fp8_any_scale): a projection is E4M3 bytes q [N, K] row-major plus
 * an FP32 grid bs [ceil(N/128), ceil(K/128)] row-major, and
 *     W[n][k] = e4m3(q[n][k]) * bs[n/128][k/128]
 * with no per-tensor scale (a per-tensor scalar is the uniform grid).
 * Reading: the roundings are those of the NVFP4 path (gate_out, up_out and
 * the activation product are bf16 buffers on the same page).
 */

static double fp8_weight(const uint8_t *q, const float *bs, int64_t K, int64_t n, int64_t k)
{
    const int64_t kb = (K + 127) / 128;
    return orc_e4m3_decode(q[n * K + k]) * (double)bs[(n / 128) * kb + k / 128];
}

/* Dequantised weight [N, K] in double. */
void orc_fp8_dequantize(const uint8_t *q, const float *bs, int64_t N, int64_t K, double *w)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = fp8_weight(q, bs, K, n, k);
}

/* y[m, n] = sum_k x[m, k] * W[n][k] in double, before the bf16 rounding. */
void orc_gemv_fp8_f64(const uint16_t *x, int64_t M, int64_t K, const uint8_t *q,
                      const float *bs, int64_t N, double *y)
{
    int64_t n;
#pragma omp parallel for schedule(static)
    for (n = 0; n < N; ++n) {
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += orc_bf16_decode(x[m * K + k]) * fp8_weight(q, bs, K, n, k);
            y[m * N + n] = acc;
        }
    }
}

/* The FP8 GEMV with its bf16 output rounding: y bf16 [M, N]. */
void orc_gemv_fp8(const uint16_t *x, int64_t M, int64_t K, const uint8_t *q, const float *bs,
                  int64_t N, uint16_t *y)
{
    double *t = (double *)malloc((size_t)(M * N > 0 ? M * N : 1) * sizeof(double));
    if (!t)
        return;
    orc_gemv_fp8_f64(x, M, K, q, bs, N, t);
    for (int64_t i = 0; i < M * N; ++i)
        y[i] = orc_bf16_from_double(t[i]);
    free(t);
}

/* h[m, i] = bf16(act(g) * u) from the bf16 projections of the FP8 gate and up. */
void orc_ffn_fp8_hidden(const uint16_t *x, int64_t M, int64_t H, int64_t I, const uint8_t *gq,
                        const float *gbs, const uint8_t *uq, const float *ubs, int act,
                        uint16_t *h)
{
    uint16_t *g = (uint16_t *)malloc((size_t)(M * I > 0 ? M * I : 1) * 2);
    uint16_t *u = (uint16_t *)malloc((size_t)(M * I > 0 ? M * I : 1) * 2);
    if (!g || !u) {
        free(g);
        free(u);
        return;
    }
    orc_gemv_fp8(x, M, H, gq, gbs, I, g);
    orc_gemv_fp8(x, M, H, uq, ubs, I, u);
    for (int64_t i = 0; i < M * I; ++i) {
        double gv = orc_bf16_decode(g[i]), uv = orc_bf16_decode(u[i]);
        double a = (act == 0) ? orc_silu(gv) : orc_gelu_tanh(gv);
        h[i] = orc_bf16_from_double(a * uv);
    }
    free(g);
    free(u);
}

/* Full FP8 FFN: out bf16 [M, H] = bf16(down(h)). */
void orc_ffn_fp8(const uint16_t *x, int64_t M, int64_t H, int64_t I, const uint8_t *gq,
                 const float *gbs, const uint8_t *uq, const float *ubs, const uint8_t *dq,
                 const float *dbs, int act, uint16_t *out)
{
    uint16_t *h = (uint16_t *)malloc((size_t)(M * I > 0 ? M * I : 1) * 2);
    if (!h)
        return;
    orc_ffn_fp8_hidden(x, M, H, I, gq, gbs, uq, ubs, act, h);
    orc_gemv_fp8(h, M, I, dq, dbs, H, out);
    free(h);
}

/* ---------------- LoRA overlay ---------------- */

/*
 * The dense-FFN page's adapter overlay (DenseFfnLayer::apply_lora_gate_up and
 * apply_lora_down): gate_out += dW_gate x and up_out += dW_up x land after the
 * gate/up projections and before the activation; output += dW_down act lands
 * after the down projection and contracts over the activation h, not over the
 * layer input.  Readings (the page names the helper's buffers, lora_xa and
 * lora_delta, but not their types or formulas):
 *   dW = B A with A [r, in] and B [out, r], both bf16, any alpha/r folded into B;
 *   xa = bf16(A v), delta = bf16(B xa) (every named buffer holds bf16, like the
 *   engine's other activations), base = bf16(base + delta).
 */

/* xa bf16 [M, r] = bf16(sum_k A[j][k] v[m][k]) for v bf16 [M, K], A bf16 [r, K]. */
void orc_lora_xa(const uint16_t *v, int64_t M, int64_t K, const uint16_t *A, int64_t r,
                 uint16_t *xa)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += orc_bf16_decode(A[j * K + k]) * orc_bf16_decode(v[m * K + k]);
            xa[m * r + j] = orc_bf16_from_double(acc);
        }
}

/* delta bf16 [M, N] = bf16(sum_j B[n][j] xa[m][j]) for xa bf16 [M, r], B bf16 [N, r]. */
void orc_lora_delta(const uint16_t *xa, int64_t M, int64_t r, const uint16_t *B, int64_t N,
                    uint16_t *delta)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t j = 0; j < r; ++j)
                acc += orc_bf16_decode(B[n * r + j]) * orc_bf16_decode(xa[m * r + j]);
            delta[m * N + n] = orc_bf16_from_double(acc);
        }
}

/* base[i] = bf16(base[i] + delta[i]) for i < n (both bf16). */
void orc_lora_add(uint16_t *base, const uint16_t *delta, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        base[i] = orc_bf16_from_double(orc_bf16_decode(base[i]) + orc_bf16_decode(delta[i]));
}

/* base bf16 [M, N] += dW v for v bf16 [M, K] (the page's apply_lora_delta). */
void orc_lora_apply(const uint16_t *v, int64_t M, int64_t K, const uint16_t *A,
                    const uint16_t *B, int64_t r, int64_t N, uint16_t *base)
{
    uint16_t *xa = (uint16_t *)malloc((size_t)(M * r > 0 ? M * r : 1) * 2);
    uint16_t *d = (uint16_t *)malloc((size_t)(M * N > 0 ? M * N : 1) * 2);
    if (xa && d) {
        orc_lora_xa(v, M, K, A, r, xa);
        orc_lora_delta(xa, M, r, B, N, d);
        orc_lora_add(base, d, M * N);
    }
    free(xa);
    free(d);
}

/*
 * The FFN with the overlay (a pair whose A is NULL is absent):
 *   g = bf16(gemv_gate x) [+ dW_gate x],  u = bf16(gemv_up x) [+ dW_up x],
 *   h = bf16(act(g) u),  out = bf16(gemv_down h) [+ dW_down h].
 * h (bf16 [M, I]) is also returned when h_out is not NULL.
 */
void orc_ffn_lora(const uint16_t *x, int64_t M, int64_t H, int64_t I,
                  const uint8_t *gc, const uint8_t *gs, float g2,
                  const uint8_t *uc, const uint8_t *us, float u2,
                  const uint8_t *dc, const uint8_t *ds, float d2, int act, int64_t r,
                  const uint16_t *gA, const uint16_t *gB, const uint16_t *uA,
                  const uint16_t *uB, const uint16_t *dA, const uint16_t *dB,
                  uint16_t *out, uint16_t *h_out)
{
    size_t n = (size_t)(M * I > 0 ? M * I : 1);
    uint16_t *g = (uint16_t *)malloc(n * 2), *u = (uint16_t *)malloc(n * 2);
    uint16_t *h = (uint16_t *)malloc(n * 2);
    if (g && u && h) {
        orc_gemv(x, M, H, gc, gs, g2, I, g);
        orc_gemv(x, M, H, uc, us, u2, I, u);
        if (gA)
            orc_lora_apply(x, M, H, gA, gB, r, I, g);
        if (uA)
            orc_lora_apply(x, M, H, uA, uB, r, I, u);
        for (int64_t i = 0; i < M * I; ++i) {
            double gv = orc_bf16_decode(g[i]), uv = orc_bf16_decode(u[i]);
            double a = (act == 0) ? orc_silu(gv) : orc_gelu_tanh(gv);
            h[i] = orc_bf16_from_double(a * uv);
        }
        orc_gemv(h, M, I, dc, ds, d2, H, out);
        if (dA)
            orc_lora_apply(h, M, I, dA, dB, r, H, out);
        if (h_out)
            memcpy(h_out, h, (size_t)(M * I) * 2);
    }
    free(g);
    free(u);
    free(h);
}

int orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* ---------------- array forms (loops over the functions above) ---------------- */

void orc_bf16_from_double_array(const double *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_from_double(v[i]);
}

/* act: 0 = SiLU, 1 = GeLU (tanh) */
void orc_act_array(const double *v, int64_t n, int act, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (act == 0) ? orc_silu(v[i]) : orc_gelu_tanh(v[i]);
}
