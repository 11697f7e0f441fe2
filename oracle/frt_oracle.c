/*
 * frt_oracle.c -- plain, slow CPU oracle of the FP8-quantised pre-norm FFN
 * sublayer (residual add + RMSNorm + E4M3 quantise, FP8 gate/up GEMM, gated
 * activation + requantise, FP8 down GEMM + residual), stacked layer by layer.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  The product (the CUDA
 * library and its Python binding) never links, imports or calls it, and this
 * file shares no code, header, table or constant generator with it.
 *
 * Arithmetic: IEEE-754 binary32, every operation rounded on its own (the file
 * is built with -ffp-contract=off and without fast-math), sums taken in
 * ascending index order, the E4M3 and BF16 encoders written out from their
 * definitions.  OpenMP only splits independent rows or output elements; it
 * never reorders an individual sum.
 *
 * Sources, by page title and section:
 *   [SUM]  agentlenshq "flashrt-project/FlashRT" summary, "Main ideas": fused
 *          residual-norm-quantise kernels; FP8 per-tensor auto-calibration
 *          cached as JSON; FP8 keeps cosine > 0.999 against FP16/BF16.
 *   [ART]  itsolotime FlashRT article: 3.3 "Pipeline layer" (rms_norm row of
 *          the kernel table); 5.2 "Pi0 vs Pi0.5 spec" (FusedGateUp + Quant,
 *          per-tensor weight scales); 7.1 "FP8 path"; 7.2 "NVFP4 path"
 *          (per-layer FFN loop: norm, gate/up GEMM, gated activation with
 *          requantise, down GEMM, residual add).
 *   [ARCH] "FlashRT docs/architecture.md": component 6 "Calibration
 *          Framework" (amax per FP8 GEMM input; alpha = act_scale x
 *          weight_scale baked as host scalars); "What happens when you call
 *          model.predict" (cache miss: run one forward, record amax).
 *
 * Readings where the pages are silent (each listed in the design notes):
 * eps = 1e-6; the norm weight is used as stored (no 1+w offset); one scale
 * for the fused gate/up weight; quantise by multiplying with the fp32
 * reciprocal of the scale; scale = amax/448 and 1 when amax == 0; NaN encodes
 * as 0x7F; out-of-range values saturate to +-448; the gate/up GEMM output is
 * rounded to BF16; the down epilogue scales, adds the BF16 residual and rounds
 * once; the hidden input is added at layer 0 only; calibration is progressive
 * (layer l is measured on the quantised output of layers < l).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float bits_f32(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

/*
 * OCP FP8 E4M3 ("fn": no infinities).  1 sign, 4 exponent bits (bias 7),
 * 3 mantissa bits.  Exponent field 0 holds subnormals m * 2^-9; fields 1..15
 * hold (1 + m/8) * 2^(e-7); 0x7F and 0xFF are NaN, so the largest finite
 * magnitude is 1.75 * 2^8 = 448 (0x7E).
 */
ORC_API float orc_e4m3_decode(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 7;
    float mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexpf((float)m, -9);
    else
        mag = ldexpf(1.0f + (float)m / 8.0f, e - 7);
    return sign ? -mag : mag;
}

/*
 * Round-to-nearest-even onto the E4M3 grid with saturation to +-448 (the
 * "satfinite" behaviour): every magnitude above 448, infinity included,
 * becomes 448.  NaN becomes the canonical 0x7F.  The sign of zero is kept.
 * The grid spacing is 2^-9 below 2^-6 and 2^(e-3) in binade [2^e, 2^(e+1)).
 */
ORC_API uint8_t orc_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    float a = fabsf(x);
    if (a > 448.0f)
        return sign | 0x7E;
    if (a < ldexpf(1.0f, -6)) {
        /* subnormal binade: q = a / 2^-9 is exact in fp32 (power-of-two
         * scaling), rintf rounds half to even in the default mode. */
        float q = rintf(ldexpf(a, 9));
        int qi = (int)q; /* 0..8; 8 is the smallest normal, code 0x08 */
        return sign | (uint8_t)qi;
    }
    int e;
    frexpf(a, &e);          /* a = f * 2^e with f in [0.5, 1) */
    e -= 1;                 /* a in [2^e, 2^(e+1)), e in [-6, 8] */
    /* position on the grid of this binade: a / 2^(e-3), in [8, 16) */
    float q = rintf(ldexpf(a, 3 - e));
    int qi = (int)q;
    if (qi == 16) {         /* rounded up into the next binade */
        qi = 8;
        e += 1;
    }
    int field = e + 7;      /* 1..15 */
    int m = qi - 8;         /* 0..7 */
    return sign | (uint8_t)((field << 3) | m);
}

/* BF16: top 16 bits of binary32, rounded to nearest even.  NaN stays a
 * quiet NaN of the same sign. */
ORC_API uint16_t orc_bf16_encode(float x)
{
    uint32_t u = f32_bits(x);
    if (isnan(x))
        return (uint16_t)((u >> 16) | 0x0040);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

ORC_API float orc_bf16_decode(uint16_t b) { return bits_f32((uint32_t)b << 16); }

/* Bulk codecs (used by the tests on whole arrays). */
ORC_API void orc_e4m3_encode_array(const float *x, int64_t n, uint8_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_e4m3_encode(x[i]);
}

ORC_API void orc_bf16_encode_array(const float *x, int64_t n, uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_bf16_encode(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Per-tensor scales ([ART] 5.2 Quant / scale_into; [ARCH] 6)                */
/* ------------------------------------------------------------------------ */

/* scale = amax / 448 (IEEE division); an all-zero tensor gets scale 1. */
ORC_API float orc_scale_from_amax(float amax)
{
    if (amax == 0.0f)
        return 1.0f;
    return amax / 448.0f;
}

ORC_API float orc_amax_bf16(const uint16_t *x, int64_t n)
{
    float m = 0.0f;
#pragma omp parallel for reduction(max : m) schedule(static)
    for (int64_t i = 0; i < n; i++) {
        float a = fabsf(orc_bf16_decode(x[i]));
        if (a > m)
            m = a;
    }
    return m;
}

/* q = E4M3(x * inv_s) with inv_s = 1/s precomputed in fp32. */
ORC_API void orc_quantize_bf16(const uint16_t *x, int64_t n, float inv_s, uint8_t *q)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++)
        q[i] = orc_e4m3_encode(orc_bf16_decode(x[i]) * inv_s);
}

/*
 * Step A0, weight preparation ([ART] 5.2: FusedGateUp(gate, up) with Quant();
 * [ART] FlashRT weight spec "scale_into").  The gate and up matrices are
 * treated as one tensor [W_gate; W_up] with one scale; the down matrix has its
 * own.  Writes the E4M3 codes and the fp32 scale.
 */
ORC_API float orc_quantize_weight(const uint16_t *w, int64_t n, uint8_t *q)
{
    float amax = orc_amax_bf16(w, n);
    float s = orc_scale_from_amax(amax);
    float inv_s = 1.0f / s;
    orc_quantize_bf16(w, n, inv_s, q);
    return s;
}

/* ------------------------------------------------------------------------ */
/* Step A1: residual add + RMSNorm ([SUM] fused residual-norm-quantise;      */
/* [ART] 3.3 rms_norm row; [ART] 7.2 "x_norm = rms_norm(x)")                 */
/* ------------------------------------------------------------------------ */

/*
 * r'  = bf16(r + h)            (h == NULL: r' = r)
 * ms  = (sum_i r'_i^2) / d     (ascending i)
 * inv = 1 / sqrt(ms + eps)
 * y_i = (r'_i * inv) * w_i     (fp32; quantised by the caller)
 */
ORC_API void orc_residual_rmsnorm(int M, int d, float eps, const uint16_t *r, const uint16_t *h,
                                  const uint16_t *w_norm, uint16_t *r_prime, float *y)
{
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; m++) {
        const uint16_t *rr = r + (int64_t)m * d;
        uint16_t *rp = r_prime + (int64_t)m * d;
        for (int i = 0; i < d; i++) {
            if (h) {
                float s = orc_bf16_decode(rr[i]) + orc_bf16_decode(h[(int64_t)m * d + i]);
                rp[i] = orc_bf16_encode(s);
            } else {
                rp[i] = rr[i];
            }
        }
        float sum = 0.0f;
        for (int i = 0; i < d; i++) {
            float v = orc_bf16_decode(rp[i]);
            sum = sum + v * v;
        }
        float ms = sum / (float)d;
        float inv = 1.0f / sqrtf(ms + eps);
        for (int i = 0; i < d; i++) {
            float v = orc_bf16_decode(rp[i]);
            y[(int64_t)m * d + i] = (v * inv) * orc_bf16_decode(w_norm[i]);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Steps A2 / A4 core: E4M3 x E4M3 -> fp32 GEMM, both operands K-major       */
/* ([ART] 7.2 gate/up and down GEMMs; [SUM] FP8 GEMM)                        */
/* ------------------------------------------------------------------------ */

/* acc[m][n] = sum_k dec(A[m][k]) * dec(B[n][k]), k ascending, fp32. */
ORC_API void orc_gemm_e4m3(int M, int N, int K, const uint8_t *A, const uint8_t *B, float *acc)
{
    float lut[256];
    for (int c = 0; c < 256; c++)
        lut[c] = orc_e4m3_decode((uint8_t)c);
#pragma omp parallel for collapse(2) schedule(static)
    for (int m = 0; m < M; m++) {
        for (int n = 0; n < N; n++) {
            const uint8_t *a = A + (int64_t)m * K;
            const uint8_t *b = B + (int64_t)n * K;
            float s = 0.0f;
            for (int k = 0; k < K; k++)
                s = s + lut[a[k]] * lut[b[k]];
            acc[(int64_t)m * N + n] = s;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Step A3: gated activation ([ART] 7.2 "GEGLU/SiLU gate + requantise")      */
/* ------------------------------------------------------------------------ */

#define ORC_ACT_GEGLU_TANH 0
#define ORC_ACT_SWIGLU 1

/* GELU, tanh form: 0.5 g (1 + tanh( sqrt(2/pi) (g + 0.044715 g^3) )). */
ORC_API float orc_gelu_tanh(float g)
{
    const float k0 = 0.7978845608028654f; /* sqrt(2/pi) */
    const float k1 = 0.044715f;
    float g3 = (g * g) * g;
    float inner = k0 * (g + k1 * g3);
    return (0.5f * g) * (1.0f + tanhf(inner));
}

/* SiLU: g / (1 + exp(-g)). */
ORC_API float orc_silu(float g) { return g / (1.0f + expf(-g)); }

/* a[m][j] = act(g[m][j]) * u[m][j] with g = gu[m][j], u = gu[m][ff + j]
 * (both BF16, as materialised by the gate/up GEMM). */
ORC_API void orc_gated_act(int M, int ff, int act, const uint16_t *gu, float *a)
{
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; m++) {
        const uint16_t *row = gu + (int64_t)m * 2 * ff;
        for (int j = 0; j < ff; j++) {
            float g = orc_bf16_decode(row[j]);
            float u = orc_bf16_decode(row[ff + j]);
            float ag = (act == ORC_ACT_SWIGLU) ? orc_silu(g) : orc_gelu_tanh(g);
            a[(int64_t)m * ff + j] = ag * u;
        }
    }
}

/* a[i] = act(g[i]) * u[i] on fp32 operands (the NVFP4 path decodes its FP4
 * gate and up values to fp32 instead of BF16). */
ORC_API void orc_gated_act_f32(int64_t n, int act, const float *g, const float *u, float *a)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) {
        float ag = (act == ORC_ACT_SWIGLU) ? orc_silu(g[i]) : orc_gelu_tanh(g[i]);
        a[i] = ag * u[i];
    }
}

static float amax_f32(const float *x, int64_t n)
{
    float m = 0.0f;
#pragma omp parallel for reduction(max : m) schedule(static)
    for (int64_t i = 0; i < n; i++) {
        float v = fabsf(x[i]);
        if (v > m)
            m = v;
    }
    return m;
}

static void quantize_f32(const float *x, int64_t n, float inv_s, uint8_t *q)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++)
        q[i] = orc_e4m3_encode(x[i] * inv_s);
}

ORC_API float orc_amax_f32(const float *x, int64_t n) { return amax_f32(x, n); }
ORC_API void orc_quantize_f32(const float *x, int64_t n, float inv_s, uint8_t *q) { quantize_f32(x, n, inv_s, q); }

/* ------------------------------------------------------------------------ */
/* One quantised layer (steps A1..A4) with fixed scales                      */
/* ------------------------------------------------------------------------ */

/*
 * Inputs: r [M,d] BF16, h [M,d] BF16 or NULL, w_norm [d] BF16,
 * wq_gu [2ff,d] E4M3 (gate rows then up rows), wq_down [d,ff] E4M3,
 * activation scales s_x, s_h and weight scales s_gu, s_d.
 * Output: out [M,d] BF16.  Optional intermediates (NULL to skip):
 * r_prime [M,d] BF16, q_x [M,d] E4M3, gu [M,2ff] BF16, q_h [M,ff] E4M3.
 *
 * alpha_gu = s_x * s_gu and alpha_d = s_h * s_d are fp32 products
 * ([ARCH] 6: alpha = act_scale x weight_scale, baked as host scalars).
 */
ORC_API int orc_ffn_layer(int M, int d, int ff, int act, float eps, const uint16_t *r, const uint16_t *h,
                          const uint16_t *w_norm, const uint8_t *wq_gu, const uint8_t *wq_down, float s_x,
                          float s_h, float s_gu, float s_d, uint16_t *out, uint16_t *r_prime_out,
                          uint8_t *q_x_out, uint16_t *gu_out, uint8_t *q_h_out)
{
    int64_t Md = (int64_t)M * d, Mff = (int64_t)M * ff;
    uint16_t *rp = (uint16_t *)malloc(sizeof(uint16_t) * Md);
    float *y = (float *)malloc(sizeof(float) * Md);
    uint8_t *qx = (uint8_t *)malloc(Md);
    float *acc_gu = (float *)malloc(sizeof(float) * Mff * 2);
    uint16_t *gu = (uint16_t *)malloc(sizeof(uint16_t) * Mff * 2);
    float *a = (float *)malloc(sizeof(float) * Mff);
    uint8_t *qh = (uint8_t *)malloc(Mff);
    float *acc_d = (float *)malloc(sizeof(float) * Md);
    if (!rp || !y || !qx || !acc_gu || !gu || !a || !qh || !acc_d) {
        free(rp); free(y); free(qx); free(acc_gu); free(gu); free(a); free(qh); free(acc_d);
        return -1;
    }
    float alpha_gu = s_x * s_gu;
    float alpha_d = s_h * s_d;
    float inv_s_x = 1.0f / s_x;
    float inv_s_h = 1.0f / s_h;

    /* A1 */
    orc_residual_rmsnorm(M, d, eps, r, h, w_norm, rp, y);
    quantize_f32(y, Md, inv_s_x, qx);
    /* A2: g, u = bf16(acc * alpha_gu) */
    orc_gemm_e4m3(M, 2 * ff, d, qx, wq_gu, acc_gu);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < Mff * 2; i++)
        gu[i] = orc_bf16_encode(acc_gu[i] * alpha_gu);
    /* A3 */
    orc_gated_act(M, ff, act, gu, a);
    quantize_f32(a, Mff, inv_s_h, qh);
    /* A4: out = bf16(r' + acc * alpha_d) */
    orc_gemm_e4m3(M, d, ff, qh, wq_down, acc_d);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < Md; i++)
        out[i] = orc_bf16_encode(orc_bf16_decode(rp[i]) + acc_d[i] * alpha_d);

    if (r_prime_out) memcpy(r_prime_out, rp, sizeof(uint16_t) * Md);
    if (q_x_out) memcpy(q_x_out, qx, Md);
    if (gu_out) memcpy(gu_out, gu, sizeof(uint16_t) * Mff * 2);
    if (q_h_out) memcpy(q_h_out, qh, Mff);
    free(rp); free(y); free(qx); free(acc_gu); free(gu); free(a); free(qh); free(acc_d);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step A6: progressive calibration of one layer ([ARCH] 6 and "What happens */
/* when you call model.predict": run one forward, record amax per FP8 GEMM   */
/* input)                                                                    */
/* ------------------------------------------------------------------------ */

/*
 * For the calibration batches b = 0..nb-1 with current residuals r_b [M,d]
 * (and hidden h_b at layer 0, else NULL):
 *   1. y_b = RMSNorm(r_b + h_b) for every batch;  s_x = max_b amax(y_b)/448
 *   2. quantise every y_b with s_x, run the gate/up GEMM and activation;
 *      s_h = max_b amax(a_b)/448
 *   3. quantise every a_b with s_h, run the down GEMM + residual; the result
 *      is written to r_out[b] and is the next layer's calibration input.
 * Returns s_x and s_h.  Every batch has M rows.
 */
ORC_API int orc_calibrate_layer(int M, int d, int ff, int act, float eps, int nb, const uint16_t *const *r_b,
                                const uint16_t *const *h_b, const uint16_t *w_norm, const uint8_t *wq_gu,
                                const uint8_t *wq_down, float s_gu, float s_d, float *s_x_out, float *s_h_out,
                                uint16_t *const *r_out)
{
    int64_t Md = (int64_t)M * d, Mff = (int64_t)M * ff;
    uint16_t *rp = (uint16_t *)malloc(sizeof(uint16_t) * Md * nb);
    float *y = (float *)malloc(sizeof(float) * Md * nb);
    float *a = (float *)malloc(sizeof(float) * Mff * nb);
    uint8_t *qx = (uint8_t *)malloc(Md);
    uint8_t *qh = (uint8_t *)malloc(Mff);
    float *acc_gu = (float *)malloc(sizeof(float) * Mff * 2);
    uint16_t *gu = (uint16_t *)malloc(sizeof(uint16_t) * Mff * 2);
    float *acc_d = (float *)malloc(sizeof(float) * Md);
    if (!rp || !y || !a || !qx || !qh || !acc_gu || !gu || !acc_d) {
        free(rp); free(y); free(a); free(qx); free(qh); free(acc_gu); free(gu); free(acc_d);
        return -1;
    }
    /* 1: amax of the gate/up GEMM input over all batches */
    float amax_x = 0.0f;
    for (int b = 0; b < nb; b++) {
        orc_residual_rmsnorm(M, d, eps, r_b[b], h_b ? h_b[b] : NULL, w_norm, rp + b * Md, y + b * Md);
        float m = amax_f32(y + b * Md, Md);
        if (m > amax_x)
            amax_x = m;
    }
    float s_x = orc_scale_from_amax(amax_x);
    float inv_s_x = 1.0f / s_x;
    float alpha_gu = s_x * s_gu;
    /* 2: amax of the down GEMM input over all batches */
    float amax_h = 0.0f;
    for (int b = 0; b < nb; b++) {
        quantize_f32(y + b * Md, Md, inv_s_x, qx);
        orc_gemm_e4m3(M, 2 * ff, d, qx, wq_gu, acc_gu);
        for (int64_t i = 0; i < Mff * 2; i++)
            gu[i] = orc_bf16_encode(acc_gu[i] * alpha_gu);
        orc_gated_act(M, ff, act, gu, a + b * Mff);
        float m = amax_f32(a + b * Mff, Mff);
        if (m > amax_h)
            amax_h = m;
    }
    float s_h = orc_scale_from_amax(amax_h);
    float inv_s_h = 1.0f / s_h;
    float alpha_d = s_h * s_d;
    /* 3: finish the layer for every batch with the new scales */
    for (int b = 0; b < nb; b++) {
        quantize_f32(a + b * Mff, Mff, inv_s_h, qh);
        orc_gemm_e4m3(M, d, ff, qh, wq_down, acc_d);
        const uint16_t *rpb = rp + b * Md;
        uint16_t *o = r_out[b];
        for (int64_t i = 0; i < Md; i++)
            o[i] = orc_bf16_encode(orc_bf16_decode(rpb[i]) + acc_d[i] * alpha_d);
    }
    *s_x_out = s_x;
    *s_h_out = s_h;
    free(rp); free(y); free(a); free(qx); free(qh); free(acc_gu); free(gu); free(acc_d);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Unquantised fp32 reference layer (the "FP16/BF16 baseline" that [SUM]    */
/* compares the FP8 path against with cosine > 0.999)                        */
/* ------------------------------------------------------------------------ */

/*
 * Same layer with no E4M3 or BF16 rounding anywhere: r' = r + h, y = RMSNorm,
 * g = y W_gate^T, u = y W_up^T, a = act(g) u, out = r' + a W_down^T, all fp32,
 * with the BF16 master weights decoded exactly.  r, h, out are fp32 [M,d].
 */
ORC_API int orc_ref_layer_f32_ex(int M, int d, int ff, int act, float eps, const float *r, const float *h,
                                 const uint16_t *w_norm, const uint16_t *w_gate, const uint16_t *w_up,
                                 const uint16_t *w_down, float *out, float *row_amax_y, float *row_amax_a);

ORC_API int orc_ref_layer_f32(int M, int d, int ff, int act, float eps, const float *r, const float *h,
                              const uint16_t *w_norm, const uint16_t *w_gate, const uint16_t *w_up,
                              const uint16_t *w_down, float *out)
{
    return orc_ref_layer_f32_ex(M, d, ff, act, eps, r, h, w_norm, w_gate, w_up, w_down, out, NULL, NULL);
}

/* The same, also reporting per row the amax of y (the normalised input of the
 * gate/up GEMM) and of a (the gated activation), when the pointers are not
 * NULL: the unquantised-forward reading of calibration. */
ORC_API int orc_ref_layer_f32_ex(int M, int d, int ff, int act, float eps, const float *r, const float *h,
                                 const uint16_t *w_norm, const uint16_t *w_gate, const uint16_t *w_up,
                                 const uint16_t *w_down, float *out, float *row_amax_y, float *row_amax_a)
{
    int64_t Md = (int64_t)M * d;
    float *rp = (float *)malloc(sizeof(float) * Md);
    float *a = (float *)malloc(sizeof(float) * (int64_t)M * ff);
    if (!rp || !a) {
        free(rp); free(a);
        return -1;
    }
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; m++) {
        float *row = rp + (int64_t)m * d;
        float sum = 0.0f;
        for (int i = 0; i < d; i++) {
            row[i] = h ? r[(int64_t)m * d + i] + h[(int64_t)m * d + i] : r[(int64_t)m * d + i];
            sum = sum + row[i] * row[i];
        }
        float inv = 1.0f / sqrtf(sum / (float)d + eps);
        float *yrow = (float *)malloc(sizeof(float) * d);
        float my = 0.0f, ma = 0.0f;
        for (int i = 0; i < d; i++) {
            yrow[i] = (row[i] * inv) * orc_bf16_decode(w_norm[i]);
            my = fmaxf(my, fabsf(yrow[i]));
        }
        for (int j = 0; j < ff; j++) {
            const uint16_t *wg = w_gate + (int64_t)j * d;
            const uint16_t *wu = w_up + (int64_t)j * d;
            float g = 0.0f, u = 0.0f;
            for (int k = 0; k < d; k++) {
                g = g + yrow[k] * orc_bf16_decode(wg[k]);
                u = u + yrow[k] * orc_bf16_decode(wu[k]);
            }
            float ag = (act == ORC_ACT_SWIGLU) ? orc_silu(g) : orc_gelu_tanh(g);
            a[(int64_t)m * ff + j] = ag * u;
            ma = fmaxf(ma, fabsf(ag * u));
        }
        if (row_amax_y)
            row_amax_y[m] = my;
        if (row_amax_a)
            row_amax_a[m] = ma;
        free(yrow);
    }
#pragma omp parallel for collapse(2) schedule(static)
    for (int m = 0; m < M; m++) {
        for (int n = 0; n < d; n++) {
            const uint16_t *wd = w_down + (int64_t)n * ff;
            const float *arow = a + (int64_t)m * ff;
            float s = 0.0f;
            for (int k = 0; k < ff; k++)
                s = s + arow[k] * orc_bf16_decode(wd[k]);
            out[(int64_t)m * d + n] = rp[(int64_t)m * d + n] + s;
        }
    }
    free(rp);
    free(a);
    return 0;
}
