/*
 * Fairy2i widely-linear layer -- reference oracle.  TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, single-threaded C, double precision.  Only the test suite, the
 * smoke check and the CPU-baseline leg of the benchmark load it; the product
 * library never links or calls it, and the two share no source, header,
 * table or helper.  Every loop follows the method's steps in the order the
 * pages state them, with no blocking, fusion or reordering.
 *
 * Pages cited (by title):
 *   [W2 card]  "Fairy2i-W2" model card (modelscope): sections
 *              "Widely-linear transformation", "Phase-aware complex
 *              quantization", "Recursive residual quantization".
 *   [Note]     "Fairy2i: Ultra-Low-Bit LLM Quantization Using Complex
 *              Weights {±1, ±i}" (zhichai.net reading note): "Step 1:
 *              Widely-linear transformation (Theorem 1)", "Step 2:
 *              Phase-aware quantization", "Step 3: Recursive residual
 *              quantization", "Industry implications: multiplication-free
 *              inference".
 *   [36kr]     "The 2-bit complex model rivals full precision ..." (36kr):
 *              sections 1-3 and the multiplication-free paragraph.
 *
 * Readings where the pages are silent (each is a stated build convention):
 *   - x~ = [Re x ; Im x] stacked as halves; R11 maps Re x -> Re y, R12 Im x ->
 *     Re y, R21 Re x -> Im y, R22 Im x -> Im y (the only stacking under which
 *     the Theorem 1 block formulas hold).
 *   - argmax ties go to the first codeword in the order (+1, -1, +i, -i).
 *   - axis scales are per matrix, per stage, per output row: s_re = mean |Re r|
 *     over the row's real-coded weights, s_im = mean |Im r| over its
 *     imaginary-coded weights; an empty axis has scale 0.  The mean is taken
 *     by the exact integer rule in row_axis_scale() so that any summation
 *     order gives the same float.
 *   - the converted weights and every residual are kept in float32 with one
 *     round-to-nearest per operation (this is the precision in which later
 *     stages' codes are decided, so it is fixed, not left to the oracle).
 *   - U and W are quantized separately, each with its own codes and scales.
 *
 * Canonical code values: 0 = +1, 1 = -1, 2 = +i, 3 = -i.
 * Layouts (all row-major, C order):
 *   R       float  [2n][2m]
 *   U, W    complex as interleaved (re, im) pairs [n][m][2]
 *   codes   uint8  [T][n][m]
 *   scales  float  [T][2][n]    (axis 0 = real, 1 = imaginary)
 *   x       bfloat16 bit patterns [M][2m]  = [Re x | Im x] per token
 *   y       double [M][2n]                 = [Re y | Im y] per token
 *
 * Parity pins live in the test suite; no function here is unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NONFINITE 2

/* ---- Step 1: widely-linear transformation ([Note] Step 1, Theorem 1;
 *      [W2 card] "Widely-linear transformation").
 *   Re U = (R11 + R22)/2   Im U = (R21 - R12)/2
 *   Re W = (R11 - R22)/2   Im W = (R12 + R21)/2
 * with R11 = R[0:n, 0:m], R12 = R[0:n, m:2m], R21 = R[n:2n, 0:m],
 * R22 = R[n:2n, m:2m].  Exact in double for float inputs. */
int oracle_convert_f64(const float *R, int64_t n, int64_t m, double *U, double *W)
{
    if (!R || !U || !W || n <= 0 || m <= 0) return ORACLE_BAD_ARG;
    const int64_t cols = 2 * m;
    for (int64_t j = 0; j < n; ++j) {
        for (int64_t k = 0; k < m; ++k) {
            double r11 = R[j * cols + k];
            double r12 = R[j * cols + m + k];
            double r21 = R[(n + j) * cols + k];
            double r22 = R[(n + j) * cols + m + k];
            double *u = U + 2 * (j * m + k);
            double *w = W + 2 * (j * m + k);
            u[0] = 0.5 * (r11 + r22);
            u[1] = 0.5 * (r21 - r12);
            w[0] = 0.5 * (r11 - r22);
            w[1] = 0.5 * (r12 + r21);
        }
    }
    return ORACLE_OK;
}

/* Same block formulas, each operation rounded to float32 (the sum, then the
 * halving), which is the precision the quantizer starts from. */
int oracle_convert_f32(const float *R, int64_t n, int64_t m, float *U, float *W)
{
    if (!R || !U || !W || n <= 0 || m <= 0) return ORACLE_BAD_ARG;
    const int64_t cols = 2 * m;
    for (int64_t j = 0; j < n; ++j) {
        for (int64_t k = 0; k < m; ++k) {
            float r11 = R[j * cols + k];
            float r12 = R[j * cols + m + k];
            float r21 = R[(n + j) * cols + k];
            float r22 = R[(n + j) * cols + m + k];
            float *u = U + 2 * (j * m + k);
            float *w = W + 2 * (j * m + k);
            float s;
            s = r11 + r22; u[0] = s * 0.5f;
            s = r21 - r12; u[1] = s * 0.5f;
            s = r11 - r22; w[0] = s * 0.5f;
            s = r12 + r21; w[1] = s * 0.5f;
        }
    }
    return ORACLE_OK;
}

/* ---- Step 2: phase-aware projection ([Note] Step 2; [W2 card]
 *      "Phase-aware complex quantization").
 *   b(w) = argmax over s in S = {+1, -1, +i, -i} of Re(w * conj(s)),
 * evaluated literally: conj(s) for the four codewords, one complex product
 * each, the first maximum wins. */
static int project_to_codebook(double re, double im)
{
    static const double conj_s_re[4] = {1.0, -1.0, 0.0, 0.0};
    static const double conj_s_im[4] = {0.0, 0.0, -1.0, 1.0};
    int best = 0;
    double best_val = -INFINITY;
    for (int c = 0; c < 4; ++c) {
        double v = re * conj_s_re[c] - im * conj_s_im[c]; /* Re(w * conj(s)) */
        if (v > best_val) { best_val = v; best = c; }
    }
    return best;
}

/* Axis-wise scale of one row ([Note] Step 2, "axis-wise scaling ... applied
 * separately to real and imaginary parts"; [W2 card]).
 * Mean of |v| over the weights coded on this axis, evaluated exactly:
 *   e    = exponent of the largest |v|  (largest in [2^e, 2^(e+1)))
 *   sum  = sum over those weights of trunc(|v| * 2^(48-e))  in int64
 *   s    = float( double( double(sum) * 2^(e-48) ) / count )
 * Every term is below 2^49, so the int64 sum cannot overflow for m < 2^14.
 * An empty axis, or an axis whose weights are all zero, has scale 0.
 * mean64 (if not NULL) receives the plain double-precision mean. */
static float row_axis_scale(const float *vals, int64_t count, double *mean64)
{
    double vmax = 0.0, plain = 0.0;
    for (int64_t i = 0; i < count; ++i) {
        double v = fabs((double)vals[i]);
        plain += v;
        if (v > vmax) vmax = v;
    }
    if (mean64) *mean64 = count > 0 ? plain / (double)count : 0.0;
    if (count == 0 || vmax == 0.0) return 0.0f;
    int E;
    (void)frexp(vmax, &E); /* vmax = f * 2^E, f in [0.5, 1) */
    int e = E - 1;
    int64_t sum = 0;
    for (int64_t i = 0; i < count; ++i) {
        double v = fabs((double)vals[i]);
        sum += (int64_t)ldexp(v, 48 - e); /* exact scaling, truncation */
    }
    double mean = ldexp((double)sum, e - 48) / (double)count;
    return (float)mean;
}

/* ---- Step 3: recursive residual quantization ([Note] Step 3; [W2 card]
 *      "Recursive residual quantization"; [36kr] section 3).
 *   r^(0) = Z;  for t = 0..T-1:
 *     codes^(t) = b(r^(t))                    elementwise
 *     s_re, s_im per row from r^(t) and codes^(t)
 *     W~^(t)    = s_re * b_re + i * s_im * b_im
 *     r^(t+1)   = r^(t) - W~^(t)               (float32, one rounding)
 * Z, resid: float (re, im) pairs [n][m][2]; resid (optional) holds
 * r^(0..T) as [T+1][n][m][2]; mean64 (optional) [T][2][n].
 * Returns ORACLE_NONFINITE (and writes nothing useful) on NaN/Inf input. */
int oracle_quantize(const float *Z, int64_t n, int64_t m, int32_t T,
                    uint8_t *codes, float *scales, float *resid, double *mean64,
                    float *work /* [n][m][2] */, float *axis_buf /* [m] */)
{
    if (!Z || !codes || !scales || !work || !axis_buf || n <= 0 || m <= 0 || T < 1)
        return ORACLE_BAD_ARG;
    const int64_t nm = n * m;
    for (int64_t i = 0; i < 2 * nm; ++i) {
        if (!isfinite(Z[i])) return ORACLE_NONFINITE;
        work[i] = Z[i];
    }
    if (resid)
        for (int64_t i = 0; i < 2 * nm; ++i) resid[i] = work[i];

    for (int32_t t = 0; t < T; ++t) {
        uint8_t *ct = codes + (int64_t)t * nm;
        /* codes of stage t */
        for (int64_t i = 0; i < nm; ++i)
            ct[i] = (uint8_t)project_to_codebook(work[2 * i], work[2 * i + 1]);
        /* per-row axis scales */
        for (int64_t j = 0; j < n; ++j) {
            for (int axis = 0; axis < 2; ++axis) {
                int64_t cnt = 0;
                for (int64_t k = 0; k < m; ++k) {
                    uint8_t c = ct[j * m + k];
                    int on_axis = axis == 0 ? (c == 0 || c == 1) : (c == 2 || c == 3);
                    if (on_axis) axis_buf[cnt++] = work[2 * (j * m + k) + axis];
                }
                double mu = 0.0;
                float s = row_axis_scale(axis_buf, cnt, &mu);
                scales[((int64_t)t * 2 + axis) * n + j] = s;
                if (mean64) mean64[((int64_t)t * 2 + axis) * n + j] = mu;
            }
        }
        /* dequantized stage and residual update */
        for (int64_t j = 0; j < n; ++j) {
            float s_re = scales[((int64_t)t * 2 + 0) * n + j];
            float s_im = scales[((int64_t)t * 2 + 1) * n + j];
            for (int64_t k = 0; k < m; ++k) {
                int64_t i = j * m + k;
                float wt_re = 0.0f, wt_im = 0.0f; /* W~ = s_re b_re + i s_im b_im */
                switch (ct[i]) {
                case 0: wt_re = s_re; break;
                case 1: wt_re = -s_re; break;
                case 2: wt_im = s_im; break;
                default: wt_im = -s_im; break;
                }
                /* only the coded component changes; the other keeps its bits */
                if (ct[i] <= 1) work[2 * i] = work[2 * i] - wt_re;
                else work[2 * i + 1] = work[2 * i + 1] - wt_im;
            }
        }
        if (resid)
            for (int64_t i = 0; i < 2 * nm; ++i) resid[(int64_t)(t + 1) * 2 * nm + i] = work[i];
    }
    return ORACLE_OK;
}

/* Dequantized sum of stages, Z^ = sum_t (s_re b_re + i s_im b_im), in double.
 * Out: (re, im) pairs [n][m][2]. ([Note] Step 2 dequantization, Step 3 sum.) */
int oracle_dequantize(const uint8_t *codes, const float *scales, int64_t n, int64_t m,
                      int32_t T, double *Zhat)
{
    if (!codes || !scales || !Zhat || n <= 0 || m <= 0 || T < 1) return ORACLE_BAD_ARG;
    const int64_t nm = n * m;
    for (int64_t i = 0; i < 2 * nm; ++i) Zhat[i] = 0.0;
    for (int32_t t = 0; t < T; ++t) {
        for (int64_t j = 0; j < n; ++j) {
            double s_re = scales[((int64_t)t * 2 + 0) * n + j];
            double s_im = scales[((int64_t)t * 2 + 1) * n + j];
            for (int64_t k = 0; k < m; ++k) {
                int64_t i = j * m + k;
                double b_re = 0.0, b_im = 0.0;
                switch (codes[(int64_t)t * nm + i]) {
                case 0: b_re = 1.0; break;
                case 1: b_re = -1.0; break;
                case 2: b_im = 1.0; break;
                default: b_im = -1.0; break;
                }
                Zhat[2 * i] += s_re * b_re;
                Zhat[2 * i + 1] += s_im * b_im;
            }
        }
    }
    return ORACLE_OK;
}

static double bf16_to_double(uint16_t h)
{
    union { uint32_t u; float f; } v;
    v.u = (uint32_t)h << 16;
    return (double)v.f;
}

/* ---- Inference, multiplication-free form ([Note] "Industry implications:
 *      multiplication-free inference"; [36kr] "no multiplication during
 *      inference"; [W2 card] y = Ux + W conj(x)).
 * For each output row j and each matrix X in {U, W} and stage t:
 *   A_re = sum over real-coded k of (+/-) x_k      (adds and subtracts only)
 *   A_im = sum over imaginary-coded k of (+/-) x_k
 * then  U part:  s_re * A_re       + i * s_im * A_im
 *       W part:  s_re * conj(A_re) + i * s_im * conj(A_im)
 * (multiplying by i swaps the real and imaginary parts with a sign flip).
 * y[tok] = [Re y | Im y], double [M][2n]. */
int oracle_linear_mulfree(const uint8_t *codesU, const float *scalesU,
                          const uint8_t *codesW, const float *scalesW,
                          int64_t n, int64_t m, int32_t T,
                          const uint16_t *x, int64_t M, double *y)
{
    if (!codesU || !scalesU || !codesW || !scalesW || !x || !y || n <= 0 || m <= 0 || T < 1 || M < 0)
        return ORACLE_BAD_ARG;
    const int64_t nm = n * m;
    for (int64_t tok = 0; tok < M; ++tok) {
        const uint16_t *xt = x + tok * 2 * m;
        for (int64_t j = 0; j < n; ++j) {
            double y_re = 0.0, y_im = 0.0;
            for (int X = 0; X < 2; ++X) {
                const uint8_t *codes = X == 0 ? codesU : codesW;
                const float *scales = X == 0 ? scalesU : scalesW;
                for (int32_t t = 0; t < T; ++t) {
                    double are_re = 0.0, are_im = 0.0, aim_re = 0.0, aim_im = 0.0;
                    const uint8_t *c = codes + (int64_t)t * nm + j * m;
                    for (int64_t k = 0; k < m; ++k) {
                        double xa = bf16_to_double(xt[k]);
                        double xb = bf16_to_double(xt[m + k]);
                        switch (c[k]) {
                        case 0: are_re += xa; are_im += xb; break;
                        case 1: are_re -= xa; are_im -= xb; break;
                        case 2: aim_re += xa; aim_im += xb; break;
                        default: aim_re -= xa; aim_im -= xb; break;
                        }
                    }
                    double s_re = scales[((int64_t)t * 2 + 0) * n + j];
                    double s_im = scales[((int64_t)t * 2 + 1) * n + j];
                    if (X == 0) {
                        /* s_re * A_re + i * s_im * A_im */
                        y_re += s_re * are_re - s_im * aim_im;
                        y_im += s_re * are_im + s_im * aim_re;
                    } else {
                        /* s_re * conj(A_re) + i * s_im * conj(A_im) */
                        y_re += s_re * are_re + s_im * aim_im;
                        y_im += -s_re * are_im + s_im * aim_re;
                    }
                }
            }
            y[tok * 2 * n + j] = y_re;
            y[tok * 2 * n + n + j] = y_im;
        }
    }
    return ORACLE_OK;
}

/* ---- Inference, dense form: y = U^ x + W^ conj(x) with U^, W^ the
 * dequantized sums of stages and ordinary complex products
 * ([W2 card] "Widely-linear transformation"; [Note] Step 1 and Step 3).
 * Uhat, What: (re, im) pairs [n][m][2] from oracle_dequantize. */
int oracle_linear_dense(const double *Uhat, const double *What, int64_t n, int64_t m,
                        const uint16_t *x, int64_t M, double *y)
{
    if (!Uhat || !What || !x || !y || n <= 0 || m <= 0 || M < 0) return ORACLE_BAD_ARG;
    for (int64_t tok = 0; tok < M; ++tok) {
        const uint16_t *xt = x + tok * 2 * m;
        for (int64_t j = 0; j < n; ++j) {
            double y_re = 0.0, y_im = 0.0;
            for (int64_t k = 0; k < m; ++k) {
                double xr = bf16_to_double(xt[k]);
                double xi = bf16_to_double(xt[m + k]);
                double ur = Uhat[2 * (j * m + k)], ui = Uhat[2 * (j * m + k) + 1];
                double wr = What[2 * (j * m + k)], wi = What[2 * (j * m + k) + 1];
                /* U x */
                y_re += ur * xr - ui * xi;
                y_im += ur * xi + ui * xr;
                /* W conj(x) = (wr + i wi)(xr - i xi) */
                y_re += wr * xr + wi * xi;
                y_im += wi * xr - wr * xi;
            }
            y[tok * 2 * n + j] = y_re;
            y[tok * 2 * n + n + j] = y_im;
        }
    }
    return ORACLE_OK;
}

/* ---- Gradient of the layer with respect to its input (for quantization-aware
 * training with the straight-through estimator: [Note] Step 3 and the QAT
 * paragraph; [W2 card] y = Ux + W conj(x)).
 * For a real loss L and g = dL/dRe y + i dL/dIm y (per token, complex [n]),
 *   dL/dRe x + i dL/dIm x = U^^H g + W^^T conj(g)
 * (the real form of the layer is a real matrix; its transpose is the real
 * form of (U^^H, W^^T)).  Multiplication-free in the codes: per row j and
 * stage t the gradient is scaled once per axis,
 *   U:  h_re = s_re g_j,          h_im = s_im (-i g_j)
 *   W:  h_re = s_re conj(g_j),    h_im = s_im (i conj(g_j))
 * and every code adds or subtracts the h of its axis into its column:
 *   gx_k += sign(code_jk) * (code_jk real-axis ? h_re : h_im).
 * g: float [M][2n] = [dRe y | dIm y];  gx: double [M][2m] = [dRe x | dIm x]. */
int oracle_linear_grad_x(const uint8_t *codesU, const float *scalesU,
                         const uint8_t *codesW, const float *scalesW,
                         int64_t n, int64_t m, int32_t T,
                         const float *g, int64_t M, double *gx)
{
    if (!codesU || !scalesU || !codesW || !scalesW || !g || !gx || n <= 0 || m <= 0 || T < 1 || M < 0)
        return ORACLE_BAD_ARG;
    const int64_t nm = n * m;
    for (int64_t tok = 0; tok < M; ++tok) {
        const float *gt = g + tok * 2 * n;
        double *out = gx + tok * 2 * m;
        for (int64_t k = 0; k < 2 * m; ++k) out[k] = 0.0;
        for (int X = 0; X < 2; ++X) {
            const uint8_t *codes = X == 0 ? codesU : codesW;
            const float *scales = X == 0 ? scalesU : scalesW;
            for (int32_t t = 0; t < T; ++t) {
                for (int64_t j = 0; j < n; ++j) {
                    const double ga = gt[j], gb = gt[n + j];   /* g_j = ga + i gb */
                    const double s_re = scales[((int64_t)t * 2 + 0) * n + j];
                    const double s_im = scales[((int64_t)t * 2 + 1) * n + j];
                    double hre_a, hre_b, him_a, him_b;         /* h = a + i b */
                    if (X == 0) {
                        hre_a = s_re * ga;  hre_b = s_re * gb;     /* s_re g */
                        him_a = s_im * gb;  him_b = -s_im * ga;    /* s_im (-i)(ga + i gb) */
                    } else {
                        hre_a = s_re * ga;  hre_b = -s_re * gb;    /* s_re (ga - i gb) */
                        him_a = s_im * gb;  him_b = s_im * ga;     /* s_im i (ga - i gb) */
                    }
                    const uint8_t *c = codes + (int64_t)t * nm + j * m;
                    for (int64_t k = 0; k < m; ++k) {
                        switch (c[k]) {
                        case 0: out[k] += hre_a; out[m + k] += hre_b; break;
                        case 1: out[k] -= hre_a; out[m + k] -= hre_b; break;
                        case 2: out[k] += him_a; out[m + k] += him_b; break;
                        default: out[k] -= him_a; out[m + k] -= him_b; break;
                        }
                    }
                }
            }
        }
    }
    return ORACLE_OK;
}
