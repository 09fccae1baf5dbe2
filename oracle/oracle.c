/*
 * oracle.c - plain, slow CPU reference for the NVFP4 sigmoid-routed MoE decode
 * path and the NVFP4 weight-only lm_head.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file; only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline
 * leg do. It shares no code with the CUDA library (csrc/): every codec,
 * quantiser, router and matrix routine below is written out here on its own.
 *
 * Sources (web pages on serving an NVFP4 Nemotron-3.5 MoE model):
 *  [worklog]  "Let's optimize Nemotron 3.5 Lightning - a worklog"
 *             Step 1 (NVFP4 = 4-bit values, group size 16; W4A16 keeps 16-bit
 *             activations), Step 3 (routed experts W4A4 with dynamic NVFP4
 *             activation quantisation; router kept high precision), Step 4
 *             (lm_head NVFP4 weight-only, 131072 x 2688), Interlude (decode is a
 *             weight stream).
 *  [card-w4a4] "nemotron35-w4a4-v13" model card, precision table (routed
 *             experts NVFP4 block 16; lm_head NVFP4 weight-only).
 *  [card-int4] "NVIDIA-Nemotron-3.5-Lightning-30B-A3B-W4A16" model card,
 *             "Checkpoint layout" (experts are per-expert up_proj/down_proj with
 *             no gate_proj: a non-gated MLP) and "Left at bfloat16" (router
 *             .gate plus its fp32 e_score_correction_bias).
 *  [super-q]  "Quantization (PTQ + QAD)" (Nemotron 3.5 Super), Precision
 *             Recipes table (router / gate compute in FP32; MoE and
 *             shared-expert GEMMs NVFP4), Deployment (Blackwell runs W4A4).
 *
 * Where the pages are silent the readings used are stated at each function:
 * NVFP4 global = tensor amax / (6*448), block scale = E4M3(block amax / 6 /
 * global), code = E2M1(x / (scale * global)); sigmoid router with the
 * correction bias used for selection only and the selected sigmoids
 * renormalised to sum 1; relu^2 activation; bf16 intermediate.
 *
 * Arithmetic: quantiser decisions are taken in IEEE binary32, one operation at
 * a time (build with -ffp-contract=off); every dot product is accumulated in
 * binary64 over exactly dequantised operands.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Codecs                                                                   */
/* ------------------------------------------------------------------------ */

/* E2M1 (OCP FP4): bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent field 0 is subnormal: value = mantissa * 0.5. No Inf/NaN. */
double orc_e2m1_value(int code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* E4M3 "FN" (OCP FP8): bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0
 * mantissa; exponent 0 is subnormal (m * 2^-9); exponent 15 with mantissa 7 is
 * NaN; no infinities; largest finite 448. */
double orc_e4m3_value(int byte) {
    int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m, -9);
    else mag = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Nearest E2M1 value by exhaustive search; an exact tie goes to the even code
 * (mantissa bit 0); beyond 6 the result saturates to 6. The sign of the input
 * is kept even when the magnitude rounds to 0 (reading: -0.2 -> code 0x8). */
int orc_e2m1_encode(float v) {
    double a = fabs((double)v);
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c < 8; ++c) {
        double d = fabs(orc_e2m1_value(c) - a);
        if (d < bestd || (d == bestd && (c & 1) == 0)) { best = c; bestd = d; }
    }
    return best | (signbit(v) ? 8 : 0);
}

/* Nearest finite E4M3 value by exhaustive search over codes 0x00..0x7E, ties
 * to the even code, saturating at 448 ("satfinite"). */
int orc_e4m3_encode(float v) {
    double a = fabs((double)v);
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(orc_e4m3_value(c) - a);
        if (d < bestd || (d == bestd && (c & 1) == 0)) { best = c; bestd = d; }
    }
    return best | (signbit(v) ? 0x80 : 0);
}

double orc_bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a binary64 value to the nearest bfloat16 (8 significant bits), ties to
 * even, in a single rounding. Finite inputs only. */
uint16_t orc_bf16_round(double x) {
    double q;
    if (x == 0.0) {
        q = x;
    } else {
        int e;
        double m = frexp(fabs(x), &e); /* |x| = m 2^e, m in [0.5, 1) */
        if (e - 1 < -126) {            /* below the normal range: fixed 2^-133 grid */
            q = nearbyint(fabs(x) * ldexp(1.0, 133)) * ldexp(1.0, -133);
        } else {
            q = ldexp(nearbyint(m * 256.0), e - 8);
        }
        if (x < 0) q = -q;
    }
    float f = (float)q; /* exact: q has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------ */
/* NVFP4 quantise / dequantise                                              */
/* ------------------------------------------------------------------------ */

/* One row segment of `cols` values quantised with global scale g, following
 * the NVFP4 recipe (block 16: worklog Step 1, card-w4a4 precision table):
 *   s_b    = E4M3( (amax_b / 6) / g )          two binary32 divisions
 *   d_b    = value(s_b) * g                    one binary32 multiply
 *   code_i = E2M1( x_i / d_b )                 one binary32 division
 * Reading: a block whose d_b is 0 (all-zero block, or a scale that rounds to
 * 0) gets all codes 0. Element 2j is the low nibble of byte j. */
static void orc_quantize_row(const float* x, int64_t cols, float g, uint8_t* codes,
                             uint8_t* scales) {
    memset(codes, 0, (size_t)(cols / 2));
    for (int64_t b = 0; b < cols / 16; ++b) {
        const float* xb = x + b * 16;
        float bamax = 0.0f;
        for (int i = 0; i < 16; ++i) {
            float a = fabsf(xb[i]);
            if (a > bamax) bamax = a;
        }
        int s = 0;
        if (g > 0.0f) {
            float t = bamax / 6.0f;
            float v = t / g;
            s = orc_e4m3_encode(v);
        }
        scales[b] = (uint8_t)s;
        float d = (float)orc_e4m3_value(s) * g;
        for (int i = 0; i < 16; ++i) {
            int c = 0;
            if (d != 0.0f) {
                float r = xb[i] / d;
                c = orc_e2m1_encode(r);
            }
            codes[b * 8 + i / 2] |= (uint8_t)(c << (4 * (i & 1)));
        }
    }
}

static float orc_amax(const float* x, int64_t n) {
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > m) m = a;
    }
    return m;
}

/* Quantise x[rows][cols] (cols % 16 == 0) to NVFP4.
 * mode 0: one global for the tensor, g = amax / 2688 (= 6 * 448), written to g_io[0];
 * mode 1: one global per row (dynamic activation quantisation, worklog Step 3),
 *         written to g_io[r];
 * mode 2: the global is given in g_io[0].
 * Returns 0, or -1 on a bad argument. */
int orc_quantize(const float* x, int64_t rows, int64_t cols, int mode, float* g_io,
                 uint8_t* codes, uint8_t* scales) {
    if (cols % 16 != 0 || rows < 0 || mode < 0 || mode > 2) return -1;
    float gt = 0.0f;
    if (mode == 0) {
        gt = orc_amax(x, rows * cols) / 2688.0f;
        g_io[0] = gt;
    } else if (mode == 2) {
        gt = g_io[0];
    }
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float g = gt;
        if (mode == 1) {
            g = orc_amax(x + r * cols, cols) / 2688.0f;
            g_io[r] = g;
        }
        orc_quantize_row(x + r * cols, cols, g, codes + r * (cols / 2), scales + r * (cols / 16));
    }
    return 0;
}

/* x_hat = E2M1 value * E4M3 value * g, exact in binary64. */
void orc_dequantize(const uint8_t* codes, const uint8_t* scales, const float* g, int per_row,
                    int64_t rows, int64_t cols, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double gr = per_row ? (double)g[r] : (double)g[0];
        for (int64_t i = 0; i < cols; ++i) {
            int byte = codes[r * (cols / 2) + i / 2];
            int c = (i & 1) ? (byte >> 4) : (byte & 15);
            double s = orc_e4m3_value(scales[r * (cols / 16) + i / 16]);
            out[r * cols + i] = orc_e2m1_value(c) * s * gr;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Router                                                                   */
/* ------------------------------------------------------------------------ */

/* Sigmoid router with correction bias (card-int4 "Left at bfloat16": .gate +
 * fp32 e_score_correction_bias; super-q: router compute FP32; this oracle
 * computes it exactly, in binary64):
 *   z_e = sum_i h_i Wg[e][i]; sigma_e = 1 / (1 + exp(-z_e)); c_e = sigma_e + bias_e
 *   select the k largest c_e (reading: an exact tie goes to the lower index);
 *   w_j = sigma_{e_j} / sum_l sigma_{e_l} (the unbiased sigmoids, renormalised).
 * Outputs per token: idx[k] and w[k] in descending c order; z[E], c[E]; and
 * tau[E], an a-priori bound on how far a binary32 evaluation of c_e may sit
 * from the exact one: 0.25 * (4 sqrt(H) 2^-24 sum_i |h_i Wg_ei| +
 * 2 * 2^-8 max_i |h_i Wg_ei|) + 2^-22 (the probabilistic dot-product bound,
 * plus one-ulp bf16 differences in up to two inputs from an RMS norm taken in
 * binary32, times max sigma' = 1/4, plus sigmoid and bias-add rounding). */
void orc_route(const uint16_t* h, int32_t T, int32_t H, const float* Wg, const float* bias,
               int32_t E, int32_t k, int32_t* idx, double* w, double* z, double* c,
               double* tau) {
#pragma omp parallel for schedule(static)
    for (int32_t t = 0; t < T; ++t) {
        double* zt = z + (int64_t)t * E;
        double* ct = c + (int64_t)t * E;
        double* taut = tau + (int64_t)t * E;
        double* sg = (double*)malloc(sizeof(double) * (size_t)E);
        unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
        for (int32_t e = 0; e < E; ++e) {
            double acc = 0.0, aacc = 0.0, amax = 0.0;
            for (int32_t i = 0; i < H; ++i) {
                double p = orc_bf16_value(h[(int64_t)t * H + i]) * (double)Wg[(int64_t)e * H + i];
                acc += p;
                aacc += fabs(p);
                if (fabs(p) > amax) amax = fabs(p);
            }
            zt[e] = acc;
            sg[e] = 1.0 / (1.0 + exp(-acc));
            ct[e] = sg[e] + (double)bias[e];
            taut[e] = 0.25 * (4.0 * sqrt((double)H) * ldexp(1.0, -24) * aacc + 2.0 * ldexp(1.0, -8) * amax) +
                      ldexp(1.0, -22);
        }
        double ssum = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || ct[e] > ct[best]) best = e;
            }
            taken[best] = 1;
            idx[(int64_t)t * k + j] = best;
            ssum += sg[best];
        }
        for (int32_t j = 0; j < k; ++j)
            w[(int64_t)t * k + j] = sg[idx[(int64_t)t * k + j]] / ssum;
        free(sg);
        free(taken);
    }
}

/* ------------------------------------------------------------------------ */
/* Expert MLP, MoE layer, lm_head                                           */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint8_t* codes;  /* [n][k/2] */
    const uint8_t* scales; /* [n][k/16] */
    float g;               /* per-tensor global */
    int64_t n, k;
} orc_mat;

/* y[n] = sum_j W_hat[n][j] * x[j], W_hat dequantised exactly, binary64. */
static void orc_matvec(const orc_mat* W, const double* x, double* y) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < W->n; ++r) {
        double acc = 0.0;
        const uint8_t* cr = W->codes + r * (W->k / 2);
        const uint8_t* sr = W->scales + r * (W->k / 16);
        for (int64_t j = 0; j < W->k; ++j) {
            int c = (j & 1) ? (cr[j / 2] >> 4) : (cr[j / 2] & 15);
            double wv = orc_e2m1_value(c) * orc_e4m3_value(sr[j / 16]) * (double)W->g;
            acc += wv * x[j];
        }
        y[r] = acc;
    }
}

/* The value a GEMM sees for one activation row held as bf16 values:
 * W4A16 - the bf16 values themselves (worklog Step 1);
 * W4A4  - the row quantised to NVFP4 with its own global (dynamic, worklog
 *         Step 3) and dequantised. */
static void orc_activation(const double* xin, int64_t n, int w4a4, double* xout) {
    if (n <= 0) return;
    if (!w4a4) {
        memcpy(xout, xin, sizeof(double) * (size_t)n);
        return;
    }
    float* xf = (float*)malloc(sizeof(float) * (size_t)n);
    uint8_t* cd = (uint8_t*)malloc((size_t)(n / 2));
    uint8_t* sc = (uint8_t*)malloc((size_t)(n / 16));
    for (int64_t i = 0; i < n; ++i) xf[i] = (float)xin[i]; /* exact: inputs are bf16 values */
    float g = orc_amax(xf, n) / 2688.0f;
    orc_quantize_row(xf, n, g, cd, sc);
    for (int64_t i = 0; i < n; ++i) {
        int byte = cd[i / 2];
        int c = (i & 1) ? (byte >> 4) : (byte & 15);
        xout[i] = orc_e2m1_value(c) * orc_e4m3_value(sc[i / 16]) * (double)g;
    }
    free(xf);
    free(cd);
    free(sc);
}

/* Non-gated expert MLP (card-int4 "Checkpoint layout": up_proj and down_proj
 * only): u = up . x; a = bf16(relu(u)^2) (reading: relu^2 activation, bf16
 * intermediate between the two GEMMs); y = down . a'. In W4A4 both x and a are
 * dynamically quantised per row before their GEMM. */
static void orc_expert(const orc_mat* up, const orc_mat* down, const double* x_bf16vals, int w4a4,
                       double* y) {
    int64_t I = up->n, H = up->k;
    double* xa = (double*)malloc(sizeof(double) * (size_t)H);
    double* u = (double*)malloc(sizeof(double) * (size_t)I);
    double* a = (double*)malloc(sizeof(double) * (size_t)I);
    double* aa = (double*)malloc(sizeof(double) * (size_t)I);
    orc_activation(x_bf16vals, H, w4a4, xa);
    orc_matvec(up, xa, u);
    for (int64_t i = 0; i < I; ++i) {
        double r = u[i] > 0.0 ? u[i] : 0.0;
        a[i] = orc_bf16_value(orc_bf16_round(r * r));
    }
    orc_activation(a, I, w4a4, aa);
    orc_matvec(down, aa, y);
    free(xa);
    free(u);
    free(a);
    free(aa);
}

/* RMS normalisation with unit weight of each bf16 row (the per-block input
 * norm of the pages' pre-norm hybrid model, whose norms stay in bf16:
 * card-int4 "Left at bfloat16"): y_i = bf16( x_i / sqrt(mean_j x_j^2 + eps) ),
 * binary64 arithmetic, one rounding. */
void orc_rms_norm(const uint16_t* h, int32_t T, int64_t H, double eps, uint16_t* out) {
    for (int32_t t = 0; t < T; ++t) {
        double ss = 0.0;
        for (int64_t i = 0; i < H; ++i) {
            double x = orc_bf16_value(h[(int64_t)t * H + i]);
            ss += x * x;
        }
        double inv = 1.0 / sqrt(ss / (double)H + eps);
        for (int64_t i = 0; i < H; ++i)
            out[(int64_t)t * H + i] = orc_bf16_round(orc_bf16_value(h[(int64_t)t * H + i]) * inv);
    }
}

/* One MoE layer for T tokens given the routing (idx, w):
 *   out_t = bf16( shared(x_t) + sum_j w_tj * expert_{idx_tj}(x_t) [+ residual_t] )
 * with one rounding at the end. `up`/`down` are indexed by expert id; only the
 * experts named in idx are read. The shared expert sees the same activation
 * treatment as the routed ones (super-q: MoE + shared-expert GEMMs NVFP4).
 * residual (optional, bf16 [T][H]) is added before the rounding; out_f64
 * (optional) receives the value before the final rounding. */
void orc_moe_layer(const uint16_t* h, int32_t T, int32_t k, const int32_t* idx, const double* w,
                   const orc_mat* up, const orc_mat* down, const orc_mat* sh_up,
                   const orc_mat* sh_down, int32_t w4a4, const uint16_t* residual, uint16_t* out_bf16,
                   double* out_f64) {
    int64_t H = sh_up->k;
    double* x = (double*)malloc(sizeof(double) * (size_t)H);
    double* y = (double*)malloc(sizeof(double) * (size_t)H);
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
    for (int32_t t = 0; t < T; ++t) {
        for (int64_t i = 0; i < H; ++i) x[i] = orc_bf16_value(h[(int64_t)t * H + i]);
        orc_expert(sh_up, sh_down, x, w4a4, acc);
        for (int32_t j = 0; j < k; ++j) {
            int32_t e = idx[(int64_t)t * k + j];
            orc_expert(&up[e], &down[e], x, w4a4, y);
            double wj = w[(int64_t)t * k + j];
            for (int64_t i = 0; i < H; ++i) acc[i] += wj * y[i];
        }
        for (int64_t i = 0; i < H; ++i) {
            double v = acc[i] + (residual ? orc_bf16_value(residual[(int64_t)t * H + i]) : 0.0);
            if (out_f64) out_f64[(int64_t)t * H + i] = v;
            out_bf16[(int64_t)t * H + i] = orc_bf16_round(v);
        }
    }
    free(x);
    free(y);
    free(acc);
}

/* NVFP4 weight-only lm_head (worklog Step 4; card-w4a4 "lm_head NVFP4
 * weight-only (W4A16)"): logits[t][v] = sum_j W_hat[v][j] * h_t[j], binary64. */
void orc_lm_head(const orc_mat* W, const uint16_t* h, int32_t T, double* logits) {
    double* x = (double*)malloc(sizeof(double) * (size_t)W->k);
    for (int32_t t = 0; t < T; ++t) {
        for (int64_t i = 0; i < W->k; ++i) x[i] = orc_bf16_value(h[(int64_t)t * W->k + i]);
        orc_matvec(W, x, logits + (int64_t)t * W->n);
    }
    free(x);
}

/* lm_head restricted to the listed rows (for sampled checks at full size). */
void orc_lm_head_rows(const orc_mat* W, const uint16_t* h, int32_t T, const int64_t* rows,
                      int64_t nrows, double* out /* [T][nrows] */) {
    for (int32_t t = 0; t < T; ++t) {
#pragma omp parallel for schedule(static)
        for (int64_t q = 0; q < nrows; ++q) {
            int64_t r = rows[q];
            double acc = 0.0;
            const uint8_t* cr = W->codes + r * (W->k / 2);
            const uint8_t* sr = W->scales + r * (W->k / 16);
            for (int64_t j = 0; j < W->k; ++j) {
                int c = (j & 1) ? (cr[j / 2] >> 4) : (cr[j / 2] & 15);
                double wv = orc_e2m1_value(c) * orc_e4m3_value(sr[j / 16]) * (double)W->g;
                acc += wv * orc_bf16_value(h[(int64_t)t * W->k + j]);
            }
            out[(int64_t)t * nrows + q] = acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* FP8 (E4M3) per-tensor W8A8: the shared expert of the W4A4 card            */
/* ------------------------------------------------------------------------ */

/* Quantise x[rows][cols] to E4M3 with one FP32 scale (W4A4 card precision
 * table: "Mamba in_proj / out_proj, shared experts: FP8 per-tensor W8A8";
 * worklog Step 3 yaml: shared experts "num_bits: e4m3"):
 *   g   = amax / 448                  one binary32 division
 *   q_i = E4M3_rn_satfinite( x_i / g )   one binary32 division
 * Reading: g = 0 (an all-zero tensor or row) gives q = 0 with the sign kept.
 * mode 0: one scale for the tensor (weights), written to g_io[0];
 * mode 1: one scale per row (activations: the dynamic per-token reading of
 *         "per-tensor" for the inputs, as for NVFP4), written to g_io[r];
 * mode 2: the scale is given in g_io[0]. Returns 0, or -1 on a bad argument. */
int orc_fp8_quantize(const float* x, int64_t rows, int64_t cols, int mode, float* g_io, uint8_t* q) {
    if (rows < 0 || cols < 1 || mode < 0 || mode > 2) return -1;
    float gt = 0.0f;
    if (mode == 0) {
        gt = orc_amax(x, rows * cols) / 448.0f;
        g_io[0] = gt;
    } else if (mode == 2) {
        gt = g_io[0];
    }
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float g = gt;
        if (mode == 1) {
            g = orc_amax(x + r * cols, cols) / 448.0f;
            g_io[r] = g;
        }
        for (int64_t i = 0; i < cols; ++i) {
            const float v = x[r * cols + i];
            q[r * cols + i] = (uint8_t)(g == 0.0f ? (signbit(v) ? 0x80 : 0) : orc_e4m3_encode(v / g));
        }
    }
    return 0;
}

/* y[n] = sum_j E4M3(W[n][j]) * x[j] (binary64; the scales are applied by the
 * caller). */
static void orc_fp8_matvec(const uint8_t* W, int64_t n, int64_t k, const double* x, double* y) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        double acc = 0.0;
        for (int64_t j = 0; j < k; ++j) acc += orc_e4m3_value(W[r * k + j]) * x[j];
        y[r] = acc;
    }
}

/* The shared expert in FP8 W8A8 for T tokens (non-gated, as the NVFP4 one:
 * card-int4 "Checkpoint layout"):
 *   x_q = FP8(x) per row, scale g_x;   u = g_up * g_x * (W_up . E4M3(x_q))
 *   a   = bf16(relu(u)^2)              (the bf16 intermediate, reading 5)
 *   a_q = FP8(a) per row, scale g_a;   y = g_dn * g_a * (W_dn . E4M3(a_q))
 * x: bf16 [T][H] (already normalised when the block is pre-normed);
 * W_up [S][H], W_dn [H][S] E4M3 with per-tensor scales g_up, g_dn.
 * Outputs y [T][H] (binary64) and the bf16 intermediate act [T][S]. */
void orc_shared_fp8(const uint16_t* x, int32_t T, int64_t H, int64_t S, const uint8_t* w_up, float g_up,
                    const uint8_t* w_dn, float g_dn, double* y, uint16_t* act) {
    float* xf = (float*)malloc(sizeof(float) * (size_t)(H > S ? H : S));
    uint8_t* q = (uint8_t*)malloc((size_t)(H > S ? H : S));
    double* v = (double*)malloc(sizeof(double) * (size_t)(H > S ? H : S));
    double* u = (double*)malloc(sizeof(double) * (size_t)S);
    for (int32_t t = 0; t < T; ++t) {
        float gx = 0.0f, ga = 0.0f;
        for (int64_t i = 0; i < H; ++i) xf[i] = (float)orc_bf16_value(x[(int64_t)t * H + i]);
        orc_fp8_quantize(xf, 1, H, 1, &gx, q);
        for (int64_t i = 0; i < H; ++i) v[i] = orc_e4m3_value(q[i]);
        orc_fp8_matvec(w_up, S, H, v, u);
        for (int64_t j = 0; j < S; ++j) {
            double uj = u[j] * (double)g_up * (double)gx;
            double r = uj > 0.0 ? uj : 0.0;
            uint16_t b = orc_bf16_round(r * r);
            act[(int64_t)t * S + j] = b;
            xf[j] = (float)orc_bf16_value(b);
        }
        orc_fp8_quantize(xf, 1, S, 1, &ga, q);
        for (int64_t j = 0; j < S; ++j) v[j] = orc_e4m3_value(q[j]);
        orc_fp8_matvec(w_dn, H, S, v, y + (int64_t)t * H);
        for (int64_t i = 0; i < H; ++i) y[(int64_t)t * H + i] *= (double)g_dn * (double)ga;
    }
    free(xf);
    free(q);
    free(v);
    free(u);
}

void orc_set_threads(int n) {
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : 1);
#else
    (void)n;
#endif
}

int orc_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
