/*
 * oracle.c - plain fp64 CPU definition of the fused DiT-block elementwise path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent reference the CUDA
 * kernels are checked against.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the library never does, and the
 * two share no code (no headers, helpers or tables).
 *
 * Source of the definitions: the TeleFuser pages on MiniMax H3 name the fused
 * ops and their order but print no formula, so each function states the
 * plain textbook definition it follows:
 *   - RMSNorm fused with the indexed AdaLN modulation (TeleFuser PR #38,
 *     section 2 "Lossless optimizations from PR #37"; TeleFuser PR #23,
 *     section Changes Made, its indexed-modulation kernel);
 *   - Q/K RMSNorm followed by NeoX RoPE (PR #38, section 2; PR #23, section
 *     Changes Made);
 *   - SwiGLU (PR #23, section Changes Made);
 *   - the valid-only gather and the zero-tail merge (PR #38, section 2).
 *
 * Arithmetic: bf16 and fp32 inputs are widened exactly to double; every
 * intermediate is a double; results are returned as doubles, and
 * oracle_round_bf16 rounds them once, to nearest with ties to even.
 * Built with -O2 -ffp-contract=off -fno-fast-math so that no multiply-add is
 * fused behind the reader's back.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ---- bf16 <-> double -------------------------------------------------- */

/* bf16 is the top half of an IEEE binary32 pattern: widen exactly. */
double oracle_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/*
 * Round a double to the nearest bf16 (8 exponent bits, 8 significant bits),
 * ties to even, in one step.  The value is rounded to the nearest integer
 * multiple of its binade's quantum 2^(e-7) (2^-133 below the normal range)
 * with rint() in the default round-to-nearest-even mode; the rounded value is
 * exactly a bf16, so its bf16 bits are the top half of its binary32 bits.
 */
uint16_t oracle_f64_to_bf16(double v) {
    if (isnan(v)) return (uint16_t)(signbit(v) ? 0xFFC0 : 0x7FC0);
    uint16_t sign = signbit(v) ? 0x8000 : 0x0000;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    int ex;
    frexp(a, &ex);                 /* a = m * 2^ex, m in [0.5, 1) */
    int e = ex - 1;                /* a in [2^e, 2^(e+1)) */
    if (e < -126) e = -126;        /* subnormal binade shares the quantum of 2^-126 */
    double quantum = ldexp(1.0, e - 7);
    double n = rint(a / quantum);  /* exact division by a power of two */
    double r = n * quantum;
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    float f = (float)r;            /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | (u >> 16));
}

void oracle_round_bf16(const double* in, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_bf16(in[i]);
}

/* ---- RMSNorm fused with indexed AdaLN modulation ----------------------- */

/*
 * For each row t, with m = mod_idx[t]:
 *   ms   = (1/hidden) * sum_j x[t,j]^2
 *   n[j] = x[t,j] / sqrt(ms + eps) * weight[j]                (RMSNorm)
 *   y[j] = n[j] * (1 + scale[m,j]) + shift[m,j]              (AdaLN modulation)
 * x is [rows, x_row_stride] bf16 (first `hidden` columns used); weight is
 * [hidden]; shift and scale are [n_mod, hidden] fp32; y is [rows, hidden].
 */
void oracle_rmsnorm_adaln_indexed(const uint16_t* x, int64_t x_row_stride, int64_t rows,
                                  int32_t hidden, const float* weight, const float* shift,
                                  const float* scale, const int32_t* mod_idx, int32_t n_mod,
                                  double eps, double* y) {
    (void)n_mod;
    for (int64_t t = 0; t < rows; ++t) {
        const uint16_t* xr = x + t * x_row_stride;
        int32_t m = mod_idx[t];
        double sum_sq = 0.0;
        for (int32_t j = 0; j < hidden; ++j) {
            double v = oracle_bf16_to_f64(xr[j]);
            sum_sq += v * v;
        }
        double ms = sum_sq / (double)hidden;
        double inv_rms = 1.0 / sqrt(ms + eps);
        for (int32_t j = 0; j < hidden; ++j) {
            double n = oracle_bf16_to_f64(xr[j]) * inv_rms * (double)weight[j];
            double s = (double)scale[(int64_t)m * hidden + j];
            double b = (double)shift[(int64_t)m * hidden + j];
            y[t * hidden + j] = n * (1.0 + s) + b;
        }
    }
}

/* ---- Q/K per-head RMSNorm and NeoX rotate-half RoPE -------------------- */

/*
 * Per-head RMSNorm: v is [rows, v_row_stride] bf16 holding n_heads heads of
 * head_dim values each; weight [head_dim] is shared by every head.
 *   out[t,h,d] = v[t,h,d] / sqrt(mean_d v[t,h,:]^2 + eps) * weight[d]
 */
void oracle_head_rmsnorm(const uint16_t* v, int64_t v_row_stride, int64_t rows, int32_t n_heads,
                         int32_t head_dim, const float* weight, double eps, double* out) {
    for (int64_t t = 0; t < rows; ++t) {
        for (int32_t h = 0; h < n_heads; ++h) {
            const uint16_t* vh = v + t * v_row_stride + (int64_t)h * head_dim;
            double* oh = out + (t * n_heads + h) * (int64_t)head_dim;
            double sum_sq = 0.0;
            for (int32_t d = 0; d < head_dim; ++d) {
                double a = oracle_bf16_to_f64(vh[d]);
                sum_sq += a * a;
            }
            double inv_rms = 1.0 / sqrt(sum_sq / (double)head_dim + eps);
            for (int32_t d = 0; d < head_dim; ++d)
                oh[d] = oracle_bf16_to_f64(vh[d]) * inv_rms * (double)weight[d];
        }
    }
}

/*
 * NeoX ("rotate-half") rotary embedding, in place on io [rows, n_heads, head_dim]:
 * dimension i < D/2 is paired with i + D/2, and the pair is turned by the
 * angle theta_i = pos[t] * base^(-2i/D):
 *   out[i]       = a*cos(theta_i) - b*sin(theta_i)
 *   out[i + D/2] = b*cos(theta_i) + a*sin(theta_i)       (a = in[i], b = in[i+D/2])
 */
void oracle_rope_neox(double* io, const int32_t* pos, int64_t rows, int32_t n_heads,
                      int32_t head_dim, double base) {
    int32_t half = head_dim / 2;
    for (int64_t t = 0; t < rows; ++t) {
        for (int32_t h = 0; h < n_heads; ++h) {
            double* vh = io + (t * n_heads + h) * (int64_t)head_dim;
            for (int32_t i = 0; i < half; ++i) {
                double inv_freq = pow(base, -(2.0 * (double)i) / (double)head_dim);
                double angle = (double)pos[t] * inv_freq;
                double c = cos(angle), s = sin(angle);
                double a = vh[i], b = vh[i + half];
                vh[i] = a * c - b * s;
                vh[i + half] = b * c + a * s;
            }
        }
    }
}

/* RMSNorm of every head, then RoPE, for q and for k (each with its own weight). */
void oracle_qk_rmsnorm_rope_neox(const uint16_t* q, const uint16_t* k, int64_t in_row_stride,
                                 int64_t rows, int32_t n_heads, int32_t head_dim,
                                 const float* q_weight, const float* k_weight,
                                 const int32_t* pos, double base, double eps,
                                 double* q_out, double* k_out) {
    oracle_head_rmsnorm(q, in_row_stride, rows, n_heads, head_dim, q_weight, eps, q_out);
    oracle_rope_neox(q_out, pos, rows, n_heads, head_dim, base);
    oracle_head_rmsnorm(k, in_row_stride, rows, n_heads, head_dim, k_weight, eps, k_out);
    oracle_rope_neox(k_out, pos, rows, n_heads, head_dim, base);
}

/* ---- SwiGLU ------------------------------------------------------------ */

/*
 * gate_up is [rows, gu_row_stride] bf16 with the gate in columns [0, ffn) and
 * the up projection in [ffn, 2*ffn):
 *   out[t,j] = silu(g) * u,   silu(g) = g / (1 + exp(-g)),
 *   g = gate_up[t,j], u = gate_up[t,ffn+j].
 */
void oracle_swiglu(const uint16_t* gate_up, int64_t gu_row_stride, int64_t rows, int32_t ffn,
                   double* out) {
    for (int64_t t = 0; t < rows; ++t) {
        const uint16_t* r = gate_up + t * gu_row_stride;
        for (int32_t j = 0; j < ffn; ++j) {
            double g = oracle_bf16_to_f64(r[j]);
            double u = oracle_bf16_to_f64(r[ffn + j]);
            double silu = g / (1.0 + exp(-g));
            out[t * ffn + j] = silu * u;
        }
    }
}

/* ---- valid-only gather and zero-tail merge ----------------------------- */

/* compact[i, :] = padded[i, :] for i < valid_rows (bit copy). */
void oracle_valid_gather(const uint16_t* padded, int64_t valid_rows, int32_t hidden,
                         uint16_t* compact) {
    for (int64_t i = 0; i < valid_rows; ++i)
        for (int32_t j = 0; j < hidden; ++j)
            compact[i * hidden + j] = padded[i * hidden + j];
}

/* padded[i, :] = compact[i, :] for i < valid_rows; +0.0 (0x0000) for the rest. */
void oracle_zero_tail_merge(const uint16_t* compact, int64_t valid_rows, int64_t padded_rows,
                            int32_t hidden, uint16_t* padded) {
    for (int64_t i = 0; i < padded_rows; ++i)
        for (int32_t j = 0; j < hidden; ++j)
            padded[i * hidden + j] = i < valid_rows ? compact[i * hidden + j] : (uint16_t)0x0000;
}
