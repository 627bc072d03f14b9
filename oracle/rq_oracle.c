/*
 * rq_oracle.c -- plain CPU oracle (TEST INFRASTRUCTURE ONLY; see
 * rq_oracle.h for the sources and the definition of every step).
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared (no fast-math):
 * each `float` expression below is one IEEE single operation, rounded to
 * nearest even, and nothing is fused into an FMA.
 */
#include "rq_oracle.h"

#include <math.h>
#include <stddef.h>

/* ---------------------------------------------------------------------------
 * Binary floating-point formats.
 *
 * A format with a p-bit significand (hidden bit included) and smallest normal
 * exponent emin represents, per binade [2^e, 2^(e+1)) with e >= emin, the
 * integers n in [2^(p-1), 2^p) times the quantum 2^(e-p+1); below 2^emin
 * (subnormals) it keeps the quantum 2^(emin-p+1).  Round-to-nearest-even picks
 * the nearest such multiple and, on a tie, the one whose integer n is even.
 *
 * The magnitude code is the bit pattern without the sign: the exponent field
 * above p-1 mantissa bits.  With qmin = emin-p+1 the value n*2^q has code
 * n + (q - qmin) * 2^(p-1): in the subnormal binade (q = qmin) that is n
 * itself, and a significand that rounded up to 2^p carries into the next
 * exponent field by itself.
 * ------------------------------------------------------------------------ */
typedef struct { int p; int emin; } fmt_t;

static const fmt_t F_BF16 = {8, -126};
static const fmt_t F_FP16 = {11, -14};
static const fmt_t F_E4M3 = {4, -6};
static const fmt_t F_E2M1 = {2, 0};

/* Round a finite a >= 0 to the nearest representable magnitude (ties to even)
 * with an unbounded exponent range above; returns its magnitude code. */
static uint32_t round_magnitude(double a, fmt_t f)
{
    if (a == 0.0) return 0;
    int E;
    (void)frexp(a, &E);               /* a = m * 2^E, 0.5 <= m < 1 */
    int lead = E - 1;                 /* a lies in [2^lead, 2^(lead+1)) */
    if (lead < f.emin) lead = f.emin; /* subnormals: quantum of the lowest binade */
    int q = lead - (f.p - 1);         /* exponent of the quantum */
    double n = nearbyint(ldexp(a, -q)); /* exact scaling; RNE to an integer */
    int qmin = f.emin - (f.p - 1);
    return (uint32_t)n + ((uint32_t)(q - qmin) << (f.p - 1));
}

static double decode_magnitude(uint32_t code, fmt_t f)
{
    uint32_t half = 1u << (f.p - 1);
    uint32_t e = code >> (f.p - 1), m = code & (half - 1);
    int qmin = f.emin - (f.p - 1);
    if (e == 0) return ldexp((double)m, qmin);
    return ldexp((double)(half + m), qmin + (int)e - 1);
}

/* ---- IEEE bfloat16 (1/8/7) and binary16 (1/5/10) ---- */
static double ieee16_decode(uint16_t b, fmt_t f, uint16_t exp_mask)
{
    double sign = (b & 0x8000u) ? -1.0 : 1.0;
    uint16_t mag = b & 0x7FFFu;
    if ((mag & exp_mask) == exp_mask)
        return (mag & (uint16_t)~exp_mask) ? NAN : sign * INFINITY;
    return sign * decode_magnitude(mag, f);
}

static uint16_t ieee16_encode(double v, fmt_t f, uint16_t exp_mask,
                              uint16_t qnan)
{
    if (isnan(v)) return qnan;
    uint16_t s = signbit(v) ? 0x8000u : 0;
    double a = fabs(v);
    if (isinf(a)) return s | exp_mask;
    uint32_t c = round_magnitude(a, f);
    if (c >= exp_mask) c = exp_mask; /* rounded past the largest finite: inf */
    return (uint16_t)(s | c);
}

double oracle_bf16_to_double(uint16_t b) { return ieee16_decode(b, F_BF16, 0x7F80u); }
double oracle_fp16_to_double(uint16_t h) { return ieee16_decode(h, F_FP16, 0x7C00u); }
uint16_t oracle_bf16_from_double(double v) { return ieee16_encode(v, F_BF16, 0x7F80u, 0x7FC0u); }
uint16_t oracle_fp16_from_double(double v) { return ieee16_encode(v, F_FP16, 0x7C00u, 0x7E00u); }

/* ---- OCP FP8 E4M3 ("fn"): no infinities, S.1111.111 is NaN, max 448 ---- */
double oracle_e4m3_to_double(uint8_t c)
{
    double sign = (c & 0x80u) ? -1.0 : 1.0;
    uint8_t mag = c & 0x7Fu;
    if (mag == 0x7Fu) return NAN;
    return sign * decode_magnitude(mag, F_E4M3);
}

uint8_t oracle_e4m3_from_double(double v)
{
    if (isnan(v)) return 0x7Fu;
    uint8_t s = signbit(v) ? 0x80u : 0;
    double a = fabs(v);
    if (a >= 448.0) return s | 0x7Eu;          /* satfinite, inf included */
    uint32_t c = round_magnitude(a, F_E4M3);
    if (c > 0x7Eu) c = 0x7Eu;
    return (uint8_t)(s | c);
}

/* ---- OCP FP4 E2M1: magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}, no inf/NaN ---- */
double oracle_e2m1_to_double(uint8_t nib)
{
    double sign = (nib & 0x8u) ? -1.0 : 1.0;
    return sign * decode_magnitude(nib & 0x7u, F_E2M1);
}

uint8_t oracle_e2m1_from_double(double v)
{
    /* The fused path never produces NaN here (finite y times a finite
     * factor); the largest magnitude is returned for it. */
    if (isnan(v)) return 0x7u;
    uint8_t s = signbit(v) ? 0x8u : 0;
    double a = fabs(v);
    if (a >= 6.0) return s | 0x7u;             /* satfinite */
    uint32_t c = round_magnitude(a, F_E2M1);
    if (c > 0x7u) c = 0x7u;
    return (uint8_t)(s | c);
}

void oracle_dt_from_double_array(int dt, const double *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = dt == RQO_BF16 ? oracle_bf16_from_double(v[i]) : oracle_fp16_from_double(v[i]);
}

void oracle_dt_to_double_array(int dt, const uint16_t *b, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = dt == RQO_BF16 ? oracle_bf16_to_double(b[i]) : oracle_fp16_to_double(b[i]);
}

void oracle_e4m3_from_double_array(const double *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_from_double(v[i]);
}

void oracle_e2m1_from_double_array(const double *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_from_double(v[i]);
}

/* value of a stored element as fp32 (exact for bf16 and fp16) */
static float ld_dt(int dt, uint16_t b)
{
    return (float)(dt == RQO_BF16 ? oracle_bf16_to_double(b) : oracle_fp16_to_double(b));
}

/* fp32 value rounded to the storage dtype */
static uint16_t st_dt(int dt, float v)
{
    return dt == RQO_BF16 ? oracle_bf16_from_double((double)v) : oracle_fp16_from_double((double)v);
}

/* rstd = 1 / sqrt(mean of squares + eps) from the double sum of squares,
 * with every step after the sum one fp32 rounding. */
static float rms_rstd(double sum_sq, int64_t n, float eps)
{
    float ss = (float)sum_sq;
    float ms = ss / (float)n;
    float t = ms + eps;
    float rt = sqrtf(t);
    float rstd = 1.0f / rt;
    return rstd;
}

/* RMSNorm of one stored row s (steps 2 and 3 below): the sum of squares of
 * s, rstd, then y = (s * rstd) * weight stored in dtype (if y is given). */
static void rmsnorm_row(int dt, const uint16_t *sr, const uint16_t *w, float eps,
                        int64_t hidden, uint16_t *yr)
{
    double sum_sq = 0.0;
    for (int64_t i = 0; i < hidden; ++i) {
        double v = (double)ld_dt(dt, sr[i]);
        sum_sq += v * v;
    }
    float rstd = rms_rstd(sum_sq, hidden, eps);
    if (yr) {
        for (int64_t i = 0; i < hidden; ++i) {
            float t = ld_dt(dt, sr[i]) * rstd;
            float u = t * ld_dt(dt, w[i]);
            yr[i] = st_dt(dt, u);
        }
    }
}

/* ---- residual add + RMSNorm ([P2] fused add + RMSNorm, [P4] local tail) ---- */
void oracle_add_rmsnorm(int dt, const uint16_t *x, const uint16_t *r,
                        const uint16_t *w, float eps, int64_t rows,
                        int64_t hidden, uint16_t *s_out, uint16_t *y_out)
{
    for (int64_t row = 0; row < rows; ++row) {
        const uint16_t *xr = x + row * hidden;
        const uint16_t *rr = r + row * hidden;
        uint16_t *sr = s_out + row * hidden;

        /* step 1: residual' = x + residual, one fp32 add, stored in dtype.
         * Reading r[i] before writing sr[i] keeps the in-place case exact. */
        for (int64_t i = 0; i < hidden; ++i) {
            float a = ld_dt(dt, xr[i]);
            float b = ld_dt(dt, rr[i]);
            float sum = a + b;
            sr[i] = st_dt(dt, sum);
        }

        /* steps 2 and 3: rstd from the stored residual', then y */
        rmsnorm_row(dt, sr, w, eps, hidden, y_out ? y_out + row * hidden : 0);
    }
}

/* ---- gated RMSNorm ([P2] the fused gated RMSNorm + NVFP4 op) ---- */
uint16_t oracle_silu_dt(int dt, uint16_t z)
{
    double zz = dt == RQO_BF16 ? oracle_bf16_to_double(z) : oracle_fp16_to_double(z);
    double v = zz / (1.0 + exp(-zz));  /* z * sigmoid(z); -0 when e^-z overflows */
    return st_dt(dt, (float)v);        /* fp32, then the storage dtype */
}

void oracle_gated_rmsnorm(int dt, const uint16_t *x, const uint16_t *z,
                          const uint16_t *w, float eps, int64_t rows,
                          int64_t hidden, uint16_t *g_out, uint16_t *y_out)
{
    for (int64_t row = 0; row < rows; ++row) {
        const uint16_t *xr = x + row * hidden;
        const uint16_t *zr = z + row * hidden;
        uint16_t *gr = g_out + row * hidden;

        /* step 1: g = x * silu(z), one fp32 multiply, stored in dtype */
        for (int64_t i = 0; i < hidden; ++i) {
            float a = ld_dt(dt, xr[i]);
            float b = ld_dt(dt, oracle_silu_dt(dt, zr[i]));
            float prod = a * b;
            gr[i] = st_dt(dt, prod);
        }

        /* steps 2 and 3 on g */
        rmsnorm_row(dt, gr, w, eps, hidden, y_out ? y_out + row * hidden : 0);
    }
}

void oracle_gated_rmsnorm_nvfp4(int dt, const uint16_t *x, const uint16_t *z,
                                const uint16_t *w, float eps, float gs,
                                int64_t rows, int64_t hidden, uint16_t *g_out,
                                uint16_t *y_out, uint8_t *packed, uint8_t *sf)
{
    oracle_gated_rmsnorm(dt, x, z, w, eps, rows, hidden, g_out, y_out);
    oracle_quant_nvfp4(dt, y_out, rows, hidden, gs, packed, sf);
}

/* ---- per-tensor FP8 E4M3 ([P1] RMSNorm with FP8 quantisation) ---- */
void oracle_quant_fp8(int dt, const uint16_t *y, int64_t n, float scale, uint8_t *q)
{
    for (int64_t i = 0; i < n; ++i) {
        float v = ld_dt(dt, y[i]) / scale;
        q[i] = oracle_e4m3_from_double((double)v);
    }
}

/* ---- NVFP4 ([P2] NVFP4 quant ops, [P4] NVFP4 tail) ---- */
void oracle_quant_nvfp4(int dt, const uint16_t *y, int64_t rows, int64_t hidden,
                        float gs, uint8_t *packed, uint8_t *sf)
{
    const int64_t nblk = hidden / 16;
    for (int64_t row = 0; row < rows; ++row) {
        for (int64_t b = 0; b < nblk; ++b) {
            const uint16_t *yb = y + row * hidden + b * 16;
            float a = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float m = fabsf(ld_dt(dt, yb[i]));
                if (m > a) a = m;
            }
            float t1 = gs * a;
            float t2 = t1 / 6.0f;
            uint8_t sfc = oracle_e4m3_from_double((double)t2);
            float sfv = (float)oracle_e4m3_to_double(sfc);
            float enc = (sfv == 0.0f) ? 0.0f : gs / sfv;
            sf[row * nblk + b] = sfc;

            uint8_t c[16];
            for (int i = 0; i < 16; ++i) {
                float v = ld_dt(dt, yb[i]) * enc;
                c[i] = oracle_e2m1_from_double((double)v);
            }
            uint8_t *pb = packed + row * (hidden / 2) + b * 8;
            for (int j = 0; j < 8; ++j)
                pb[j] = (uint8_t)(c[2 * j] | (c[2 * j + 1] << 4));
        }
    }
}

void oracle_add_rmsnorm_fp8(int dt, const uint16_t *x, const uint16_t *r,
                            const uint16_t *w, float eps, float scale,
                            int64_t rows, int64_t hidden, uint16_t *s_out,
                            uint16_t *y_out, uint8_t *q)
{
    oracle_add_rmsnorm(dt, x, r, w, eps, rows, hidden, s_out, y_out);
    oracle_quant_fp8(dt, y_out, rows * hidden, scale, q);
}

void oracle_add_rmsnorm_nvfp4(int dt, const uint16_t *x, const uint16_t *r,
                              const uint16_t *w, float eps, float gs,
                              int64_t rows, int64_t hidden, uint16_t *s_out,
                              uint16_t *y_out, uint8_t *packed, uint8_t *sf)
{
    oracle_add_rmsnorm(dt, x, r, w, eps, rows, hidden, s_out, y_out);
    oracle_quant_nvfp4(dt, y_out, rows, hidden, gs, packed, sf);
}

int64_t oracle_nvfp4_swizzled_scale_bytes(int64_t rows, int64_t hidden)
{
    int64_t nb = hidden / 16;
    int64_t rows_pad = (rows + 127) / 128 * 128;
    int64_t cols_pad = (nb + 3) / 4 * 4;
    return rows_pad * cols_pad;
}

void oracle_nvfp4_swizzle_scales(const uint8_t *sf, int64_t rows,
                                 int64_t hidden, uint8_t *out)
{
    int64_t nb = hidden / 16;
    int64_t rows_pad = (rows + 127) / 128 * 128;
    int64_t cols_pad = (nb + 3) / 4 * 4;
    int64_t tiles_per_row = cols_pad / 4;
    for (int64_t r = 0; r < rows_pad; ++r) {
        for (int64_t c = 0; c < cols_pad; ++c) {
            uint8_t v = (r < rows && c < nb) ? sf[r * nb + c] : 0;
            int64_t tile = (r / 128) * tiles_per_row + c / 4;
            int64_t rr = r % 128, cc = c % 4;
            out[tile * 512 + 16 * (rr % 32) + 4 * (rr / 32) + cc] = v;
        }
    }
}

float oracle_amax(int dt, const uint16_t *v, int64_t n)
{
    float a = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float m = fabsf(ld_dt(dt, v[i]));
        if (m > a) a = m;
    }
    return a;
}

float oracle_fp8_scale_from_amax(float amax) { float s = amax / 448.0f; return s; }
float oracle_nvfp4_gs_from_amax(float amax) { float g = 2688.0f / amax; return g; }

/* ---- dynamic scales (the plain formulas, with 1 for a zero maximum) ---- */
float oracle_fp8_dynamic_scale(float amax)
{
    return amax > 0.0f ? oracle_fp8_scale_from_amax(amax) : 1.0f;
}

float oracle_nvfp4_dynamic_gs(float amax)
{
    return amax > 0.0f ? oracle_nvfp4_gs_from_amax(amax) : 1.0f;
}

void oracle_quant_fp8_per_row(int dt, const uint16_t *y, int64_t rows,
                              int64_t hidden, uint8_t *q, float *row_scales)
{
    for (int64_t row = 0; row < rows; ++row) {
        float scale = oracle_fp8_dynamic_scale(oracle_amax(dt, y + row * hidden, hidden));
        row_scales[row] = scale;
        oracle_quant_fp8(dt, y + row * hidden, hidden, scale, q + row * hidden);
    }
}

/* ---- Q/K RMSNorm + NeoX RoPE ([P1] fused Q/K RMSNorm and RoPE,
 *      [P3] norm + RoPE + uniform FP8 store) ---- */
void oracle_qk_rmsnorm_rope(int dt, const uint16_t *src, int64_t token_stride,
                            int64_t n_tokens, int n_heads, int head_dim,
                            const uint16_t *w, float eps, const int32_t *pos,
                            const float *cos_sin, int64_t max_pos, uint16_t *o)
{
    const int half = head_dim / 2;
    uint16_t n[1024];
    if (head_dim <= 0 || head_dim > 1024 || head_dim % 2 != 0) return;
    for (int64_t t = 0; t < n_tokens; ++t) {
        int64_t p = pos[t];
        if (p < 0) p = 0;
        if (p >= max_pos) p = max_pos - 1;
        const float *cs = cos_sin + p * head_dim;
        for (int h = 0; h < n_heads; ++h) {
            const uint16_t *xh = src + t * token_stride + (int64_t)h * head_dim;
            uint16_t *oh = o + (t * n_heads + h) * (int64_t)head_dim;

            double sum_sq = 0.0;
            for (int i = 0; i < head_dim; ++i) {
                double v = (double)ld_dt(dt, xh[i]);
                sum_sq += v * v;
            }
            float rstd = rms_rstd(sum_sq, head_dim, eps);
            for (int i = 0; i < head_dim; ++i) {
                float a = ld_dt(dt, xh[i]) * rstd;
                float b = a * ld_dt(dt, w[i]);
                n[i] = st_dt(dt, b);
            }

            /* NeoX rotation of the pairs (i, i + half) by the angle of
             * frequency i at position p */
            for (int i = 0; i < half; ++i) {
                float c = cs[i], s = cs[half + i];
                float lo = ld_dt(dt, n[i]), hi = ld_dt(dt, n[half + i]);
                float a1 = lo * c, a2 = hi * s;
                float olo = a1 - a2;
                float b1 = hi * c, b2 = lo * s;
                float ohi = b1 + b2;
                oh[i] = st_dt(dt, olo);
                oh[half + i] = st_dt(dt, ohi);
            }
        }
    }
}

void oracle_qk_rmsnorm_rope_fp8(int dt, const uint16_t *src,
                                int64_t token_stride, int64_t n_tokens,
                                int n_heads, int head_dim, const uint16_t *w,
                                float eps, const int32_t *pos,
                                const float *cos_sin, int64_t max_pos,
                                float scale, uint16_t *o, uint8_t *q)
{
    oracle_qk_rmsnorm_rope(dt, src, token_stride, n_tokens, n_heads, head_dim,
                           w, eps, pos, cos_sin, max_pos, o);
    oracle_quant_fp8(dt, o, n_tokens * (int64_t)n_heads * head_dim, scale, q);
}

/* ---- Q/K RMSNorm + NeoX RoPE over the last rope_dim elements of each head
 *      ([P3] review thread: the FlashMLA counterpart's fp8-nope + bf16-rope
 *      KV pool; the split of the head is a reading) ---- */
void oracle_qk_rmsnorm_rope_partial(int dt, const uint16_t *src,
                                    int64_t token_stride, int64_t n_tokens,
                                    int n_heads, int head_dim, int rope_dim,
                                    const uint16_t *w, float eps,
                                    const int32_t *pos, const float *cos_sin,
                                    int64_t max_pos, uint16_t *o)
{
    const int nope = head_dim - rope_dim;
    const int half = rope_dim / 2;
    uint16_t n[1024];
    if (head_dim <= 0 || head_dim > 1024 || rope_dim < 2 || rope_dim > head_dim ||
        rope_dim % 2 != 0)
        return;
    for (int64_t t = 0; t < n_tokens; ++t) {
        int64_t p = pos[t];
        if (p < 0) p = 0;
        if (p >= max_pos) p = max_pos - 1;
        const float *cs = cos_sin + p * rope_dim;   /* rope_dim/2 cos, then sin */
        for (int h = 0; h < n_heads; ++h) {
            const uint16_t *xh = src + t * token_stride + (int64_t)h * head_dim;
            uint16_t *oh = o + (t * n_heads + h) * (int64_t)head_dim;

            /* RMSNorm over the whole head, rounded to dt */
            double sum_sq = 0.0;
            for (int i = 0; i < head_dim; ++i) {
                double v = (double)ld_dt(dt, xh[i]);
                sum_sq += v * v;
            }
            float rstd = rms_rstd(sum_sq, head_dim, eps);
            for (int i = 0; i < head_dim; ++i) {
                float a = ld_dt(dt, xh[i]) * rstd;
                float b = a * ld_dt(dt, w[i]);
                n[i] = st_dt(dt, b);
            }

            /* the first `nope` elements pass unrotated */
            for (int i = 0; i < nope; ++i) oh[i] = n[i];

            /* NeoX rotation of the pairs (nope + i, nope + half + i) */
            for (int i = 0; i < half; ++i) {
                float c = cs[i], s = cs[half + i];
                float lo = ld_dt(dt, n[nope + i]), hi = ld_dt(dt, n[nope + half + i]);
                float a1 = lo * c, a2 = hi * s;
                float olo = a1 - a2;
                float b1 = hi * c, b2 = lo * s;
                float ohi = b1 + b2;
                oh[nope + i] = st_dt(dt, olo);
                oh[nope + half + i] = st_dt(dt, ohi);
            }
        }
    }
}
