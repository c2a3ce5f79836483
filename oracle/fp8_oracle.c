/*
 * fp8_oracle.c — the oracle: a plain, slow, obviously-correct CPU statement of
 * what the FP8 delayed-scaling linear layer computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the timed CPU
 * baseline of the benchmark may load this library.  It shares no code, header,
 * table or constant with the CUDA path, and never imports it.
 *
 * Sources (web pages, cited by title and section):
 *   [TE-brief]  "FP8 低精度训练：Transformer Engine 简析" (m.haoling.cc) —
 *               §一 "什么是FP8" (formats and ranges), §三.1 "宏观实现框架"
 *               (per-tensor scaling, delayed scaling, the scale formula, the
 *               recipe parameters), §三.3 "FP8框架TE计算流程" (cast, amax
 *               recording, fp8_gemm), §三.4 "Tensor Core如何进行FP8训练"
 *               (high-precision GEMM output, dimensions multiple of 16).
 *   [TE-readme] "NVIDIA Transformer Engine" README (gittoolsai.com
 *               translation) — "亮点" (MXFP8 on Blackwell), "示例 PyTorch".
 *   [TE-tutor]  "NVIDIA Transformer Engine 加速训练教程" (wqu.guru) — the
 *               HYBRID recipe, history 16, "max"; LayerNormMLP; nn.GELU.
 *
 * Where the pages leave a point open the reading taken is stated beside the
 * function.  Floating point: FP8 scale arithmetic is fp32 (the precision the
 * scale is stored in); sums of products are accumulated in fp64.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -fPIC -shared (no FMA
 * contraction: every fp32 product below is rounded once, on its own).
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* FP8 formats — [TE-brief] §一: E4M3 spans [-448, 448] (weights and         */
/* activations), E5M2 a wider range (gradients).  The page prints the E5M2   */
/* bound as "57334"; the largest E5M2 value is 1.75*2^15 = 57344, which is   */
/* what this code derives from the bit layout below.                         */
/*                                                                          */
/* Layouts (the 8-bit formats the page refers to, arXiv:2209.05433):        */
/*   E4M3: sign | 4 exponent bits, bias 7 | 3 mantissa bits.  No infinity;  */
/*         S.1111.111 is NaN, so S.1111.110 = 1.75 * 2^8 = 448 is the max.  */
/*   E5M2: sign | 5 exponent bits, bias 15 | 2 mantissa bits, IEEE-like:     */
/*         S.11111.00 = infinity, S.11111.{01,10,11} = NaN.                  */
/* ------------------------------------------------------------------------ */
enum { ORC_E4M3 = 0, ORC_E5M2 = 1 };

double orc_fp8_decode(int fmt, uint8_t code)
{
    const int mbits = (fmt == ORC_E4M3) ? 3 : 2;
    const int ebits = (fmt == ORC_E4M3) ? 4 : 5;
    const int bias = (fmt == ORC_E4M3) ? 7 : 15;
    const int sign = code >> 7;
    const int e = (code >> mbits) & ((1 << ebits) - 1);
    const int m = code & ((1 << mbits) - 1);
    double mag;
    if (fmt == ORC_E4M3 && e == 15 && m == 7)
        return NAN;
    if (fmt == ORC_E5M2 && e == 31) {
        if (m != 0)
            return NAN;
        return sign ? -INFINITY : INFINITY;
    }
    if (e == 0) /* subnormal: 0.m * 2^(1-bias) */
        mag = ldexp((double)m / (double)(1 << mbits), 1 - bias);
    else        /* normal: 1.m * 2^(e-bias) */
        mag = ldexp(1.0 + (double)m / (double)(1 << mbits), e - bias);
    return sign ? -mag : mag;
}

/* Largest finite magnitude code of each format. */
static uint8_t orc_max_code(int fmt) { return fmt == ORC_E4M3 ? 0x7E : 0x7B; }

double orc_fp8_max(int fmt) { return orc_fp8_decode(fmt, orc_max_code(fmt)); }

/* Decoded value of every code, filled once when the library is loaded. */
static double orc_table[2][256];

__attribute__((constructor)) static void orc_fill_tables(void)
{
    int f, c;
    for (f = 0; f < 2; f++)
        for (c = 0; c < 256; c++)
            orc_table[f][c] = orc_fp8_decode(f, (uint8_t)c);
}

/*
 * Encode one fp32 value.  Reading (the pages give only the ranges):
 * round to the nearest representable value, ties to the code with an even
 * mantissa (even code), and saturate: every finite value at or beyond the
 * largest finite magnitude, and +-infinity, maps to +-max.  NaN maps to a NaN
 * code (0x7F with the input's sign bit).  Values that round below the
 * smallest subnormal go to a signed zero.
 *
 * The nearest code is found by comparing |v| against the decoded magnitudes
 * of all non-negative finite codes, which are increasing in the code.  The
 * distances are exact in double (|v| has 24 significant bits, the codes 4).
 */
uint8_t orc_fp8_encode(int fmt, float v)
{
    const double *tab = orc_table[fmt == ORC_E4M3 ? 0 : 1];
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    const uint8_t top = orc_max_code(fmt);
    double a = fabs((double)v);
    uint8_t lo = 0, hi = top, mid;
    double dlo, dhi;
    if (isnan(v))
        return (uint8_t)(sign | 0x7F);
    if (a >= tab[top])
        return (uint8_t)(sign | top);
    /* binary search: tab[lo] <= a < tab[hi] */
    while (hi - lo > 1) {
        mid = (uint8_t)((lo + hi) / 2);
        if (tab[mid] <= a)
            lo = mid;
        else
            hi = mid;
    }
    dlo = a - tab[lo];
    dhi = tab[hi] - a;
    if (dlo < dhi)
        return (uint8_t)(sign | lo);
    if (dhi < dlo)
        return (uint8_t)(sign | hi);
    return (uint8_t)(sign | ((lo & 1) ? hi : lo)); /* tie: even code */
}

/* ------------------------------------------------------------------------ */
/* Inputs: fp32 (kind 0) or bf16 (kind 1, the upper 16 bits of an fp32).     */
/* ------------------------------------------------------------------------ */
static float orc_load(const void *x, int kind, int64_t i)
{
    if (kind == 0)
        return ((const float *)x)[i];
    {
        uint32_t bits = (uint32_t)((const uint16_t *)x)[i] << 16;
        float f;
        memcpy(&f, &bits, 4);
        return f;
    }
}

/*
 * Per-tensor quantisation — [TE-brief] §三.1: symmetric linear quantisation,
 * only a scale, no zero point; §三.3: input/weight are cast to FP8 with the
 * scale held in fp8_meta.  Reading: the product x*scale is rounded to fp32
 * (round to nearest even) and then encoded: q = enc(fl32(x * scale)).
 * Writes q[i] for i in [0, n).
 */
void orc_quantize(int fmt, const void *x, int kind, int64_t n, float scale, uint8_t *q)
{
    int64_t i;
    for (i = 0; i < n; i++) {
        float p = orc_load(x, kind, i) * scale;
        q[i] = orc_fp8_encode(fmt, p);
    }
}

/*
 * amax — [TE-brief] §三.1/§三.3: the cast records the tensor's absolute
 * maximum into the amax history.  Reading: the maximum of |x| over the
 * high-precision, pre-scale values (NaN is skipped), as fp32.
 */
float orc_amax(const void *x, int kind, int64_t n)
{
    float m = 0.0f;
    int64_t i;
    for (i = 0; i < n; i++) {
        float a = fabsf(orc_load(x, kind, i));
        if (a > m)
            m = a;
    }
    return m;
}

/* Column sums of a [rows x cols] row-major tensor in fp64 (the bias gradient
 * of a linear layer is the sum of grad_output over the token rows). */
void orc_colsum(const void *x, int kind, int64_t rows, int64_t cols, double *sum, double *abs_sum)
{
    int64_t r, c;
    for (c = 0; c < cols; c++) {
        sum[c] = 0.0;
        abs_sum[c] = 0.0;
    }
    for (r = 0; r < rows; r++)
        for (c = 0; c < cols; c++) {
            double v = (double)orc_load(x, kind, r * cols + c);
            sum[c] += v;
            abs_sum[c] += fabs(v);
        }
}

/* ------------------------------------------------------------------------ */
/* Delayed scaling — [TE-brief] §三.1:                                       */
/*   FP8_MAX = largest value of the format                                  */
/*   new_scale = (FP8_MAX / amax) / 2^margin                                */
/* where amax is the maximum of the amax history over its window (the      */
/* "max" algorithm, [TE-tutor]); `interval` = update the scale every that   */
/* many steps.  Readings:                                                    */
/*   - every call pushes the step's recorded amax into a ring of length L   */
/*     and clears it; the scale is recomputed when step % interval == 0;    */
/*   - arithmetic in fp32, divide first then divide by 2^margin (as the     */
/*     formula is written); scale_inv = fl32(1 / scale);                    */
/*   - a window max that is zero or not finite, or a new scale that is not  */
/*     finite and positive, keeps the previous scale and scale_inv.         */
/* ------------------------------------------------------------------------ */
static void orc_recompute(int fmt, int margin, int hist_len, const float *hist,
                          float *scale, float *scale_inv)
{
    float a = 0.0f, s, p;
    int i;
    for (i = 0; i < hist_len; i++)
        if (hist[i] > a)
            a = hist[i];
    if (!(a > 0.0f) || isinf(a))
        return;
    s = (float)orc_fp8_max(fmt) / a;
    p = ldexpf(1.0f, margin); /* 2^margin, exact */
    s = s / p;
    if (!(s > 0.0f) || isinf(s))
        return;
    *scale = s;
    *scale_inv = 1.0f / s;
}

void orc_update_scale(int fmt, int margin, int interval, int hist_len, int64_t step,
                      float *hist, int32_t *pos, float *amax_cur, float *scale, float *scale_inv)
{
    hist[*pos] = *amax_cur;
    *pos = (*pos + 1) % hist_len;
    *amax_cur = 0.0f;
    if (step % interval != 0)
        return;
    orc_recompute(fmt, margin, hist_len, hist, scale, scale_inv);
}

/* First step: the history is filled with the first step's own amax (an
 * amax-only pass), then the scale is derived from it before any cast. */
void orc_seed_history(int fmt, int margin, int hist_len, float *hist, int32_t *pos,
                      float *amax_cur, float *scale, float *scale_inv)
{
    int i;
    for (i = 0; i < hist_len; i++)
        hist[i] = *amax_cur;
    *pos = 0;
    *amax_cur = 0.0f;
    orc_recompute(fmt, margin, hist_len, hist, scale, scale_inv);
}

/* ------------------------------------------------------------------------ */
/* FP8 GEMM — [TE-brief] §三.3/§三.4: fp8_gemm multiplies two FP8 matrices   */
/* on the tensor cores and returns a high-precision (FP16/FP32) result; the  */
/* stored scale_inv of each operand dequantises it.                          */
/* Convention (all GEMMs of the layer): D[M,N] = A[M,K] * B[N,K]^T, both     */
/* operands row-major with K contiguous.                                    */
/* Reading: ref = (sum_k dec(a)*dec(b), in fp64) * fl32(sa_inv*sb_inv)       */
/*          + bias[n];   the tolerance term abs = sum_k |dec(a)*dec(b)| * s. */
/* Computed for a list of (m, n) output elements.                            */
/* ------------------------------------------------------------------------ */
void orc_gemm_elems(const uint8_t *A, int afmt, const uint8_t *B, int bfmt,
                    int64_t M, int64_t N, int64_t K, float sa_inv, float sb_inv,
                    const void *bias, int bias_kind, int64_t n_elems,
                    const int64_t *ms, const int64_t *ns, double *ref, double *abs_ref)
{
    double ta[256], tb[256];
    float s = sa_inv * sb_inv;
    int64_t e, k;
    int c;
    (void)M;
    (void)N;
    for (c = 0; c < 256; c++) {
        ta[c] = orc_fp8_decode(afmt, (uint8_t)c);
        tb[c] = orc_fp8_decode(bfmt, (uint8_t)c);
    }
    for (e = 0; e < n_elems; e++) {
        const uint8_t *arow = A + ms[e] * K;
        const uint8_t *brow = B + ns[e] * K;
        double acc = 0.0, aacc = 0.0;
        for (k = 0; k < K; k++) {
            double p = ta[arow[k]] * tb[brow[k]];
            acc += p;
            aacc += fabs(p);
        }
        ref[e] = acc * (double)s + (bias ? (double)orc_load(bias, bias_kind, ns[e]) : 0.0);
        abs_ref[e] = aacc * (double)s;
    }
}

/* ------------------------------------------------------------------------ */
/* MXFP8 — named, not defined, by [TE-readme] "亮点" (MXFP8 on Blackwell).   */
/* Reading: blocks of 32 consecutive elements along the reduction axis, one */
/* E8M0 scale per block (a biased power of two, code = e + 127), E4M3 data. */
/* The block exponent is the power-of-two restriction of the per-tensor     */
/* scale FP8_MAX/amax: the smallest integer e with amax_b * 2^-e <= 448, so */
/* the block maximum never saturates.  Writing amax_b = f * 2^E, f in [1,2): */
/* e = E - 8 when f <= 1.75, else E - 7; clamped to [-127, 127]; amax_b = 0 */
/* gives e = 0.  Data: q = enc_e4m3(fl32(x * 2^-e)).                          */
/* ------------------------------------------------------------------------ */
int orc_e8m0_exponent(float amax_b)
{
    int E, e;
    float f;
    if (amax_b == 0.0f)
        return 0;
    f = frexpf(amax_b, &E); /* amax_b = f * 2^E, f in [0.5, 1) */
    f *= 2.0f;              /* exact: now f in [1, 2), amax_b = f * 2^(E-1) */
    E -= 1;
    e = (f <= 1.75f) ? E - 8 : E - 7;
    if (e < -127)
        e = -127;
    if (e > 127)
        e = 127;
    return e;
}

/* Row-wise MX quantisation of a bf16/fp32 [rows x cols] matrix, cols % 32 == 0:
 * q [rows x cols] E4M3 codes, s [rows x cols/32] E8M0 codes. */
void orc_mx_quantize_rows(const void *x, int kind, int64_t rows, int64_t cols, uint8_t *q, uint8_t *s)
{
    int64_t r, b, j;
    for (r = 0; r < rows; r++)
        for (b = 0; b < cols / 32; b++) {
            float amax_b = 0.0f, mult;
            int e;
            for (j = 0; j < 32; j++) {
                float a = fabsf(orc_load(x, kind, r * cols + b * 32 + j));
                if (a > amax_b)
                    amax_b = a;
            }
            e = orc_e8m0_exponent(amax_b);
            mult = ldexpf(1.0f, -e); /* exact power of two, possibly subnormal */
            s[r * (cols / 32) + b] = (uint8_t)(e + 127);
            for (j = 0; j < 32; j++)
                q[r * cols + b * 32 + j] = orc_fp8_encode(ORC_E4M3, orc_load(x, kind, r * cols + b * 32 + j) * mult);
        }
}

/* MX GEMM, D[M,N] = A[M,K] * B[N,K]^T with E4M3 data and one E8M0 scale per
 * 32 consecutive K of each row: ref = sum_b 2^(ea+eb) * sum_{k in b} a*b
 * (fp64) + bias[n]; abs_ref the same with |a*b|. */
void orc_mx_gemm_elems(const uint8_t *A, const uint8_t *As, const uint8_t *B, const uint8_t *Bs,
                       int64_t M, int64_t N, int64_t K, const void *bias, int bias_kind,
                       int64_t n_elems, const int64_t *ms, const int64_t *ns, double *ref, double *abs_ref)
{
    double t[256];
    int64_t e, b, k;
    int c;
    (void)M;
    (void)N;
    for (c = 0; c < 256; c++)
        t[c] = orc_fp8_decode(ORC_E4M3, (uint8_t)c);
    for (e = 0; e < n_elems; e++) {
        const uint8_t *arow = A + ms[e] * K, *brow = B + ns[e] * K;
        const uint8_t *asr = As + ms[e] * (K / 32), *bsr = Bs + ns[e] * (K / 32);
        double acc = 0.0, aacc = 0.0;
        for (b = 0; b < K / 32; b++) {
            double blk = 0.0, ablk = 0.0;
            double sc = ldexp(1.0, (int)asr[b] - 127 + (int)bsr[b] - 127);
            for (k = b * 32; k < b * 32 + 32; k++) {
                double p = t[arow[k]] * t[brow[k]];
                blk += p;
                ablk += fabs(p);
            }
            acc += sc * blk;
            aacc += sc * ablk;
        }
        ref[e] = acc + (bias ? (double)orc_load(bias, bias_kind, ns[e]) : 0.0);
        abs_ref[e] = aacc;
    }
}

/* ------------------------------------------------------------------------ */
/* LayerNormMLP pieces — [TE-tutor]: te.LayerNormMLP (LayerNorm, fc1, GELU,   */
/* fc2), whose plain-PyTorch mirror uses nn.LayerNorm and nn.GELU (the erf  */
/* form).  Textbook definitions in fp64; the pages fix no precision or eps  */
/* beyond the workload's eps = 1e-5 and the biased variance of LayerNorm.   */
/* Parameters gamma/beta use the same kinds as the inputs (fp32 or bf16).   */
/* ------------------------------------------------------------------------ */
/* y = (x - mu) / sqrt(var + eps) * gamma + beta per row, var biased;
 * also mu and rsigma = 1/sqrt(var + eps) per row. */
void orc_layernorm_fwd(const void *x, int kind, int64_t rows, int64_t cols, const void *gamma, const void *beta,
                       int pkind, double eps, double *y, double *mu, double *rsigma)
{
    int64_t r, c;
    for (r = 0; r < rows; r++) {
        double m = 0.0, v = 0.0, rs;
        for (c = 0; c < cols; c++)
            m += (double)orc_load(x, kind, r * cols + c);
        m /= (double)cols;
        for (c = 0; c < cols; c++) {
            double d = (double)orc_load(x, kind, r * cols + c) - m;
            v += d * d;
        }
        v /= (double)cols;
        rs = 1.0 / sqrt(v + eps);
        mu[r] = m;
        rsigma[r] = rs;
        for (c = 0; c < cols; c++)
            y[r * cols + c] = ((double)orc_load(x, kind, r * cols + c) - m) * rs * (double)orc_load(gamma, pkind, c) +
                              (double)orc_load(beta, pkind, c);
    }
}

/* GELU, erf form: g = 0.5 * h * (1 + erf(h / sqrt(2))). */
void orc_gelu(const void *h, int kind, int64_t n, double *g)
{
    int64_t i;
    for (i = 0; i < n; i++) {
        double v = (double)orc_load(h, kind, i);
        g[i] = 0.5 * v * (1.0 + erf(v / sqrt(2.0)));
    }
}

/* Backward of GELU: dh = dg * (0.5 * (1 + erf(h/sqrt2)) + h * exp(-h^2/2) / sqrt(2 pi)). */
void orc_dgelu(const void *dg, const void *h, int kind, int64_t n, double *dh)
{
    const double inv_sqrt_2pi = 0.3989422804014327;
    int64_t i;
    for (i = 0; i < n; i++) {
        double v = (double)orc_load(h, kind, i);
        double d = 0.5 * (1.0 + erf(v / sqrt(2.0))) + v * exp(-0.5 * v * v) * inv_sqrt_2pi;
        dh[i] = (double)orc_load(dg, kind, i) * d;
    }
}

/* Backward of LayerNorm given the forward's per-row mu and rsigma:
 *   xhat = (x - mu) * rsigma, g = dy * gamma
 *   dx = rsigma * (g - mean(g) - xhat * mean(g * xhat))
 *   dgamma = sum_rows dy * xhat,  dbeta = sum_rows dy
 * The *_abs outputs are the same expressions over absolute values (for error
 * bounds of an fp32 implementation). */
void orc_layernorm_bwd(const void *dy, const void *x, int kind, int64_t rows, int64_t cols, const void *gamma,
                       int pkind, const double *mu, const double *rsigma, double *dx, double *dgamma, double *dbeta,
                       double *dx_abs, double *dgamma_abs, double *dbeta_abs)
{
    int64_t r, c;
    for (c = 0; c < cols; c++) {
        dgamma[c] = dbeta[c] = dgamma_abs[c] = dbeta_abs[c] = 0.0;
    }
    for (r = 0; r < rows; r++) {
        double s1 = 0.0, s2 = 0.0, a1 = 0.0, a2 = 0.0;
        for (c = 0; c < cols; c++) {
            double d = (double)orc_load(dy, kind, r * cols + c);
            double xh = ((double)orc_load(x, kind, r * cols + c) - mu[r]) * rsigma[r];
            double g = d * (double)orc_load(gamma, pkind, c);
            s1 += g;
            s2 += g * xh;
            a1 += fabs(g);
            a2 += fabs(g * xh);
            dgamma[c] += d * xh;
            dbeta[c] += d;
            dgamma_abs[c] += fabs(d * xh);
            dbeta_abs[c] += fabs(d);
        }
        s1 /= (double)cols;
        s2 /= (double)cols;
        a1 /= (double)cols;
        a2 /= (double)cols;
        for (c = 0; c < cols; c++) {
            double d = (double)orc_load(dy, kind, r * cols + c);
            double xh = ((double)orc_load(x, kind, r * cols + c) - mu[r]) * rsigma[r];
            double g = d * (double)orc_load(gamma, pkind, c);
            dx[r * cols + c] = rsigma[r] * (g - s1 - xh * s2);
            dx_abs[r * cols + c] = rsigma[r] * (fabs(g) + a1 + fabs(xh) * a2);
        }
    }
}
