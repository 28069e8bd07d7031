/*
 * rmsnorm_oracle.c -- CPU oracle for RMSNorm forward and backward (fp64).
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the CPU-baseline
 * legs of the benchmark load this library. The CUDA library never links it,
 * and it shares no code, header or table with the CUDA kernels.
 *
 * What it computes (plain definition, one row at a time, every step in
 * double; inputs are decoded exactly from their storage type):
 *
 *   forward   h_j   = x_j                      plain
 *             h_j   = R(x_j + r_j)             fused residual add (exact double
 *                                              sum, one rounding to storage type)
 *             ms    = (1/N) sum_j h_j^2
 *             rstd  = 1 / sqrt(ms + eps)
 *             y_j   = h_j * rstd * (offset + w_j)
 *
 *   backward  xhat_j = h_j * rstd
 *             g_j    = dy_j * (offset + w_j)
 *             c      = (1/N) sum_j g_j * xhat_j
 *             dx_j   = rstd * (g_j - xhat_j * c)   [+ dres_j in the fused variant]
 *             dW_j   = sum_rows dy_j * xhat_j
 *
 * Sources: "perf(cutedsl): add Blackwell fast path to RMSNorm" (Liger-Kernel
 * PR #1388, Summary and section 2: llama-mode RMSNorm, offset as a runtime
 * scalar, fused backward producing dX and dW) and "[Perf] Optimize RMSNorm
 * backward with staged reduction and vec8 I/O" (ROCm/FlyDSL PR #855,
 * Implementation: plain and fused-add backward, dx == dresidual, dweight
 * written in the parameter dtype, round-to-nearest-even bf16 stores).
 * The pages print no formula; the one above is the definition of RMSNorm
 * with weight (offset + w) and its exact gradient:
 *   d rstd / d h_k = -rstd^3 h_k / N, hence
 *   dL/dh_k = rstd g_k - (rstd^3 h_k / N) sum_j g_j h_j = rstd (g_k - xhat_k c).
 *
 * The weight w and its gradient dW may have their own storage type
 * (wdtype), e.g. fp32 master weights with bf16 activations.
 *
 * Non-affine RMSNorm (w == NULL): the weight factor (offset + w_j) is
 * replaced by 1, so y_j = h_j * rstd, g_j = dy_j, and there is no dW (the
 * Liger-Kernel page's "non-affine" case, Validation).
 *
 * R() is round-to-nearest-even to the storage type: bf16 and fp16 are
 * rounded from the double value in ONE step (no detour through binary32);
 * fp32 by the C cast. f64 "storage" (dtype 2) means no rounding at all; the pins use it
 * for finite differences.
 *
 * fp8 output (E4M3, the output type of a norm whose consumer is an fp8
 * GEMM; the TransformerEngine page's kernel key carries otype kFloat8E4M3,
 * "[ROCm] RMSNorm tuning", Description and the key round-trip check in the
 * review): the unrounded y is multiplied by a scale s and rounded once to
 * E4M3 (nearest-even, saturating to +-448). Two scalings:
 *   per tensor  s is given (delayed scaling); amax = max_ij |y_ij| is reported
 *   per row     a_i = max_j |y_ij|, s_i = 448 / a_i (1 when a_i = 0), so each
 *               row uses the full E4M3 range; 1 / s_i is reported per row
 * The pages give the output type only; the scalings are the two plain
 * readings (a given scale, or one derived from the row's own maximum).
 *
 * LayerNorm (the sibling norm the TransformerEngine tuning page registers
 * tuned configs for beside RMSNorm, "[ROCm] RMSNorm tuning", Description),
 * in the same precision rules, with the standard definition:
 *   forward   mu    = (1/N) sum_j h_j
 *             var   = (1/N) sum_j (h_j - mu)^2        (biased, two-pass)
 *             rstd  = 1 / sqrt(var + eps)
 *             xhat  = (h_j - mu) * rstd
 *             y_j   = xhat_j * (offset + gamma_j) + beta_j
 *   backward  g_j   = dy_j * (offset + gamma_j)
 *             dx_j  = rstd * (g_j - mean(g) - xhat_j * mean(g xhat)) [+ dres_j]
 *             dgamma_j = sum_rows dy_j xhat_j,  dbeta_j = sum_rows dy_j
 * gamma == NULL: factor 1 (no dgamma); beta == NULL: no bias (no dbeta).
 * The gradient follows from d mu / d h_k = 1/N and
 * d rstd / d h_k = -rstd^3 (h_k - mu) / N.
 *
 * Parity pins live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_BF16 = 1, OR_F64 = 2, OR_F16 = 3 };

/* ---------------------------------------------------------------- bf16 -- */

/* bf16 is the upper half of an IEEE binary32, so decoding is exact. */
double oracle_bf16_decode(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round a double to bf16, nearest with ties to even, in a single step.
 * bf16: 1 sign bit, 8 exponent bits (bias 127), 7 stored fraction bits.
 * Returns 0 when the result is an ordinary finite value (normal, subnormal
 * or zero), 1 when v is NaN or the rounded value overflows to infinity.
 */
int oracle_bf16_round(double v, uint16_t *out)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isnan(v)) { *out = 0x7fc0u; return 1; }
    if (isinf(v)) { *out = (uint16_t)(sign | 0x7f80u); return 1; }
    if (a == 0.0) { *out = sign; return 0; }

    const double min_normal = ldexp(1.0, -126);
    if (a < min_normal) {
        /* Subnormal range: the quantum is 2^-133. rint() rounds to nearest,
         * ties to even, in the default rounding mode. A result of 128 is
         * the smallest normal, whose encoding is also 128 (0x0080). */
        double q = rint(ldexp(a, 133));
        *out = (uint16_t)(sign | (uint16_t)q);
        return 0;
    }
    int e;
    double m = frexp(a, &e);          /* a = m * 2^e, 0.5 <= m < 1 */
    double q = rint(ldexp(m, 8));     /* 8 significant bits: 128..256 */
    if (q == 256.0) { q = 128.0; e += 1; }
    /* value = q * 2^(e-8) with 128 <= q <= 255; biased exponent of the
     * leading bit is (e - 1) + 127. */
    int be = e - 1 + 127;
    if (be >= 255) { *out = (uint16_t)(sign | 0x7f80u); return 1; }
    uint16_t frac = (uint16_t)((int)q - 128);
    *out = (uint16_t)(sign | (uint16_t)(be << 7) | frac);
    return 0;
}

/* ---------------------------------------------------------------- fp16 -- */

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_decode(uint16_t b)
{
    const int sign = (b >> 15) & 1;
    const int e = (b >> 10) & 0x1f;
    const int f = b & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                  /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);      /* (1024 + f) * 2^(e-15-10) */
    return sign ? -v : v;
}

/*
 * Round a double to binary16, nearest with ties to even, in a single step.
 * Returns 0 for an ordinary finite result (normal, subnormal or zero), 1
 * when v is NaN or the rounded value overflows to infinity.
 */
int oracle_f16_round(double v, uint16_t *out)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isnan(v)) { *out = 0x7e00u; return 1; }
    if (isinf(v)) { *out = (uint16_t)(sign | 0x7c00u); return 1; }
    if (a == 0.0) { *out = sign; return 0; }
    if (a < ldexp(1.0, -14)) {
        /* subnormal range, quantum 2^-24; 1024 is the smallest normal,
         * whose encoding is also 1024 (0x0400) */
        double q = rint(ldexp(a, 24));
        *out = (uint16_t)(sign | (uint16_t)q);
        return 0;
    }
    int e;
    double m = frexp(a, &e);          /* a = m * 2^e, 0.5 <= m < 1 */
    double q = rint(ldexp(m, 11));    /* 11 significant bits: 1024..2048 */
    if (q == 2048.0) { q = 1024.0; e += 1; }
    int be = e - 1 + 15;
    if (be >= 31) { *out = (uint16_t)(sign | 0x7c00u); return 1; }
    *out = (uint16_t)(sign | (uint16_t)(be << 10) | (uint16_t)((int)q - 1024));
    return 0;
}

/* ---------------------------------------------------------------- E4M3 -- */

/* E4M3 (the "fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 fraction
 * bits; exponent field 0 is subnormal (f * 2^-9); no infinities; S.1111.111
 * is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448. */
double oracle_e4m3_decode(uint8_t b)
{
    const int sign = (b >> 7) & 1;
    const int e = (b >> 3) & 0xf;
    const int f = b & 0x7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);
    else
        v = ldexp((double)(f + 8), e - 10);         /* (8 + f) * 2^(e-7-3) */
    return sign ? -v : v;
}

/*
 * Round a double to E4M3, nearest with ties to even, in one step; finite
 * values beyond the largest finite magnitude saturate to +-448 (no
 * infinities in this format). NaN maps to the NaN code. Returns 1 for NaN,
 * 0 otherwise.
 */
int oracle_e4m3_round(double v, uint8_t *out)
{
    uint8_t sign = signbit(v) ? 0x80u : 0u;
    double a = fabs(v);
    if (isnan(v)) { *out = (uint8_t)(sign | 0x7fu); return 1; }
    if (a >= 448.0) { *out = (uint8_t)(sign | 0x7eu); return 0; }
    if (a < ldexp(1.0, -6)) {
        /* subnormal range, quantum 2^-9; q = 8 is the smallest normal,
         * whose encoding is also 8 (0x08) */
        double q = rint(ldexp(a, 9));
        *out = (uint8_t)(sign | (uint8_t)q);
        return 0;
    }
    int e;
    double m = frexp(a, &e);          /* a = m * 2^e, 0.5 <= m < 1 */
    double q = rint(ldexp(m, 4));     /* 4 significant bits: 8..16 */
    if (q == 16.0) { q = 8.0; e += 1; }
    const int be = e - 1 + 7;
    /* a < 448 rounds to at most 448 (ties at 464 are not reachable here) */
    *out = (uint8_t)(sign | (uint8_t)(be << 3) | (uint8_t)((int)q - 8));
    return 0;
}

/* ------------------------------------------------------- storage access -- */

static double load_elem(int dtype, const void *p, int64_t i)
{
    switch (dtype) {
    case OR_BF16: return oracle_bf16_decode(((const uint16_t *)p)[i]);
    case OR_F32:  return (double)((const float *)p)[i];
    case OR_F16:  return oracle_f16_decode(((const uint16_t *)p)[i]);
    default:      return ((const double *)p)[i];
    }
}

/* Stores R(v); returns 1 if the rounding overflowed or v was not finite. */
static int store_elem(int dtype, void *p, int64_t i, double v)
{
    switch (dtype) {
    case OR_BF16: {
        uint16_t b;
        int bad = oracle_bf16_round(v, &b);
        ((uint16_t *)p)[i] = b;
        return bad;
    }
    case OR_F32: {
        float f = (float)v;
        ((float *)p)[i] = f;
        return !isfinite(f);
    }
    case OR_F16: {
        uint16_t b;
        int bad = oracle_f16_round(v, &b);
        ((uint16_t *)p)[i] = b;
        return bad;
    }
    default:
        ((double *)p)[i] = v;
        return !isfinite(v);
    }
}

/* R(v) as a double: the value a store of v would hold. */
static double round_to(int dtype, double v)
{
    switch (dtype) {
    case OR_BF16: {
        uint16_t b;
        oracle_bf16_round(v, &b);
        return oracle_bf16_decode(b);
    }
    case OR_F32: return (double)(float)v;
    case OR_F16: {
        uint16_t b;
        oracle_f16_round(v, &b);
        return oracle_f16_decode(b);
    }
    default:     return v;
    }
}

/* ------------------------------------------------------------- forward -- */

typedef struct {
    int dtype, wdtype;  /* activations / weight storage types */
    int64_t row0, row1, N;
    const void *x, *residual, *w;
    double eps, offset;
    void *y;            /* storage type, may be NULL */
    double *y64;        /* unrounded y, may be NULL */
    void *h_out;        /* storage type (fused: residual_out), may be NULL */
    double *rstd64;     /* may be NULL */
    float *rstd32;      /* may be NULL */
    /* fp8 output: mode -1 none, 0 per-tensor scale, 1 per-row scale */
    int fp8_mode;
    double fp8_scale;   /* per-tensor mode: the given scale */
    uint8_t *yq;        /* E4M3 codes, may be NULL */
    double *scaled64;   /* y * s before the E4M3 rounding, may be NULL */
    double *amax_row;   /* max_j |y_ij| per row, may be NULL */
    double *scale_inv;  /* 1 / s per row, may be NULL */
    int bad;
} fwd_job;

static void fwd_rows(fwd_job *jb)
{
    const int64_t N = jb->N;
    double *h = (double *)malloc((size_t)N * sizeof(double));
    double *yrow = (double *)malloc((size_t)N * sizeof(double));
    for (int64_t i = jb->row0; i < jb->row1; ++i) {
        const int64_t base = i * N;
        /* h: the row that is normalised */
        for (int64_t j = 0; j < N; ++j) {
            double xv = load_elem(jb->dtype, jb->x, base + j);
            if (jb->residual)
                h[j] = round_to(jb->dtype, xv + load_elem(jb->dtype, jb->residual, base + j));
            else
                h[j] = xv;
        }
        double ss = 0.0;
        for (int64_t j = 0; j < N; ++j) ss += h[j] * h[j];
        const double ms = ss / (double)N;
        const double rstd = 1.0 / sqrt(ms + jb->eps);
        double amax = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            const double factor = jb->w ? jb->offset + load_elem(jb->wdtype, jb->w, j) : 1.0;
            const double yj = h[j] * rstd * factor;
            yrow[j] = yj;
            if (fabs(yj) > amax) amax = fabs(yj);
            if (jb->y64) jb->y64[base + j] = yj;
            if (jb->y) jb->bad |= store_elem(jb->dtype, jb->y, base + j, yj);
            if (jb->h_out) jb->bad |= store_elem(jb->dtype, jb->h_out, base + j, h[j]);
        }
        if (jb->rstd64) jb->rstd64[i] = rstd;
        if (jb->rstd32) jb->rstd32[i] = (float)rstd;
        if (jb->fp8_mode >= 0) {
            double sc = jb->fp8_scale;
            if (jb->fp8_mode == 1) sc = amax > 0.0 ? 448.0 / amax : 1.0;
            for (int64_t j = 0; j < N; ++j) {
                const double v = yrow[j] * sc;
                if (jb->scaled64) jb->scaled64[base + j] = v;
                if (jb->yq) jb->bad |= oracle_e4m3_round(v, &jb->yq[base + j]);
            }
            if (jb->amax_row) jb->amax_row[i] = amax;
            if (jb->scale_inv) jb->scale_inv[i] = 1.0 / sc;
        }
    }
    free(h);
    free(yrow);
}

static void *fwd_thread(void *arg) { fwd_rows((fwd_job *)arg); return NULL; }

/* Runs the forward rows of `proto` over nthreads threads in contiguous row
 * ranges (rows are independent, so the thread count changes no result).
 * Returns the number of non-finite or overflowing stores. */
static int run_fwd(const fwd_job *proto, int64_t M, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = (int)(M > 0 ? M : 1);
    fwd_job *jobs = (fwd_job *)calloc((size_t)nthreads, sizeof(fwd_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        jobs[t].row0 = M * t / nthreads;
        jobs[t].row1 = M * (t + 1) / nthreads;
        jobs[t].bad = 0;
    }
    if (nthreads == 1) {
        fwd_rows(&jobs[0]);
    } else {
        for (int t = 0; t < nthreads; ++t) pthread_create(&tid[t], NULL, fwd_thread, &jobs[t]);
        for (int t = 0; t < nthreads; ++t) pthread_join(tid[t], NULL);
    }
    int bad = 0;
    for (int t = 0; t < nthreads; ++t) bad += jobs[t].bad;
    free(jobs); free(tid);
    return bad;
}

/*
 * Forward over an M x N row-major block. residual == NULL gives plain
 * RMSNorm; otherwise h = R(x + residual) is normalised and, if h_out is
 * given, stored there (the fused variant's residual_out).
 * Returns the number of non-finite or overflowing stores (0 expected).
 */
int oracle_rmsnorm_fwd(int dtype, int wdtype, int64_t M, int64_t N,
                       const void *x, const void *residual, const void *w,
                       double eps, double offset,
                       void *y, double *y64, void *h_out,
                       double *rstd64, float *rstd32, int nthreads)
{
    fwd_job jb;
    memset(&jb, 0, sizeof jb);
    jb.dtype = dtype; jb.wdtype = wdtype; jb.N = N;
    jb.x = x; jb.residual = residual; jb.w = w;
    jb.eps = eps; jb.offset = offset;
    jb.y = y; jb.y64 = y64; jb.h_out = h_out;
    jb.rstd64 = rstd64; jb.rstd32 = rstd32;
    jb.fp8_mode = -1;
    return run_fwd(&jb, M, nthreads);
}

/*
 * Forward with E4M3 output: yq = E4M3(y * s), s the given scale (mode 0)
 * or 448 / max_j |y_ij| per row (mode 1). y64, scaled64, amax_row,
 * scale_inv, h_out, rstd64, rstd32 may each be NULL.
 */
int oracle_rmsnorm_fwd_fp8(int dtype, int wdtype, int64_t M, int64_t N,
                           const void *x, const void *residual, const void *w,
                           double eps, double offset, int mode, double scale,
                           uint8_t *yq, double *y64, double *scaled64, double *amax_row, double *scale_inv,
                           void *h_out, double *rstd64, float *rstd32, int nthreads)
{
    if (mode != 0 && mode != 1) return -1;
    fwd_job jb;
    memset(&jb, 0, sizeof jb);
    jb.dtype = dtype; jb.wdtype = wdtype; jb.N = N;
    jb.x = x; jb.residual = residual; jb.w = w;
    jb.eps = eps; jb.offset = offset;
    jb.y64 = y64; jb.h_out = h_out;
    jb.rstd64 = rstd64; jb.rstd32 = rstd32;
    jb.fp8_mode = mode; jb.fp8_scale = scale;
    jb.yq = yq; jb.scaled64 = scaled64; jb.amax_row = amax_row; jb.scale_inv = scale_inv;
    return run_fwd(&jb, M, nthreads);
}

/* ------------------------------------------------------------ backward -- */

typedef struct {
    int dtype, wdtype;  /* activations / weight storage types */
    int64_t row0, row1, N;
    const void *dy, *h, *w, *dres;
    const float *rstd_in;
    double eps, offset;
    void *dx;
    double *dx64, *dx_scale, *dx_cscale;
    double *dw, *dw_abs;   /* this job's own partial sums, length N */
    int bad;
} bwd_job;

static void bwd_rows(bwd_job *jb)
{
    const int64_t N = jb->N;
    double *hv = (double *)malloc((size_t)N * sizeof(double));
    double *wpo = (double *)malloc((size_t)N * sizeof(double));
    for (int64_t j = 0; j < N; ++j) wpo[j] = jb->w ? jb->offset + load_elem(jb->wdtype, jb->w, j) : 1.0;
    for (int64_t i = jb->row0; i < jb->row1; ++i) {
        const int64_t base = i * N;
        for (int64_t j = 0; j < N; ++j) hv[j] = load_elem(jb->dtype, jb->h, base + j);
        double rstd;
        if (jb->rstd_in) {
            rstd = (double)jb->rstd_in[i];
        } else {
            double ss = 0.0;
            for (int64_t j = 0; j < N; ++j) ss += hv[j] * hv[j];
            rstd = 1.0 / sqrt(ss / (double)N + jb->eps);
        }
        /* c = (1/N) sum_j g_j xhat_j; cabs = (1/N) sum_j |g_j xhat_j| */
        double c = 0.0, cabs = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            const double g = load_elem(jb->dtype, jb->dy, base + j) * wpo[j];
            c += g * (hv[j] * rstd);
            cabs += fabs(g * (hv[j] * rstd));
        }
        c /= (double)N;
        cabs /= (double)N;
        for (int64_t j = 0; j < N; ++j) {
            const double dyj = load_elem(jb->dtype, jb->dy, base + j);
            const double xhat = hv[j] * rstd;
            const double g = dyj * wpo[j];
            double dxj = rstd * (g - xhat * c);
            double scale = rstd * (fabs(g) + fabs(xhat * c));
            if (jb->dres) {
                const double d = load_elem(jb->dtype, jb->dres, base + j);
                dxj += d;
                scale += fabs(d);
            }
            if (jb->dx64) jb->dx64[base + j] = dxj;
            if (jb->dx_scale) jb->dx_scale[base + j] = scale;
            if (jb->dx_cscale) jb->dx_cscale[base + j] = rstd * fabs(xhat) * cabs;
            if (jb->dx) jb->bad |= store_elem(jb->dtype, jb->dx, base + j, dxj);
            jb->dw[j] += dyj * xhat;
            jb->dw_abs[j] += fabs(dyj * xhat);
        }
    }
    free(hv);
    free(wpo);
}

static void *bwd_thread(void *arg) { bwd_rows((bwd_job *)arg); return NULL; }

/*
 * Backward over an M x N block.
 *   h        the normalised input (x for plain RMSNorm, residual_out of the
 *            fused forward)
 *   rstd_in  NULL: rstd is recomputed in double from h (the exact gradient);
 *            otherwise the given fp32 values are used.
 *   dres     NULL or the incoming residual-stream gradient (fused variant)
 * Outputs (each may be NULL except dw64):
 *   dx       R(dx) in the storage type
 *   dx64     unrounded dx
 *   dx_scale rstd (|g| + |xhat c|) [+ |dres|]: the magnitude of the terms
 *            whose difference is dx, used to bound cancellation error
 *   dx_cscale rstd |xhat| (1/N) sum_j |g_j xhat_j|: how far dx moves per
 *            unit relative error of the terms summed into c (a sum of
 *            g xhat can cancel, so its rounding error scales with the sum
 *            of magnitudes, not with |c|)
 *   dw64     sum over rows of dy * xhat (length N)
 *   dw_abs   sum over rows of |dy * xhat| (length N)
 *   dw       R(dw64) in the weight's storage type
 * Rows are split into nthreads contiguous ranges; each range keeps its own
 * dW partial and the partials are added in range order.
 * Returns the number of non-finite or overflowing stores.
 */
int oracle_rmsnorm_bwd(int dtype, int wdtype, int64_t M, int64_t N,
                       const void *dy, const void *h, const void *w,
                       const float *rstd_in, const void *dres,
                       double eps, double offset,
                       void *dx, double *dx64, double *dx_scale, double *dx_cscale,
                       double *dw64, double *dw_abs, void *dw, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = (int)(M > 0 ? M : 1);
    bwd_job *jobs = (bwd_job *)calloc((size_t)nthreads, sizeof(bwd_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t) {
        bwd_job *jb = &jobs[t];
        jb->dtype = dtype; jb->wdtype = wdtype; jb->N = N;
        jb->row0 = M * t / nthreads; jb->row1 = M * (t + 1) / nthreads;
        jb->dy = dy; jb->h = h; jb->w = w; jb->dres = dres; jb->rstd_in = rstd_in;
        jb->eps = eps; jb->offset = offset;
        jb->dx = dx; jb->dx64 = dx64; jb->dx_scale = dx_scale; jb->dx_cscale = dx_cscale;
        jb->dw = (double *)calloc((size_t)N, sizeof(double));
        jb->dw_abs = (double *)calloc((size_t)N, sizeof(double));
    }
    if (nthreads == 1) {
        bwd_rows(&jobs[0]);
    } else {
        for (int t = 0; t < nthreads; ++t) pthread_create(&tid[t], NULL, bwd_thread, &jobs[t]);
        for (int t = 0; t < nthreads; ++t) pthread_join(tid[t], NULL);
    }
    int bad = 0;
    for (int64_t j = 0; j < N; ++j) {
        double s = 0.0, sa = 0.0;
        for (int t = 0; t < nthreads; ++t) { s += jobs[t].dw[j]; sa += jobs[t].dw_abs[j]; }
        dw64[j] = s;
        if (dw_abs) dw_abs[j] = sa;
        if (dw) bad |= store_elem(wdtype, dw, j, s);
    }
    for (int t = 0; t < nthreads; ++t) {
        bad += jobs[t].bad;
        free(jobs[t].dw);
        free(jobs[t].dw_abs);
    }
    free(jobs); free(tid);
    return bad;
}

/* ----------------------------------------------------------- LayerNorm -- */

typedef struct {
    int dtype, wdtype;
    int64_t row0, row1, N;
    const void *x, *residual, *gamma, *beta;
    double eps, offset;
    void *y;
    double *y64;
    void *h_out;
    double *mean64, *rstd64;
    float *mean32, *rstd32;
    int bad;
} ln_fwd_job;

static void ln_fwd_rows(ln_fwd_job *jb)
{
    const int64_t N = jb->N;
    double *h = (double *)malloc((size_t)N * sizeof(double));
    for (int64_t i = jb->row0; i < jb->row1; ++i) {
        const int64_t base = i * N;
        for (int64_t j = 0; j < N; ++j) {
            double xv = load_elem(jb->dtype, jb->x, base + j);
            if (jb->residual)
                h[j] = round_to(jb->dtype, xv + load_elem(jb->dtype, jb->residual, base + j));
            else
                h[j] = xv;
        }
        double sum = 0.0;
        for (int64_t j = 0; j < N; ++j) sum += h[j];
        const double mu = sum / (double)N;
        double sq = 0.0;
        for (int64_t j = 0; j < N; ++j) sq += (h[j] - mu) * (h[j] - mu);
        const double var = sq / (double)N;
        const double rstd = 1.0 / sqrt(var + jb->eps);
        for (int64_t j = 0; j < N; ++j) {
            const double factor = jb->gamma ? jb->offset + load_elem(jb->wdtype, jb->gamma, j) : 1.0;
            const double bias = jb->beta ? load_elem(jb->wdtype, jb->beta, j) : 0.0;
            const double yj = (h[j] - mu) * rstd * factor + bias;
            if (jb->y64) jb->y64[base + j] = yj;
            if (jb->y) jb->bad |= store_elem(jb->dtype, jb->y, base + j, yj);
            if (jb->h_out) jb->bad |= store_elem(jb->dtype, jb->h_out, base + j, h[j]);
        }
        if (jb->mean64) jb->mean64[i] = mu;
        if (jb->mean32) jb->mean32[i] = (float)mu;
        if (jb->rstd64) jb->rstd64[i] = rstd;
        if (jb->rstd32) jb->rstd32[i] = (float)rstd;
    }
    free(h);
}

static void *ln_fwd_thread(void *arg) { ln_fwd_rows((ln_fwd_job *)arg); return NULL; }

/*
 * LayerNorm forward over an M x N block; residual, h_out, gamma, beta and
 * every output may be NULL as in oracle_rmsnorm_fwd (gamma NULL: factor 1,
 * beta NULL: no bias). mean and rstd are reported in double and rounded to
 * float32. Returns the number of non-finite or overflowing stores.
 */
int oracle_layernorm_fwd(int dtype, int wdtype, int64_t M, int64_t N,
                         const void *x, const void *residual, const void *gamma, const void *beta,
                         double eps, double offset,
                         void *y, double *y64, void *h_out,
                         double *mean64, float *mean32, double *rstd64, float *rstd32, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = (int)(M > 0 ? M : 1);
    ln_fwd_job *jobs = (ln_fwd_job *)calloc((size_t)nthreads, sizeof(ln_fwd_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t) {
        ln_fwd_job *jb = &jobs[t];
        jb->dtype = dtype; jb->wdtype = wdtype; jb->N = N;
        jb->row0 = M * t / nthreads; jb->row1 = M * (t + 1) / nthreads;
        jb->x = x; jb->residual = residual; jb->gamma = gamma; jb->beta = beta;
        jb->eps = eps; jb->offset = offset;
        jb->y = y; jb->y64 = y64; jb->h_out = h_out;
        jb->mean64 = mean64; jb->mean32 = mean32; jb->rstd64 = rstd64; jb->rstd32 = rstd32;
    }
    if (nthreads == 1) {
        ln_fwd_rows(&jobs[0]);
    } else {
        for (int t = 0; t < nthreads; ++t) pthread_create(&tid[t], NULL, ln_fwd_thread, &jobs[t]);
        for (int t = 0; t < nthreads; ++t) pthread_join(tid[t], NULL);
    }
    int bad = 0;
    for (int t = 0; t < nthreads; ++t) bad += jobs[t].bad;
    free(jobs); free(tid);
    return bad;
}

typedef struct {
    int dtype, wdtype;
    int64_t row0, row1, N;
    const void *dy, *h, *gamma, *dres;
    const float *mean_in, *rstd_in;
    double eps, offset;
    void *dx;
    double *dx64, *dx_scale, *dx_cscale;
    double *dg, *dg_abs, *db, *db_abs;   /* this job's partial sums, length N */
    int bad;
} ln_bwd_job;

static void ln_bwd_rows(ln_bwd_job *jb)
{
    const int64_t N = jb->N;
    double *hv = (double *)malloc((size_t)N * sizeof(double));
    double *gpo = (double *)malloc((size_t)N * sizeof(double));
    for (int64_t j = 0; j < N; ++j)
        gpo[j] = jb->gamma ? jb->offset + load_elem(jb->wdtype, jb->gamma, j) : 1.0;
    for (int64_t i = jb->row0; i < jb->row1; ++i) {
        const int64_t base = i * N;
        for (int64_t j = 0; j < N; ++j) hv[j] = load_elem(jb->dtype, jb->h, base + j);
        double mu, rstd;
        if (jb->rstd_in) {
            mu = (double)jb->mean_in[i];
            rstd = (double)jb->rstd_in[i];
        } else {
            double sum = 0.0;
            for (int64_t j = 0; j < N; ++j) sum += hv[j];
            mu = sum / (double)N;
            double sq = 0.0;
            for (int64_t j = 0; j < N; ++j) sq += (hv[j] - mu) * (hv[j] - mu);
            rstd = 1.0 / sqrt(sq / (double)N + jb->eps);
        }
        /* mg = mean(g), c = mean(g xhat), and their absolute counterparts */
        double mg = 0.0, c = 0.0, mgabs = 0.0, cabs = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            const double g = load_elem(jb->dtype, jb->dy, base + j) * gpo[j];
            const double xhat = (hv[j] - mu) * rstd;
            mg += g;
            c += g * xhat;
            mgabs += fabs(g);
            cabs += fabs(g * xhat);
        }
        mg /= (double)N;
        c /= (double)N;
        mgabs /= (double)N;
        cabs /= (double)N;
        for (int64_t j = 0; j < N; ++j) {
            const double dyj = load_elem(jb->dtype, jb->dy, base + j);
            const double xhat = (hv[j] - mu) * rstd;
            const double g = dyj * gpo[j];
            double dxj = rstd * (g - mg - xhat * c);
            double scale = rstd * (fabs(g) + fabs(mg) + fabs(xhat * c));
            if (jb->dres) {
                const double d = load_elem(jb->dtype, jb->dres, base + j);
                dxj += d;
                scale += fabs(d);
            }
            if (jb->dx64) jb->dx64[base + j] = dxj;
            if (jb->dx_scale) jb->dx_scale[base + j] = scale;
            if (jb->dx_cscale) jb->dx_cscale[base + j] = rstd * (mgabs + fabs(xhat) * cabs);
            if (jb->dx) jb->bad |= store_elem(jb->dtype, jb->dx, base + j, dxj);
            jb->dg[j] += dyj * xhat;
            jb->dg_abs[j] += fabs(dyj * xhat);
            jb->db[j] += dyj;
            jb->db_abs[j] += fabs(dyj);
        }
    }
    free(hv);
    free(gpo);
}

static void *ln_bwd_thread(void *arg) { ln_bwd_rows((ln_bwd_job *)arg); return NULL; }

/*
 * LayerNorm backward over an M x N block. mean_in/rstd_in: both NULL
 * (recomputed in double from h) or both the forward's fp32 values.
 * Outputs as in oracle_rmsnorm_bwd, with dx_cscale = rstd (mean|g| + |xhat|
 * mean|g xhat|) (the sensitivity of dx to the two row sums), plus dgamma
 * (dg64, dg_abs = sum |dy xhat|, dg in the weight type) and dbeta (db64,
 * db_abs = sum |dy|, db). Each output may be NULL except dg64 and db64.
 */
int oracle_layernorm_bwd(int dtype, int wdtype, int64_t M, int64_t N,
                         const void *dy, const void *h, const void *gamma,
                         const float *mean_in, const float *rstd_in, const void *dres,
                         double eps, double offset,
                         void *dx, double *dx64, double *dx_scale, double *dx_cscale,
                         double *dg64, double *dg_abs, void *dg,
                         double *db64, double *db_abs, void *db, int nthreads)
{
    if ((mean_in == NULL) != (rstd_in == NULL)) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = (int)(M > 0 ? M : 1);
    ln_bwd_job *jobs = (ln_bwd_job *)calloc((size_t)nthreads, sizeof(ln_bwd_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t) {
        ln_bwd_job *jb = &jobs[t];
        jb->dtype = dtype; jb->wdtype = wdtype; jb->N = N;
        jb->row0 = M * t / nthreads; jb->row1 = M * (t + 1) / nthreads;
        jb->dy = dy; jb->h = h; jb->gamma = gamma; jb->dres = dres;
        jb->mean_in = mean_in; jb->rstd_in = rstd_in;
        jb->eps = eps; jb->offset = offset;
        jb->dx = dx; jb->dx64 = dx64; jb->dx_scale = dx_scale; jb->dx_cscale = dx_cscale;
        jb->dg = (double *)calloc((size_t)N, sizeof(double));
        jb->dg_abs = (double *)calloc((size_t)N, sizeof(double));
        jb->db = (double *)calloc((size_t)N, sizeof(double));
        jb->db_abs = (double *)calloc((size_t)N, sizeof(double));
    }
    if (nthreads == 1) {
        ln_bwd_rows(&jobs[0]);
    } else {
        for (int t = 0; t < nthreads; ++t) pthread_create(&tid[t], NULL, ln_bwd_thread, &jobs[t]);
        for (int t = 0; t < nthreads; ++t) pthread_join(tid[t], NULL);
    }
    int bad = 0;
    for (int64_t j = 0; j < N; ++j) {
        double sg = 0.0, sga = 0.0, sb = 0.0, sba = 0.0;
        for (int t = 0; t < nthreads; ++t) {
            sg += jobs[t].dg[j]; sga += jobs[t].dg_abs[j];
            sb += jobs[t].db[j]; sba += jobs[t].db_abs[j];
        }
        dg64[j] = sg;
        db64[j] = sb;
        if (dg_abs) dg_abs[j] = sga;
        if (db_abs) db_abs[j] = sba;
        if (dg) bad |= store_elem(wdtype, dg, j, sg);
        if (db) bad |= store_elem(wdtype, db, j, sb);
    }
    for (int t = 0; t < nthreads; ++t) {
        bad += jobs[t].bad;
        free(jobs[t].dg); free(jobs[t].dg_abs); free(jobs[t].db); free(jobs[t].db_abs);
    }
    free(jobs); free(tid);
    return bad;
}

/* Round an array of doubles to bf16 (for the tests of the rounding rule). */
int oracle_bf16_round_array(const double *v, int64_t n, uint16_t *out)
{
    int bad = 0;
    for (int64_t i = 0; i < n; ++i) bad += oracle_bf16_round(v[i], &out[i]);
    return bad;
}

/* Round an array of doubles to binary16 (for the tests of the rounding rule). */
int oracle_f16_round_array(const double *v, int64_t n, uint16_t *out)
{
    int bad = 0;
    for (int64_t i = 0; i < n; ++i) bad += oracle_f16_round(v[i], &out[i]);
    return bad;
}

/* Round an array of doubles to E4M3 codes (for the tests of the rounding rule). */
int oracle_e4m3_round_array(const double *v, int64_t n, uint8_t *out)
{
    int bad = 0;
    for (int64_t i = 0; i < n; ++i) bad += oracle_e4m3_round(v[i], &out[i]);
    return bad;
}

/* Decode an array of E4M3 codes. */
void oracle_e4m3_decode_array(const uint8_t *b, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(b[i]);
}
