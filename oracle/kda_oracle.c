/*
 * kda_oracle.c -- plain CPU oracle for the KDA decode projections.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file; only the tests, the package's smoke check and the benchmark's CPU
 * baseline do. It shares no code, header or constant with the CUDA library.
 *
 * What it computes is the plain definition of the method, with no blocking,
 * fusion or reordering:
 *
 *   y[m, n] = sum_{k = 0 .. K-1} x[m, k] * W[n, k]           (C = A * B^T)
 *
 * on the bf16 inputs widened exactly to double, summed in ascending k, one
 * output at a time. This is the skinny GEMM of the Kimi K3 support page, part 1
 * (vllm PR #50089 digest, section "关键源码片段", CuteSkinnyGemm docstring: C[M,N] =
 * A[M,K] @ B[N,K].T with fp32 accumulation, bf16/fp16 inputs). The oracle uses
 * double instead of fp32 so that its own rounding error is far below the
 * comparison tolerance; the result is left in double.
 *
 * The full KDA projection ("[Kimi-K3] Overlap low-M TP8 KDA projections",
 * section "关键源码片段", run_kda_projection_overlap / run_qkvg / run_fab_fb and
 * KimiK3DeltaAttention.forward's sequential branch) is, in that page's order:
 *
 *   qkvg = x * W_packed[0 : N_qkvg]^T
 *   fab  = x * W_packed[N_qkvg : N_qkvg + N_fab]^T
 *   f_a  = bf16(fab[:, 0 : 128])      (the F_A half of the split, as bf16)
 *   fb   = f_a * W_fb^T
 *
 * f_a is rounded to bf16 (round-to-nearest-even) before F_B because the page
 * feeds the bf16 F_A output tensor into the F_B GEMM; no activation sits
 * between them.
 *
 * bf16 conversions are written from the IEEE-754 binary16-brain-float
 * definition: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits;
 * subnormals down to 2^-133; round to nearest, ties to even.
 *
 * The same page's kernel also takes fp16 inputs and an optional residual:
 * C = A * B^T + residual, the residual (same element type, [M, N]) added to
 * the fp32 accumulator after the K loop, before the single conversion to the
 * output type. kdo_gemm_ex computes that in double: the K-sum as above, then
 * one addition of the widened residual. fp16 is widened from the IEEE-754
 * binary16 layout: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits,
 * subnormals (exponent field 0) = fraction x 2^-24.
 *
 * Build: gcc -O2 -fPIC -shared -pthread -ffp-contract=off (no fused
 * multiply-add contraction, no fast-math), so each product and each sum is a
 * separately rounded IEEE double operation on every host.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 bits -> double: the 16 bits are the top half of an IEEE binary32. */
double kdo_bf16_to_f64(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* fp16 bits -> double: (1024 + fraction) x 2^(exponent - 25) for a normal
 * number, fraction x 2^-24 for a subnormal one (exponent field 0); exponent
 * field 31 is infinity (fraction 0) or NaN. */
double kdo_fp16_to_f64(uint16_t h)
{
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25);
    return (h & 0x8000) ? -v : v;
}

/* element widening for the two 16-bit input types: 0 = bf16, 1 = fp16 */
static double widen(uint16_t b, int dtype)
{
    return dtype ? kdo_fp16_to_f64(b) : kdo_bf16_to_f64(b);
}

/* double -> bf16 bits, round to nearest, ties to even, with subnormals and
 * overflow to infinity. The value is scaled by the bf16 quantum at its
 * exponent, rounded to an integer with rint() (ties-to-even in the default
 * rounding mode) and scaled back; the result is then exactly representable in
 * bf16 and in binary32, whose top 16 bits are the answer. */
uint16_t kdo_f64_to_bf16_rne(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0x0000;
    double a = fabs(v);
    if (isinf(a))
        return sign | 0x7F80;
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e);          /* a = f * 2^e, f in [0.5, 1) */
    int E = e - 1;               /* a = (2f) * 2^E, 2f in [1, 2) */
    int qexp = (E < -126) ? -133 : (E - 7);
    double r = rint(ldexp(a, -qexp));
    double q = ldexp(r, qexp);
    /* largest finite bf16 is (2 - 2^-7) * 2^127; anything that rounds past it
     * is infinity */
    if (q >= ldexp(1.0, 128))
        return sign | 0x7F80;
    float f = (float)q;          /* exact: q has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

void kdo_round_bf16(const double *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kdo_f64_to_bf16_rne(in[i]);
}

void kdo_widen_bf16(const uint16_t *in, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kdo_bf16_to_f64(in[i]);
}

void kdo_widen_fp16(const uint16_t *in, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kdo_fp16_to_f64(in[i]);
}

/* ---- y = x * W^T, one output at a time, k ascending --------------------- */

typedef struct {
    const uint16_t *x;
    int64_t ldx;
    const uint16_t *W;
    int64_t ldw;
    const uint16_t *res;   /* NULL: no residual */
    int64_t ldr;
    int dtype;             /* 0 = bf16, 1 = fp16 (x, W and the residual) */
    double *y;
    int64_t ldy;
    int M, N, K;
    int n_begin, n_end;
} gemm_job;

static void gemm_columns(const gemm_job *j)
{
    for (int m = 0; m < j->M; ++m) {
        const uint16_t *xr = j->x + (int64_t)m * j->ldx;
        for (int n = j->n_begin; n < j->n_end; ++n) {
            const uint16_t *wr = j->W + (int64_t)n * j->ldw;
            double acc = 0.0;
            for (int k = 0; k < j->K; ++k) {
                double p = widen(xr[k], j->dtype) * widen(wr[k], j->dtype);
                acc = acc + p;
            }
            if (j->res)
                acc = acc + widen(j->res[(int64_t)m * j->ldr + n], j->dtype);
            j->y[(int64_t)m * j->ldy + n] = acc;
        }
    }
}

static void *gemm_thread(void *arg)
{
    gemm_columns((const gemm_job *)arg);
    return NULL;
}

/* x: [M, K] with row stride ldx elements; W: [N, K] with row stride ldw;
 * res: NULL or [M, N] with row stride ldr; all three of type dtype (0 = bf16,
 * 1 = fp16). y: [M, N] doubles with row stride ldy. nthreads > 1 splits the N
 * columns into contiguous ranges, one per thread; every output is still
 * computed by one thread with the same loop, so the result does not depend on
 * nthreads. Returns 0, or -1 on a bad argument. */
int kdo_gemm_ex(const uint16_t *x, int64_t ldx, const uint16_t *W, int64_t ldw,
                const uint16_t *res, int64_t ldr, int dtype,
                double *y, int64_t ldy, int M, int N, int K, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || ldx < K || ldw < K || ldy < N || (res && ldr < N) ||
        (dtype != 0 && dtype != 1))
        return -1;
    if (M == 0 || N == 0)
        return 0;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > N)
        nthreads = N;
    gemm_job *jobs = (gemm_job *)calloc((size_t)nthreads, sizeof(gemm_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -1;
    }
    for (int t = 0; t < nthreads; ++t) {
        gemm_job *j = &jobs[t];
        j->x = x; j->ldx = ldx; j->W = W; j->ldw = ldw;
        j->res = res; j->ldr = ldr; j->dtype = dtype;
        j->y = y; j->ldy = ldy; j->M = M; j->N = N; j->K = K;
        j->n_begin = (int)(((int64_t)N * t) / nthreads);
        j->n_end = (int)(((int64_t)N * (t + 1)) / nthreads);
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, gemm_thread, &jobs[t]) != 0)
            break;
        started = t;
    }
    gemm_columns(&jobs[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(th[t], NULL);
    /* ranges whose thread could not be started run here */
    for (int t = started + 1; t < nthreads; ++t)
        gemm_columns(&jobs[t]);
    free(jobs);
    free(th);
    return 0;
}

/* bf16 inputs, no residual (the projections' GEMM). */
int kdo_gemm(const uint16_t *x, int64_t ldx, const uint16_t *W, int64_t ldw,
             double *y, int64_t ldy, int M, int N, int K, int nthreads)
{
    return kdo_gemm_ex(x, ldx, W, ldw, NULL, 0, 0, y, ldy, M, N, K, nthreads);
}

/* The full projection, in the page's order (see the header comment).
 *   x        [M, K]                  bf16 bits, row-major
 *   Wp       [N_qkvg + N_fab, K]     bf16 bits, row-major (Q/K/V/G rows first)
 *   Wfb      [N_fb, N_fa]            bf16 bits, row-major
 *   qkvg     [M, N_qkvg]             double out
 *   fab      [M, N_fab]              double out
 *   fa_bf16  [M, N_fa]               bf16 bits out (rounded F_A, F_B's input)
 *   fb       [M, N_fb]               double out
 * N_fa is the width of the F_A half (128 on the pages). */
int kdo_kda_proj(const uint16_t *x, const uint16_t *Wp, const uint16_t *Wfb,
                 double *qkvg, double *fab, uint16_t *fa_bf16, double *fb,
                 int M, int K, int N_qkvg, int N_fab, int N_fa, int N_fb,
                 int nthreads)
{
    if (N_fa > N_fab || N_fa < 0)
        return -1;
    int rc = kdo_gemm(x, K, Wp, K, qkvg, N_qkvg, M, N_qkvg, K, nthreads);
    if (rc)
        return rc;
    rc = kdo_gemm(x, K, Wp + (int64_t)N_qkvg * K, K, fab, N_fab, M, N_fab, K, nthreads);
    if (rc)
        return rc;
    for (int m = 0; m < M; ++m)
        for (int j = 0; j < N_fa; ++j)
            fa_bf16[(int64_t)m * N_fa + j] = kdo_f64_to_bf16_rne(fab[(int64_t)m * N_fab + j]);
    return kdo_gemm(fa_bf16, N_fa, Wfb, N_fa, fb, N_fb, M, N_fb, N_fa, nthreads);
}
