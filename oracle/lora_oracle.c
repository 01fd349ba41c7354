/*
 * lora_oracle.c -- plain, slow CPU oracle for the batch-invariant shared LoRA
 * delta operator.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call this file;
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load it. It shares no source, header, table or helper with the CUDA library.
 *
 * What it computes (page "[DSv4][P5-3] shared_grouped_lora_delta: CUDA +
 * Triton, both batch-invariant", section "Summary"):
 *
 *   forward   U  = X @ A^T        FP32 accumulate, round to BF16
 *             dY_lora = (U @ B^T) * alpha   FP32 accumulate, FP32 output
 *   backward  dV = dY * alpha     (rounded to BF16, "D4")
 *             dU = dV @ B         (rounded to BF16, "D4")
 *             dB = dV^T @ U,  dX = dU @ A,  dA = dU^T @ X   (FP32)
 *   No base-weight gradient.
 *
 * Layouts (row-major, contiguous): x[M][K], a[R][K], b[N][R], u[M][R],
 * dy[M][N], dv[M][N], du[M][R], delta_y[M][N], dx[M][K], da[R][K], db[N][R].
 *
 * Arithmetic. Every BF16 x BF16 product has at most 16 significant bits, so it
 * is exact in binary64 (and in binary32: same page, section "Agreement with
 * the oracle"). Each output element is the binary64 sum of its exact products
 * taken in ascending index order, then rounded once to binary32 (rn32) -- the
 * "FP32 accumulate" result up to the summation order, which the page leaves
 * to the implementation. Where the page says "round to BF16", the binary32
 * value is then rounded to bfloat16 (rnbf). Both roundings are IEEE-754
 * round-to-nearest-even. Alongside each output the oracle can return
 * S = sum of |products| (times |alpha| where alpha scales the result), the
 * scale of the parity tolerance.
 *
 * Threads split output rows only; every element is one fixed-order sum, so
 * the thread count never changes a bit.
 *
 * Build: cc -O2 -ffp-contract=off -fPIC -shared (no fast-math).
 * Compiling with -DORACLE_MUTANT=n plants mistake n (tests only; see the
 * MUTANT blocks) so the test suite can show that its pins catch it.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ---------------------------------------------------------------- rounding */

/* binary64 -> binary32, round to nearest even: the C conversion under the
 * default rounding mode is exactly that. */
static float rn32(double v) { return (float)v; }

/* binary32 -> bfloat16 (1 sign, 8 exponent, 7 fraction bits: the upper half
 * of a binary32), round to nearest even written out from its definition:
 * keep the upper 16 bits, round up when the dropped 16 bits exceed half an
 * ulp, or equal half an ulp and the kept part is odd. A carry out of the
 * fraction bumps the exponent, which is the correct result (and gives
 * infinity past the largest finite value). NaN stays NaN (quiet bit set). */
static uint16_t rnbf(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    if ((bits & 0x7f800000u) == 0x7f800000u && (bits & 0x007fffffu) != 0u)
        return (uint16_t)((bits >> 16) | 0x0040u);
    uint32_t kept = bits >> 16;
    uint32_t dropped = bits & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

/* bfloat16 bits -> exact binary64 value */
static double bf2d(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------- the one primitive */

/*
 * out[i][j] = sum over t = 0..T-1, ascending, of P(i,t) * Q(j,t), in binary64,
 * where P(i,t) = p[i*p_i + t*p_t] and Q(j,t) = q[j*q_j + t*q_t] are bfloat16.
 * absout[i][j] (optional) = sum of |P(i,t) * Q(j,t)|.
 */
typedef struct {
    const uint16_t *p; int64_t p_i, p_t;
    const uint16_t *q; int64_t q_j, q_t;
    int64_t I, J, T;
    double *out, *absout;
    int64_t i0, i1;
} dot_job;

static void dot_rows(const dot_job *d)
{
    for (int64_t i = d->i0; i < d->i1; ++i) {
        for (int64_t j = 0; j < d->J; ++j) {
            double s = 0.0, sa = 0.0;
            int64_t T = d->T;
#if ORACLE_MUTANT == 1   /* planted: drops the last term of every sum */
            T = T > 0 ? T - 1 : 0;
#endif
            for (int64_t t = 0; t < T; ++t) {
                double pv = bf2d(d->p[i * d->p_i + t * d->p_t]);
                double qv = bf2d(d->q[j * d->q_j + t * d->q_t]);
                double prod = pv * qv;           /* exact: <= 16 significant bits */
                s += prod;
                sa += fabs(prod);
            }
            d->out[i * d->J + j] = s;
            if (d->absout) d->absout[i * d->J + j] = sa;
        }
    }
}

static void *dot_thread(void *arg) { dot_rows((const dot_job *)arg); return NULL; }

static int n_threads(int requested)
{
    if (requested > 0) return requested;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void dot_all(dot_job job, int threads)
{
    int nt = n_threads(threads);
    if (nt > job.I) nt = (int)(job.I > 0 ? job.I : 1);
    if (nt <= 1) { job.i0 = 0; job.i1 = job.I; dot_rows(&job); return; }
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    dot_job *jobs = (dot_job *)malloc(sizeof(dot_job) * (size_t)nt);
    int started = 0;
    for (int w = 0; w < nt; ++w) {
        jobs[w] = job;
        jobs[w].i0 = job.I * w / nt;
        jobs[w].i1 = job.I * (w + 1) / nt;
        if (pthread_create(&tid[w], NULL, dot_thread, &jobs[w]) != 0) {
            dot_rows(&jobs[w]);          /* no thread: do that share here */
            tid[w] = (pthread_t)0;
        } else {
            ++started;
        }
    }
    for (int w = 0; w < nt; ++w)
        if (tid[w] != (pthread_t)0) pthread_join(tid[w], NULL);
    (void)started;
    free(jobs);
    free(tid);
}

/* scratch for the binary64 sums; the caller's S buffer is used when given */
static double *alloc_d(int64_t n) { return (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1)); }

/* ------------------------------------------------------ the operator steps */

/*
 * U[m][r] = rnbf(rn32(sum_k x[m][k] * a[r][k]))
 * ("U = X @ A^T, FP32 accumulate, round to BF16", section "Summary").
 * s_u (optional) = sum_k |x[m][k] * a[r][k]|.  f32_u (optional) = the rn32 value.
 */
int ora_u(const uint16_t *x, const uint16_t *a, int64_t M, int64_t K, int64_t R,
          uint16_t *u, float *f32_u, double *s_u, int threads)
{
    double *sum = alloc_d(M * R);
    if (!sum) return 1;
#if ORACLE_MUTANT == 2   /* planted: transposed operand (reads a as [K][R]) */
    dot_job j = { x, K, 1, a, 1, R, M, R, K, sum, s_u, 0, 0 };
#else
    dot_job j = { x, K, 1, a, K, 1, M, R, K, sum, s_u, 0, 0 };
#endif
    dot_all(j, threads);
    for (int64_t e = 0; e < M * R; ++e) {
        float f = rn32(sum[e]);
        if (f32_u) f32_u[e] = f;
#if ORACLE_MUTANT == 3   /* planted: skips the BF16 rounding point of U (truncates instead) */
        uint32_t bits; memcpy(&bits, &f, 4); u[e] = (uint16_t)(bits >> 16);
#else
        u[e] = rnbf(f);
#endif
    }
    free(sum);
    return 0;
}

/*
 * delta_y[m][n] = rn32( rn32(sum_r u[m][r] * b[n][r]) * alpha )
 * ("dY = (U @ B^T) * alpha, FP32 accumulate, FP32 output", section "Summary":
 * the accumulation is rounded to FP32, then scaled by alpha as one FP32
 * multiply). s_y (optional) = |alpha| * sum_r |u[m][r] * b[n][r]|.
 */
int ora_delta_y(const uint16_t *u, const uint16_t *b, float alpha, int64_t M, int64_t N,
                int64_t R, float *delta_y, double *s_y, int threads)
{
    double *sum = alloc_d(M * N);
    if (!sum) return 1;
    dot_job j = { u, R, 1, b, R, 1, M, N, R, sum, s_y, 0, 0 };
    dot_all(j, threads);
    for (int64_t e = 0; e < M * N; ++e) {
#if ORACLE_MUTANT == 4   /* planted: alpha never applied */
        delta_y[e] = rn32(sum[e]);
#elif ORACLE_MUTANT == 5 /* planted: wrong sign of the scale */
        delta_y[e] = rn32((double)rn32(sum[e]) * -(double)alpha);
#else
        delta_y[e] = rn32((double)rn32(sum[e]) * (double)alpha);
#endif
        if (s_y) s_y[e] *= fabs((double)alpha);
    }
    free(sum);
    return 0;
}

/*
 * delta_y_bf16[m][n] = rnbf(delta_y[m][n]): the BF16 output variant, the FP32
 * result of ora_delta_y rounded once more to bfloat16 (round to nearest even);
 * the half-size output asked for in the review thread of page "[DSv4][P5-3]
 * shared_grouped_lora_delta: CUDA + Triton, both batch-invariant".
 */
int ora_delta_y_bf16(const uint16_t *u, const uint16_t *b, float alpha, int64_t M, int64_t N,
                     int64_t R, uint16_t *delta_y_bf16, int threads)
{
    float *y = (float *)malloc((size_t)(M * N > 0 ? M * N : 1) * sizeof(float));
    if (!y) return 1;
    int rc = ora_delta_y(u, b, alpha, M, N, R, y, NULL, threads);
    for (int64_t e = 0; rc == 0 && e < M * N; ++e) {
#if ORACLE_MUTANT == 10  /* planted: the BF16 output truncated instead of rounded */
        uint32_t bits;
        memcpy(&bits, &y[e], 4);
        delta_y_bf16[e] = (uint16_t)(bits >> 16);
#else
        delta_y_bf16[e] = rnbf(y[e]);
#endif
    }
    free(y);
    return rc;
}

/*
 * dv[m][n] = rnbf(rn32(dy[m][n] * alpha))  ("dV = dY * alpha", rounded to BF16
 * between the GEMMs: "D4", section "Summary").
 */
int ora_dv(const uint16_t *dy, float alpha, int64_t M, int64_t N, uint16_t *dv)
{
    for (int64_t e = 0; e < M * N; ++e) {
#if ORACLE_MUTANT == 6   /* planted: dY * alpha kept at FP32 precision, then truncated */
        float f = rn32(bf2d(dy[e]) * (double)alpha);
        uint32_t bits; memcpy(&bits, &f, 4); dv[e] = (uint16_t)(bits >> 16);
#else
        dv[e] = rnbf(rn32(bf2d(dy[e]) * (double)alpha));
#endif
    }
    return 0;
}

/*
 * The FP32-dY input variant (the input counterpart of the BF16 output asked
 * for in the review thread of page "[DSv4][P5-3] shared_grouped_lora_delta:
 * CUDA + Triton, both batch-invariant"):
 * dv[m][n] = rnbf(rn32(dy[m][n] * alpha)) with dy read as binary32 (the product
 * of two binary32 values is exact in binary64; it is rounded to binary32, then
 * to bfloat16: two roundings, as for BF16 dY).
 */
int ora_dv_f32(const float *dy, float alpha, int64_t M, int64_t N, uint16_t *dv)
{
    for (int64_t e = 0; e < M * N; ++e) {
#if ORACLE_MUTANT == 11  /* planted: the binary32 product truncated to bfloat16 */
        float f = rn32((double)dy[e] * (double)alpha);
        uint32_t bits; memcpy(&bits, &f, 4); dv[e] = (uint16_t)(bits >> 16);
#else
        dv[e] = rnbf(rn32((double)dy[e] * (double)alpha));
#endif
    }
    return 0;
}

/*
 * du[m][r] = rnbf(rn32(sum_n dv[m][n] * b[n][r]))  ("dU = dV @ B", rounded to
 * BF16 between the GEMMs, section "Summary"). f32_du (optional) = the rn32 value.
 */
int ora_du(const uint16_t *dv, const uint16_t *b, int64_t M, int64_t N, int64_t R,
           uint16_t *du, float *f32_du, double *s_du, int threads)
{
    double *sum = alloc_d(M * R);
    if (!sum) return 1;
#if ORACLE_MUTANT == 9   /* planted: transposed operand (reads b as [R][N]) */
    dot_job j = { dv, N, 1, b, N, 1, M, R, N, sum, s_du, 0, 0 };
#else
    dot_job j = { dv, N, 1, b, 1, R, M, R, N, sum, s_du, 0, 0 };
#endif
    dot_all(j, threads);
    for (int64_t e = 0; e < M * R; ++e) {
        float f = rn32(sum[e]);
        if (f32_du) f32_du[e] = f;
        du[e] = rnbf(f);
    }
    free(sum);
    return 0;
}

/*
 * db[n][r] = rn32(sum_m dv[m][n] * u[m][r])  ("dB = dV^T @ U", FP32).
 */
int ora_db(const uint16_t *dv, const uint16_t *u, int64_t M, int64_t N, int64_t R,
           float *db, double *s_db, int threads)
{
    double *sum = alloc_d(N * R);
    if (!sum) return 1;
#if ORACLE_MUTANT == 7   /* planted: uses dU's partner U with the row index off by one */
    dot_job j = { dv, 1, N, u + R, 1, R, N, R, M - 1, sum, s_db, 0, 0 };
#else
    dot_job j = { dv, 1, N, u, 1, R, N, R, M, sum, s_db, 0, 0 };
#endif
    dot_all(j, threads);
    for (int64_t e = 0; e < N * R; ++e) db[e] = rn32(sum[e]);
    free(sum);
    return 0;
}

/*
 * dx[m][k] = rn32(sum_r du[m][r] * a[r][k])  ("dX = dU @ A", FP32).
 */
int ora_dx(const uint16_t *du, const uint16_t *a, int64_t M, int64_t K, int64_t R,
           float *dx, double *s_dx, int threads)
{
    double *sum = alloc_d(M * K);
    if (!sum) return 1;
    dot_job j = { du, R, 1, a, 1, K, M, K, R, sum, s_dx, 0, 0 };
    dot_all(j, threads);
    for (int64_t e = 0; e < M * K; ++e) dx[e] = rn32(sum[e]);
    free(sum);
    return 0;
}

/*
 * da[r][k] = rn32(sum_m du[m][r] * x[m][k])  ("dA = dU^T @ X", FP32).
 */
int ora_da(const uint16_t *du, const uint16_t *x, int64_t M, int64_t K, int64_t R,
           float *da, double *s_da, int threads)
{
    double *sum = alloc_d(R * K);
    if (!sum) return 1;
#if ORACLE_MUTANT == 8   /* planted: transposed operand (reads du as [R][M]) */
    dot_job j = { du, M, 1, x, 1, K, R, K, M, sum, s_da, 0, 0 };
#else
    dot_job j = { du, 1, R, x, 1, K, R, K, M, sum, s_da, 0, 0 };
#endif
    dot_all(j, threads);
    for (int64_t e = 0; e < R * K; ++e) da[e] = rn32(sum[e]);
    free(sum);
    return 0;
}

/* exported helpers so the tests can check the two rounding functions against
 * an independent exact-rational rounding */
float ora_rn32(double v) { return rn32(v); }
uint16_t ora_rnbf(float f) { return rnbf(f); }
int ora_mutant(void) { return ORACLE_MUTANT; }
int ora_threads(int requested) { return n_threads(requested); }
