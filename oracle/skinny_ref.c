/*
 * oracle/skinny_ref.c -- CPU oracle for the skinny BF16 projection GEMM with a
 * fused residual add.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and
 * the benchmark's CPU-baseline leg load it; the product path never does.  It
 * shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (vLLM "benchmark_k3_cutedsl_residual.py", module docstring:
 * BF16[M,3584] @ BF16[7168,3584].T + BF16[M,7168] with FP32 accumulation and
 * BF16 output; the same page's correctness() check builds its reference as
 * a.float() @ w.float().t() + r.float()):
 *
 *     Y[m,n] = bf16_rne( sum_k A[m,k] * W[n,k]  +  R[m,n] )
 *
 * Reading taken where the pages differ: the product is rounded to BF16 ONCE.
 * The vLLM "fused_add_multicast_skinny_gemm" page rounds the FP32 sum to BF16,
 * adds the residual in FP32 and rounds again (its kernel epilogue); the plain
 * definition has one rounding, and that is what this oracle returns.
 *
 * Arithmetic: every BF16 input is decoded exactly to double; each product of
 * two BF16 values is exact in double (8 + 8 significant bits); the sum runs in
 * FP64 with k ascending, then R is added in FP64, then the double is rounded
 * straight to BF16 with round-to-nearest-even (no intermediate float rounding).
 * The FP64 sum is within K * 2^-53 * sum|a*w| of the real value, far below one
 * BF16 unit in the last place, so the result is the correctly rounded value
 * except in ties closer than that bound.
 *
 * Layouts: A is [M,K] with row stride lda, W is [N,K] with row stride ldw (the
 * nn.Linear weight layout), R and Y are [M,N] with row strides ldr and ldy;
 * all strides in elements, inner stride 1.  BF16 values travel as uint16_t
 * bit patterns.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -pthread ... -lm
 * (no -ffast-math: the k order of the sum is part of the definition above).
 *
 * SGR_REF_MUTANT (compile-time, default 0) plants one known mistake so that
 * the test suite can show its pins catch it; a normal build never sets it.
 */
#define _POSIX_C_SOURCE 200809L
#include <fenv.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef SGR_REF_MUTANT
#define SGR_REF_MUTANT 0
#endif

/* Exact BF16 -> double: a BF16 pattern is the upper half of an IEEE binary32. */
static double bf16_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * Round a double to the nearest BF16 value, ties to the even significand
 * (IEEE 754 roundTiesToEven into a format with 8 significant bits and the
 * binary32 exponent range).  Steps: write |t| = f * 2^e with f in [0.5, 1);
 * BF16 numbers in [2^(e-1), 2^e) are spaced 2^(e-8) apart, and subnormal
 * BF16 numbers are spaced 2^-133 apart, so the quantum is q = 2^max(e-8,-133).
 * |t|/q is exact (a power-of-two scaling), nearbyint() rounds it to an
 * integer with ties to even under the default rounding mode, and the result
 * times q is a BF16 value (or 2^128, which overflows to infinity).
 */
uint16_t sgr_ref_round_bf16(double t)
{
    if (isnan(t))
        return 0x7FC0;
    uint16_t sign = signbit(t) ? 0x8000 : 0x0000;
    double a = fabs(t);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80);
    int e;
    (void)frexp(a, &e);
    int qexp = e - 8;
    if (qexp < -133)
        qexp = -133;
    double scaled = ldexp(a, -qexp);
#if SGR_REF_MUTANT == 5
    double r = trunc(scaled);                 /* planted: round toward zero */
#elif SGR_REF_MUTANT == 6
    double r = round(scaled);                 /* planted: ties away from zero */
#else
    double r = nearbyint(scaled);
#endif
    double y = ldexp(r, qexp);
    if (y >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80);
    float f = (float)y; /* exact: y has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

void sgr_ref_round_bf16_array(const double *t, uint16_t *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = sgr_ref_round_bf16(t[i]);
}

double sgr_ref_bf16_to_double(uint16_t h) { return bf16_to_double(h); }

/* The unrounded FP64 value t = sum_k a[k]*w[k] + r for one output element. */
static double dot_plus_residual(const uint16_t *a, const uint16_t *w, uint16_t r, long K)
{
    double s = 0.0;
#if SGR_REF_MUTANT == 3
    for (long k = 0; k + 1 < K; ++k)          /* planted: last k dropped */
#else
    for (long k = 0; k < K; ++k)
#endif
    {
#if SGR_REF_MUTANT == 7
        s = (double)(float)(s + bf16_to_double(a[k]) * bf16_to_double(w[k])); /* planted: FP32 sum */
#else
        s += bf16_to_double(a[k]) * bf16_to_double(w[k]);
#endif
    }
#if SGR_REF_MUTANT == 1
    (void)r;
    return s;                                 /* planted: residual dropped */
#elif SGR_REF_MUTANT == 2
    return bf16_to_double(sgr_ref_round_bf16(s)) + bf16_to_double(r); /* planted: round, then add */
#elif SGR_REF_MUTANT == 4
    return s - bf16_to_double(r);             /* planted: residual sign */
#else
    return s + bf16_to_double(r);
#endif
}

typedef struct {
    const uint16_t *A, *W, *R;
    uint16_t *Y;      /* rounded output, or NULL */
    double *T;        /* unrounded output, or NULL */
    long lda, ldw, ldr, ldy, ldt;
    long M, K;
    long n0, n1;      /* this worker's output columns [n0, n1) */
} ref_job;

static void *ref_worker(void *p)
{
    const ref_job *j = (const ref_job *)p;
    for (long m = 0; m < j->M; ++m) {
        for (long n = j->n0; n < j->n1; ++n) {
#if SGR_REF_MUTANT == 8
            long rrow = j->M - 1 - m;         /* planted: residual from the wrong row */
#else
            long rrow = m;
#endif
            double t = dot_plus_residual(j->A + m * j->lda, j->W + n * j->ldw,
                                         j->R[rrow * j->ldr + n], j->K);
            long out = m * j->ldy + n;
            if (j->Y)
                j->Y[out] = sgr_ref_round_bf16(t);
            if (j->T)
                j->T[m * j->ldt + n] = t;
        }
    }
    return NULL;
}

/* Returns 0 on success, -1 on bad arguments, -2 if threads could not start,
 * -3 if the FP rounding mode is not round-to-nearest. */
static int run_ref(const uint16_t *A, long lda, const uint16_t *W, long ldw,
                   const uint16_t *R, long ldr, uint16_t *Y, long ldy,
                   double *T, long ldt, long M, long N, long K, int threads)
{
    if (!A || !W || !R || (!Y && !T) || M < 0 || N < 0 || K < 0)
        return -1;
    if (lda < K || ldw < K || ldr < N || (Y && ldy < N) || (T && ldt < N))
        return -1;
    if (fegetround() != FE_TONEAREST)
        return -3;
    if (M == 0 || N == 0)
        return 0;
    if (threads < 1)
        threads = 1;
    if (threads > 256)
        threads = 256;
    if (threads > N)
        threads = (int)N;
    ref_job jobs[256];
    pthread_t tids[256];
    for (int i = 0; i < threads; ++i) {
        ref_job j = {A, W, R, Y, T, lda, ldw, ldr, ldy, ldt, M, K,
                     N * i / threads, N * (i + 1) / threads};
        jobs[i] = j;
    }
    int started = 0, rc = 0;
    for (int i = 1; i < threads; ++i) {
        if (pthread_create(&tids[i], NULL, ref_worker, &jobs[i]) != 0) {
            rc = -2;
            break;
        }
        ++started;
    }
    if (rc == 0)
        ref_worker(&jobs[0]);
    for (int i = 1; i <= started; ++i)
        pthread_join(tids[i], NULL);
    return rc;
}

/* Y = bf16_rne(A . W^T + R), every element. */
int sgr_ref_gemm_residual(const uint16_t *A, long lda, const uint16_t *W, long ldw,
                          const uint16_t *R, long ldr, uint16_t *Y, long ldy,
                          long M, long N, long K, int threads)
{
    return run_ref(A, lda, W, ldw, R, ldr, Y, ldy, NULL, 0, M, N, K, threads);
}

/* T = A . W^T + R in FP64, unrounded (for error analysis). */
int sgr_ref_gemm_residual_f64(const uint16_t *A, long lda, const uint16_t *W, long ldw,
                              const uint16_t *R, long ldr, double *T, long ldt,
                              long M, long N, long K, int threads)
{
    return run_ref(A, lda, W, ldw, R, ldr, NULL, 0, T, ldt, M, N, K, threads);
}

/* Selected elements only: out[i] = Y[ms[i], ns[i]].  For full-size checks
 * where computing every element would take too long. */
int sgr_ref_sample(const uint16_t *A, long lda, const uint16_t *W, long ldw,
                   const uint16_t *R, long ldr, long M, long N, long K,
                   const long *ms, const long *ns, long count, uint16_t *out)
{
    if (!A || !W || !R || !ms || !ns || !out || count < 0 || lda < K || ldw < K || ldr < N)
        return -1;
    if (fegetround() != FE_TONEAREST)
        return -3;
    for (long i = 0; i < count; ++i) {
        long m = ms[i], n = ns[i];
        if (m < 0 || m >= M || n < 0 || n >= N)
            return -1;
        out[i] = sgr_ref_round_bf16(dot_plus_residual(A + m * lda, W + n * ldw, R[m * ldr + n], K));
    }
    return 0;
}

int sgr_ref_mutant(void) { return SGR_REF_MUTANT; }
