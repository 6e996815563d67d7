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
 * Low-bit weight variant (sgr_ref_gemm_residual_w8): the weight arrives as
 * one FP8 code per element plus one FP32 scale per output column n, as in the
 * FP8 / k-bit weight work of the bitsandbytes "QLORA-2" page (its scalar
 * GEMV, "Three-Kernel Strategy": quantized weights, BF16 activations, the
 * block scale applied to the dot product).  The pages do not fix the FP8
 * encoding; the reading taken is OCP E4M3 without infinities (bias 7, three
 * fraction bits, subnormals, S.1111.111 = NaN), the format of
 * torch.float8_e4m3fn and of the tensor cores' e4m3 type:
 *
 *     Y[m,n] = bf16_rne( scale[n] * sum_k A[m,k] * e4m3(Wq[n,k])  +  R[m,n] )
 *
 * Each decoded code is exact in double; each product of a BF16 value and an
 * E4M3 value is exact (8 + 4 significant bits); the scale multiplies the FP64
 * sum once (one FP64 rounding), then R is added and the double is rounded to
 * BF16 as above.
 *
 * NVFP4 weight variant (sgr_ref_gemm_residual_w4): the pages name NVFP4
 * weights (the bitsandbytes "QLORA-2" page's NVFP4 sm100 GEMM targets) without
 * defining the format; the reading taken is the published NVFP4 layout: each
 * weight is a 4-bit E2M1 code (sign, 2 exponent bits with bias 1, 1 fraction
 * bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), two codes per byte with element
 * 2i in the low nibble and 2i+1 in the high nibble; every 16 consecutive
 * elements of a row share one E4M3 block scale; one FP32 scale covers the
 * whole tensor:
 *
 *     Y[m,n] = bf16_rne( gs * sum_k A[m,k] * e2m1(Wq[n,k]) * e4m3(bs[n,k/16])  +  R[m,n] )
 *
 * Each product of a BF16 value, an E2M1 value and an E4M3 value is exact in
 * double (8 + 2 + 4 significant bits); the sum runs in FP64 with k ascending;
 * gs multiplies it once; R is added and the double is rounded to BF16 once.
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
 * Exact E4M3 -> double.  Fields: sign s (bit 7), exponent e (bits 6-3, bias
 * 7), fraction f (bits 2-0).  e > 0: (1 + f/8) * 2^(e-7) = (8 + f) * 2^(e-10);
 * e = 0: subnormal f/8 * 2^-6 = f * 2^-9; e = 15 with f = 7 is NaN (the format
 * has no infinities, so e = 15, f < 7 are ordinary numbers up to 448).
 */
static double e4m3_to_double(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 15, f = b & 7;
#if SGR_REF_MUTANT == 12
    if (e == 15 && f == 7)
        return s ? -480.0 : 480.0;            /* planted: no NaN code */
#else
    if (e == 15 && f == 7)
        return NAN;
#endif
    double mag;
#if SGR_REF_MUTANT == 9
    mag = ldexp(8 + f, e - 10);               /* planted: subnormals read as normals */
#elif SGR_REF_MUTANT == 10
    mag = e == 0 ? ldexp(f, -10) : ldexp(8 + f, e - 11); /* planted: bias 8 */
#else
    mag = e == 0 ? ldexp(f, -9) : ldexp(8 + f, e - 10);
#endif
    return s ? -mag : mag;
}

/*
 * Exact E2M1 -> double for the 4-bit code in the low bits of c.  Fields: sign
 * s (bit 3), exponent e (bits 2-1, bias 1), fraction f (bit 0).  e > 0:
 * (1 + f/2) * 2^(e-1) = (2 + f) * 2^(e-2); e = 0: subnormal f/2.  The format
 * has neither infinities nor NaN.
 */
static double e2m1_to_double(uint8_t c)
{
    int s = (c >> 3) & 1, e = (c >> 1) & 3, f = c & 1;
    double mag;
#if SGR_REF_MUTANT == 16
    mag = ldexp(2 + f, e - 2);                /* planted: subnormals read as normals */
#else
    mag = e == 0 ? 0.5 * f : ldexp(2 + f, e - 2);
#endif
    return s ? -mag : mag;
}

/* Code of element k of a packed NVFP4 row (two codes per byte). */
static uint8_t e2m1_code(const uint8_t *row, long k)
{
    uint8_t b = row[k >> 1];
#if SGR_REF_MUTANT == 14
    return (k & 1) ? (b & 15) : (b >> 4);    /* planted: nibble order swapped */
#else
    return (k & 1) ? (b >> 4) : (b & 15);
#endif
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

/* The same for the low-bit weight variant:
 * t = scale * sum_k a[k]*e4m3(wq[k]) + r. */
static double dot_w8_plus_residual(const uint16_t *a, const uint8_t *wq, float scale,
                                   uint16_t r, long K)
{
    double s = 0.0;
    for (long k = 0; k < K; ++k)
        s += bf16_to_double(a[k]) * e4m3_to_double(wq[k]);
#if SGR_REF_MUTANT == 11
    return (double)scale * (s + bf16_to_double(r)); /* planted: residual scaled too */
#else
    return (double)scale * s + bf16_to_double(r);
#endif
}

/* The same for the NVFP4 variant:
 * t = gs * sum_k a[k]*e2m1(code k)*e4m3(bs[k/16]) + r. */
static double dot_w4_plus_residual(const uint16_t *a, const uint8_t *wq4, const uint8_t *bs, float gs,
                                   uint16_t r, long K)
{
    double s = 0.0;
    for (long k = 0; k < K; ++k) {
#if SGR_REF_MUTANT == 15
        double scale = e4m3_to_double(bs[k / 32]); /* planted: blocks of 32 */
#else
        double scale = e4m3_to_double(bs[k / 16]);
#endif
        s += bf16_to_double(a[k]) * e2m1_to_double(e2m1_code(wq4, k)) * scale;
    }
#if SGR_REF_MUTANT == 17
    return (double)gs * (s + bf16_to_double(r)); /* planted: residual scaled too */
#else
    return (double)gs * s + bf16_to_double(r);
#endif
}

typedef struct {
    const uint16_t *A, *W, *R;
    const uint8_t *Wq;    /* low-bit weights (W unused), or NULL */
    const float *scale;   /* per-column scales of Wq */
    const uint8_t *Wq4;   /* NVFP4 codes (W, Wq unused), or NULL */
    const uint8_t *bs;    /* E4M3 block scales of Wq4, row stride ldbs bytes */
    long ldbs;
    float gs;             /* tensor scale of Wq4 */
    uint16_t *Y;      /* rounded output, or NULL */
    double *T;        /* unrounded output, or NULL */
    long lda, ldw, ldr, ldy, ldt;
    long M, K, N;
    long n0, n1;      /* this worker's output columns [n0, n1) */
} ref_job;

/* Scale of output column n. */
static float column_scale(const float *scale, long n, long N)
{
#if SGR_REF_MUTANT == 13
    return scale[(n + 1) % N];                /* planted: neighbouring column's scale */
#else
    (void)N;
    return scale[n];
#endif
}

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
            double t = j->Wq4
                ? dot_w4_plus_residual(j->A + m * j->lda, j->Wq4 + n * j->ldw, j->bs + n * j->ldbs, j->gs,
                                       j->R[rrow * j->ldr + n], j->K)
                : j->Wq
                ? dot_w8_plus_residual(j->A + m * j->lda, j->Wq + n * j->ldw,
                                       column_scale(j->scale, n, j->N),
                                       j->R[rrow * j->ldr + n], j->K)
                : dot_plus_residual(j->A + m * j->lda, j->W + n * j->ldw,
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
static int run_ref4(const uint16_t *A, long lda, const uint16_t *W, const uint8_t *Wq,
                    const float *scale, const uint8_t *Wq4, const uint8_t *bs, long ldbs, float gs,
                    long ldw, const uint16_t *R, long ldr, uint16_t *Y, long ldy, double *T, long ldt,
                    long M, long N, long K, int threads)
{
    if (!A || (!W && !(Wq && scale) && !(Wq4 && bs)) || !R || (!Y && !T) || M < 0 || N < 0 || K < 0)
        return -1;
    if (Wq4 ? (K % 2 != 0 || ldw < K / 2 || ldbs < (K + 15) / 16) : ldw < K)
        return -1;
    if (lda < K || ldr < N || (Y && ldy < N) || (T && ldt < N))
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
        ref_job j = {A, W, R, Wq, scale, Wq4, bs, ldbs, gs, Y, T, lda, ldw, ldr, ldy, ldt, M, K, N,
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

static int run_ref(const uint16_t *A, long lda, const uint16_t *W, const uint8_t *Wq,
                   const float *scale, long ldw, const uint16_t *R, long ldr, uint16_t *Y,
                   long ldy, double *T, long ldt, long M, long N, long K, int threads)
{
    return run_ref4(A, lda, W, Wq, scale, NULL, NULL, 0, 0.0f, ldw, R, ldr, Y, ldy, T, ldt, M, N, K, threads);
}

/* Y = bf16_rne(A . W^T + R), every element. */
int sgr_ref_gemm_residual(const uint16_t *A, long lda, const uint16_t *W, long ldw,
                          const uint16_t *R, long ldr, uint16_t *Y, long ldy,
                          long M, long N, long K, int threads)
{
    return run_ref(A, lda, W, NULL, NULL, ldw, R, ldr, Y, ldy, NULL, 0, M, N, K, threads);
}

/* T = A . W^T + R in FP64, unrounded (for error analysis). */
int sgr_ref_gemm_residual_f64(const uint16_t *A, long lda, const uint16_t *W, long ldw,
                              const uint16_t *R, long ldr, double *T, long ldt,
                              long M, long N, long K, int threads)
{
    return run_ref(A, lda, W, NULL, NULL, ldw, R, ldr, NULL, 0, T, ldt, M, N, K, threads);
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

/* Low-bit weights: Y = bf16_rne(scale[n] * A . e4m3(Wq)^T + R), every
 * element.  Wq is [N,K] bytes with row stride ldw, scale has N entries. */
int sgr_ref_gemm_residual_w8(const uint16_t *A, long lda, const uint8_t *Wq, long ldw,
                             const float *scale, const uint16_t *R, long ldr, uint16_t *Y,
                             long ldy, long M, long N, long K, int threads)
{
    if (!Wq || !scale)
        return -1;
    return run_ref(A, lda, NULL, Wq, scale, ldw, R, ldr, Y, ldy, NULL, 0, M, N, K, threads);
}

/* Selected elements of the low-bit variant: out[i] = Y[ms[i], ns[i]]. */
int sgr_ref_sample_w8(const uint16_t *A, long lda, const uint8_t *Wq, long ldw,
                      const float *scale, const uint16_t *R, long ldr, long M, long N, long K,
                      const long *ms, const long *ns, long count, uint16_t *out)
{
    if (!A || !Wq || !scale || !R || !ms || !ns || !out || count < 0 || lda < K || ldw < K ||
        ldr < N)
        return -1;
    if (fegetround() != FE_TONEAREST)
        return -3;
    for (long i = 0; i < count; ++i) {
        long m = ms[i], n = ns[i];
        if (m < 0 || m >= M || n < 0 || n >= N)
            return -1;
        out[i] = sgr_ref_round_bf16(dot_w8_plus_residual(
            A + m * lda, Wq + n * ldw, column_scale(scale, n, N), R[m * ldr + n], K));
    }
    return 0;
}

double sgr_ref_e4m3_to_double(uint8_t b) { return e4m3_to_double(b); }

/* NVFP4 weights: Y = bf16_rne(gs * A . (e2m1(Wq4) * e4m3(bs))^T + R), every
 * element.  Wq4 is [N, K/2] bytes (two codes each) with row stride ldw bytes;
 * bs is [N, ceil(K/16)] E4M3 block scales with row stride ldbs bytes; K even. */
int sgr_ref_gemm_residual_w4(const uint16_t *A, long lda, const uint8_t *Wq4, long ldw, const uint8_t *bs,
                             long ldbs, float gs, const uint16_t *R, long ldr, uint16_t *Y, long ldy,
                             long M, long N, long K, int threads)
{
    if (!Wq4 || !bs)
        return -1;
    return run_ref4(A, lda, NULL, NULL, NULL, Wq4, bs, ldbs, gs, ldw, R, ldr, Y, ldy, NULL, 0, M, N, K, threads);
}

/* Selected elements of the NVFP4 variant: out[i] = Y[ms[i], ns[i]]. */
int sgr_ref_sample_w4(const uint16_t *A, long lda, const uint8_t *Wq4, long ldw, const uint8_t *bs, long ldbs,
                      float gs, const uint16_t *R, long ldr, long M, long N, long K, const long *ms,
                      const long *ns, long count, uint16_t *out)
{
    if (!A || !Wq4 || !bs || !R || !ms || !ns || !out || count < 0 || K % 2 != 0 || lda < K ||
        ldw < K / 2 || ldbs < (K + 15) / 16 || ldr < N)
        return -1;
    if (fegetround() != FE_TONEAREST)
        return -3;
    for (long i = 0; i < count; ++i) {
        long m = ms[i], n = ns[i];
        if (m < 0 || m >= M || n < 0 || n >= N)
            return -1;
        out[i] = sgr_ref_round_bf16(
            dot_w4_plus_residual(A + m * lda, Wq4 + n * ldw, bs + n * ldbs, gs, R[m * ldr + n], K));
    }
    return 0;
}

double sgr_ref_e2m1_to_double(uint8_t c) { return e2m1_to_double(c); }

int sgr_ref_mutant(void) { return SGR_REF_MUTANT; }
