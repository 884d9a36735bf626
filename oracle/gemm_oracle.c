/*
 * gemm_oracle.c -- CPU oracle for D = alpha * op(A) * op(B) + beta * C.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain reference that the
 * CUDA library is checked against.  Only the test suite, the package's smoke
 * check and the benchmark's CPU-baseline / reference arm may load it.  It
 * shares no code, header, table or helper with the CUDA library, and the
 * library never calls it.
 *
 * What it computes (the GEMM definition, "GEMM on NVIDIA GPUs: from naive
 * kernel to tiled pipeline", section 1 "GEMM definition"):
 *
 *     D_ij = alpha * sum_{k=0}^{K-1} A_ik * B_kj + beta * C_ij
 *
 * for every 0 <= i < M, 0 <= j < N, with op(A) an M x K matrix and op(B) a
 * K x N matrix ("op" is identity or transpose; here it is expressed as the
 * storage order of each operand, see below).
 *
 * How:
 *   - Inputs are exactly the bits the GPU receives: FP32 values, or BF16 or
 *     FP16 values (raw 16-bit patterns) widened exactly to double.
 *   - Every product A_ik * B_kj is formed in double.  It is exact: a product
 *     of two FP32 (24-bit significand), FP16 (11-bit) or BF16 (8-bit)
 *     numbers needs at most 48 significand bits, and double has 53; FP16
 *     products span at most 2^-48 .. 2^32, well inside double's range.
 *   - The products are summed over k in increasing order in double, then
 *     d = alpha * s + beta * C_ij in double (IEEE round-to-nearest-even, no
 *     contraction: build with -ffp-contract=off).
 *   - beta == 0: C is not read (it may be NULL).  alpha == 0: A and B are not
 *     read and the sum is taken as zero.  K == 0: the sum is empty (zero).
 *     These follow the reading that C traffic only counts when beta != 0
 *     ("GEMM on NVIDIA GPUs", section 2 "GEMM arithmetic intensity") and the
 *     usual BLAS convention for alpha == 0.
 *   - Alongside d it returns S_ij = sum_k |alpha * A_ik * B_kj| in double,
 *     the scale that the error bounds of the GPU comparison are written in.
 *
 * Storage orders: for an operand X with logical shape R x Q and leading
 * dimension ld, ORDER_ROW stores X(r, q) at X[r * ld + q] and ORDER_COL at
 * X[r + q * ld].  D and S are written dense row-major (M x N).
 *
 * Threading: rows of D (or the list of sample points) are split into
 * contiguous blocks, one POSIX thread per block.  Each output entry is
 * computed by exactly the same sequential loop whatever the thread count,
 * so results do not depend on it.
 *
 * Parity pins (tests/test_oracle_pins.py): the 4x4 product with 2x2 tiles
 * traced by hand in "Understanding roofline and tiling through matrix
 * multiplication", section 6.2; identity and permutation matrices; the
 * alpha/beta closed forms; brute force over tiny shapes and every storage
 * order against an independent loop; tiled == naive at N = 2, 4, 8 with
 * small integers (same page, section 10.3).
 */
#define _DEFAULT_SOURCE /* M_PI */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_IN_F32 0
#define ORACLE_IN_BF16 1
#define ORACLE_IN_F16 2
#define ORACLE_ROW 0
#define ORACLE_COL 1
#define ORACLE_MAX_THREADS 256

typedef struct {
    int in_type;
    int64_t M, N, K;
    double alpha, beta;
    const void *A;
    int64_t lda;
    int order_a;
    const void *B;
    int64_t ldb;
    int order_b;
    const float *C;
    int64_t ldc;
    int order_c;
} problem_t;

/* A BF16 number is the upper half of an FP32 bit pattern: widen exactly. */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE 754 binary16: sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Normal numbers are (1024 + fraction) * 2^(exponent - 25), subnormals
 * fraction * 2^-24; exponent 31 holds infinities and NaNs.  Exact in double. */
static double f16_to_double(uint16_t bits) {
    const int sign = bits >> 15, exponent = (bits >> 10) & 0x1f, fraction = bits & 0x3ff;
    double v;
    if (exponent == 0)
        v = ldexp((double)fraction, -24);
    else if (exponent == 31)
        v = fraction ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + fraction), exponent - 25);
    return sign ? -v : v;
}

static int64_t offset(int order, int64_t ld, int64_t r, int64_t q) {
    return order == ORACLE_ROW ? r * ld + q : r + q * ld;
}

static double load_in(const problem_t *p, const void *base, int64_t off) {
    if (p->in_type == ORACLE_IN_F32) return (double)((const float *)base)[off];
    if (p->in_type == ORACLE_IN_F16) return f16_to_double(((const uint16_t *)base)[off]);
    return bf16_to_double(((const uint16_t *)base)[off]);
}

/* One output entry: the definition written out. */
static void entry(const problem_t *p, int64_t i, int64_t j, double *d_out, double *s_out) {
    double sum = 0.0, scale = 0.0;
    if (p->alpha != 0.0) {
        for (int64_t k = 0; k < p->K; ++k) {
            double a = load_in(p, p->A, offset(p->order_a, p->lda, i, k));
            double b = load_in(p, p->B, offset(p->order_b, p->ldb, k, j));
            double prod = a * b; /* exact in double */
            sum += prod;
            scale += fabs(p->alpha * prod);
        }
    }
    double d = p->alpha * sum;
    if (p->beta != 0.0) {
        double c = (double)p->C[offset(p->order_c, p->ldc, i, j)];
        d = d + p->beta * c;
    }
    *d_out = d;
    if (s_out) *s_out = scale;
}

typedef struct {
    const problem_t *p;
    int64_t first, last; /* half-open range of work items */
    /* full mode: items are rows; points mode: items are indices into I/J */
    const int64_t *I, *J;
    double *D, *S;
} work_t;

static void *run_rows(void *arg) {
    work_t *w = (work_t *)arg;
    const problem_t *p = w->p;
    for (int64_t i = w->first; i < w->last; ++i)
        for (int64_t j = 0; j < p->N; ++j)
            entry(p, i, j, &w->D[i * p->N + j], w->S ? &w->S[i * p->N + j] : NULL);
    return NULL;
}

static void *run_points(void *arg) {
    work_t *w = (work_t *)arg;
    for (int64_t t = w->first; t < w->last; ++t)
        entry(w->p, w->I[t], w->J[t], &w->D[t], w->S ? &w->S[t] : NULL);
    return NULL;
}

static int pick_threads(int nthreads, int64_t items) {
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    if (nthreads > ORACLE_MAX_THREADS) nthreads = ORACLE_MAX_THREADS;
    if ((int64_t)nthreads > items) nthreads = items > 0 ? (int)items : 1;
    return nthreads;
}

static int run_parallel(const problem_t *p, int64_t items, void *(*fn)(void *), const int64_t *I,
                        const int64_t *J, double *D, double *S, int nthreads) {
    nthreads = pick_threads(nthreads, items);
    pthread_t tid[ORACLE_MAX_THREADS];
    work_t work[ORACLE_MAX_THREADS];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        work[t].p = p;
        work[t].first = items * t / nthreads;
        work[t].last = items * (t + 1) / nthreads;
        work[t].I = I;
        work[t].J = J;
        work[t].D = D;
        work[t].S = S;
    }
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, fn, &work[t]) != 0) break;
        started = t;
    }
    /* the calling thread takes block 0, and any block whose thread failed to start */
    fn(&work[0]);
    for (int t = started + 1; t < nthreads; ++t) fn(&work[t]);
    for (int t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
    return 0;
}

static int check(const problem_t *p) {
    if (p->M < 0 || p->N < 0 || p->K < 0) return -1;
    if (p->in_type != ORACLE_IN_F32 && p->in_type != ORACLE_IN_BF16 && p->in_type != ORACLE_IN_F16)
        return -1;
    if ((p->order_a | p->order_b | p->order_c) & ~1) return -1;
    if (p->alpha != 0.0 && p->K > 0 && p->M > 0 && p->N > 0 && (!p->A || !p->B)) return -1;
    if (p->beta != 0.0 && p->M > 0 && p->N > 0 && !p->C) return -1;
    return 0;
}

/* Full result: D and S (S may be NULL) dense row-major M x N.  Returns 0, or -1 on bad arguments. */
int oracle_gemm(int in_type, int64_t M, int64_t N, int64_t K, double alpha, const void *A,
                int64_t lda, int order_a, const void *B, int64_t ldb, int order_b, double beta,
                const float *C, int64_t ldc, int order_c, double *D, double *S, int nthreads) {
    problem_t p = {in_type, M, N, K, alpha, beta, A, lda, order_a, B, ldb, order_b, C, ldc, order_c};
    if (check(&p) != 0 || (M > 0 && N > 0 && !D)) return -1;
    if (M == 0 || N == 0) return 0;
    return run_parallel(&p, M, run_rows, NULL, NULL, D, S, nthreads);
}

/* Selected entries: D[t], S[t] for the point (I[t], J[t]), t < npts. */
int oracle_gemm_points(int in_type, int64_t M, int64_t N, int64_t K, double alpha, const void *A,
                       int64_t lda, int order_a, const void *B, int64_t ldb, int order_b,
                       double beta, const float *C, int64_t ldc, int order_c, int64_t npts,
                       const int64_t *I, const int64_t *J, double *D, double *S, int nthreads) {
    problem_t p = {in_type, M, N, K, alpha, beta, A, lda, order_a, B, ldb, order_b, C, ldc, order_c};
    if (check(&p) != 0 || npts < 0 || (npts > 0 && (!I || !J || !D))) return -1;
    for (int64_t t = 0; t < npts; ++t)
        if (I[t] < 0 || I[t] >= M || J[t] < 0 || J[t] >= N) return -1;
    if (npts == 0) return 0;
    return run_parallel(&p, npts, run_points, I, J, D, S, nthreads);
}

/*
 * Fused epilogue, in place on a dense row-major M x N result D (double):
 * D_ij = act(D_ij + bias_j) -- bias_j added to column j when bias != NULL --
 * with act = identity (0), ReLU max(x, 0) (1) or GELU in its tanh form
 * 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) (2), in double.  This is
 * the "bias, activation" step of the epilogue in "GEMM on NVIDIA GPUs",
 * section 4 "Epilogue"; the GELU form is the published tanh approximation
 * (Hendrycks & Gimpel).  Returns 0, or -1 for an unknown activation.
 */
int oracle_epilogue(int64_t M, int64_t N, double *D, const float *bias, int act) {
    if (act < 0 || act > 2 || M < 0 || N < 0) return -1;
    const double sqrt_2_over_pi = sqrt(2.0 / M_PI);
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double x = D[i * N + j];
            if (bias) x += (double)bias[j];
            if (act == 1)
                x = x > 0.0 ? x : 0.0;
            else if (act == 2)
                x = 0.5 * x * (1.0 + tanh(sqrt_2_over_pi * (x + 0.044715 * x * x * x)));
            D[i * N + j] = x;
        }
    }
    return 0;
}

/* Threads the oracle uses for nthreads <= 0 (for reporting). */
int oracle_default_threads(void) { return pick_threads(0, 1 << 30); }
