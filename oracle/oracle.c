/*
 * oracle.c -- the CPU reference for the dense GEMM hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * includes this file; only the tests, the smoke check and the bench's CPU
 * baseline leg load it (through oracle/__init__.py).  It shares no header,
 * helper, table or constant with the CUDA sources.
 *
 * What it computes, and where that is defined:
 *
 *   C[b][i][j] = alpha * sum_{k<K} A[b][i][k] * opB[b][k][j] + beta * C0[b][i][j]
 *
 *   - "4.1 Toi uu hieu nang toan tu GEMM tren CUDA" (infra-guide), section 1.1
 *     (GEMM definition, C = alpha*A*B + beta*C; the formula itself was lost in
 *     extraction, the surrounding text names A as MxK, B as KxN, C as MxN) and
 *     section 3.1 (row-major indexing A[row*K+k], B[k*N+col]).
 *   - MUSA learning centre lesson m11-l5, Case 4 "GEMM": C_ij = sum_k A_ik B_kj.
 *   - "Operator & Runtime" (AI infra book ch. 5), section 5.2.1: the i,j,k
 *     element loop, the i,k,j reordering that walks W rows contiguously, and
 *     F_gemm = 2MKN.
 *   - Same page, sections 5.4.2-5.4.3: the accumulator is kept wide for the
 *     whole K reduction and is rounded to BF16 exactly once afterwards.
 *   - The batch dimension ("Batched GEMM" in multi-head attention, GEMM page
 *     section 1.2) is a plain loop over independent problems with element
 *     strides between them.
 *
 * Arithmetic: every input is widened exactly to IEEE double (float32 and
 * bfloat16 are subsets of double), alpha and beta are the float32 values the
 * GPU receives, widened.  The sum over k is taken in double in increasing k
 * order, one row at a time (the i,k,j order of section 5.2.1).  No blocking,
 * no fusion and no reordering beyond that.
 *
 * BF16 output rounding (oracle_round_bf16) is written from the IEEE-754
 * definition of round-to-nearest-even on the 8-bit significand of bfloat16.
 *
 * Pins (tests/test_oracle_pins.py): hand-computed 2x2 / 3x3 products
 * (tests/golden/), identity and permutation matrices, the rank-1 closed form,
 * alpha/beta special cases, numpy's float64 matmul on small integer inputs,
 * BF16 rounding of values whose rounding the IEEE definition fixes, and the
 * FLOP / byte counts printed by the "Operator & Runtime" page (103 GFLOP,
 * 128 MiB).  Every function below is pinned by at least one of them.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Element types of the input arrays. */
enum { OR_F32 = 0, OR_BF16 = 1, OR_F64 = 2 };

/* Exact widening of one input element to double. */
static double load_elem(const void *p, int type, int64_t idx) {
    if (type == OR_F32) return (double)((const float *)p)[idx];
    if (type == OR_F64) return ((const double *)p)[idx];
    /* bfloat16: the upper 16 bits of an IEEE binary32 */
    uint32_t bits = (uint32_t)((const uint16_t *)p)[idx] << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

/* Widens n bfloat16 values (given as raw 16-bit patterns) to double. */
void oracle_bf16_to_double(const uint16_t *in, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = load_elem(in, OR_BF16, i);
}

/* One GEMM problem description, shared by the worker threads. */
typedef struct {
    int64_t M, N, K;
    double alpha, beta;
    const void *A; int a_type; int64_t lda;
    const void *B; int b_type; int64_t ldb; int op_b;
    const void *C0; int c_type; int64_t ldc;
    double *C;         /* output, row stride ldo */
    int64_t ldo;
    int absolute;      /* 1: accumulate |alpha*a*b| and add |beta*c0| */
    const double *Bd;  /* op(B) widened to double, K x N, row-major */
    int64_t row_begin, row_end;
} job_t;

/* op(B)[k][j]: N -> B[k*ldb + j]; T -> B[j*ldb + k]. */
static double load_opb(const job_t *j, int64_t k, int64_t col) {
    int64_t idx = j->op_b ? col * j->ldb + k : k * j->ldb + col;
    return load_elem(j->B, j->b_type, idx);
}

/* Rows [row_begin, row_end) of one problem, in the i,k,j order of the
 * "Operator & Runtime" page, section 5.2.1. */
static void *rows_worker(void *arg) {
    const job_t *j = (const job_t *)arg;
    double *acc = (double *)malloc(sizeof(double) * (size_t)(j->N > 0 ? j->N : 1));
    for (int64_t i = j->row_begin; i < j->row_end; ++i) {
        for (int64_t c = 0; c < j->N; ++c) acc[c] = 0.0;
        for (int64_t k = 0; k < j->K; ++k) {
            double a = load_elem(j->A, j->a_type, i * j->lda + k);
            const double *brow = j->Bd + k * j->N;
            if (j->absolute) {
                for (int64_t c = 0; c < j->N; ++c) acc[c] += fabs(j->alpha * a * brow[c]);
            } else {
                for (int64_t c = 0; c < j->N; ++c) acc[c] += a * brow[c];
            }
        }
        for (int64_t c = 0; c < j->N; ++c) {
            double c0 = 0.0;
            /* beta == 0: C0 is not read, so NaN/Inf in it cannot reach C
             * (the BLAS convention; the pages are silent). */
            if (j->beta != 0.0 && j->C0) c0 = load_elem(j->C0, j->c_type, i * j->ldc + c);
            double out;
            if (j->absolute) out = acc[c] + fabs(j->beta * c0);
            else out = j->alpha * acc[c] + j->beta * c0;
            j->C[i * j->ldo + c] = out;
        }
    }
    free(acc);
    return NULL;
}

/* Runs one problem over nthreads threads split by rows. */
static int run_problem(job_t *base, int nthreads) {
    if (base->M <= 0 || base->N <= 0) return 0;
    /* op(B) as a K x N double matrix: one exact widening per element. */
    double *Bd = (double *)malloc(sizeof(double) * (size_t)(base->K > 0 ? base->K : 1) * (size_t)base->N);
    if (!Bd) return -1;
    for (int64_t k = 0; k < base->K; ++k)
        for (int64_t c = 0; c < base->N; ++c) Bd[k * base->N + c] = load_opb(base, k, c);
    base->Bd = Bd;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > base->M) nthreads = (int)base->M;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)nthreads);
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *base;
        jobs[t].row_begin = base->M * t / nthreads;
        jobs[t].row_end = base->M * (t + 1) / nthreads;
        if (nthreads == 1 || pthread_create(&th[t], NULL, rows_worker, &jobs[t]) != 0) {
            rows_worker(&jobs[t]);
            th[t] = 0;
        } else {
            ++started;
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (th[t]) pthread_join(th[t], NULL);
    (void)started;
    free(jobs);
    free(th);
    free(Bd);
    return 0;
}

static int gemm_common(int64_t batch, int64_t M, int64_t N, int64_t K, double alpha,
                       const void *A, int a_type, int64_t lda, int64_t strideA,
                       const void *B, int b_type, int64_t ldb, int64_t strideB, int op_b,
                       double beta, const void *C0, int c_type, int64_t ldc, int64_t strideC,
                       double *C, int64_t ldo, int64_t strideO, int absolute, int nthreads) {
    if (batch < 0 || M < 0 || N < 0 || K < 0) return -2;
    size_t esz_a = a_type == OR_F32 ? 4 : a_type == OR_BF16 ? 2 : 8;
    size_t esz_b = b_type == OR_F32 ? 4 : b_type == OR_BF16 ? 2 : 8;
    size_t esz_c = c_type == OR_F32 ? 4 : c_type == OR_BF16 ? 2 : 8;
    for (int64_t b = 0; b < batch; ++b) {
        job_t j;
        memset(&j, 0, sizeof j);
        j.M = M; j.N = N; j.K = K; j.alpha = alpha; j.beta = beta;
        j.A = (const char *)A + (size_t)(b * strideA) * esz_a; j.a_type = a_type; j.lda = lda;
        j.B = (const char *)B + (size_t)(b * strideB) * esz_b; j.b_type = b_type; j.ldb = ldb; j.op_b = op_b;
        j.C0 = C0 ? (const char *)C0 + (size_t)(b * strideC) * esz_c : NULL; j.c_type = c_type; j.ldc = ldc;
        j.C = C + b * strideO; j.ldo = ldo;
        j.absolute = absolute;
        if (run_problem(&j, nthreads) != 0) return -1;
    }
    return 0;
}

/*
 * Strided-batched GEMM in double.  Output C is double, row stride ldo, batch
 * stride strideO (elements).  a/b/c types: 0 float32, 1 bfloat16 bits, 2 double.
 * op_b: 0 -> op(B)[k][j] = B[k*ldb+j]; 1 -> op(B)[k][j] = B[j*ldb+k].
 * C0 may be NULL (treated as zeros).  Returns 0 on success.
 */
int oracle_gemm(int64_t batch, int64_t M, int64_t N, int64_t K, double alpha,
                const void *A, int a_type, int64_t lda, int64_t strideA,
                const void *B, int b_type, int64_t ldb, int64_t strideB, int op_b,
                double beta, const void *C0, int c_type, int64_t ldc, int64_t strideC,
                double *C, int64_t ldo, int64_t strideO, int nthreads) {
    return gemm_common(batch, M, N, K, alpha, A, a_type, lda, strideA, B, b_type, ldb, strideB,
                       op_b, beta, C0, c_type, ldc, strideC, C, ldo, strideO, 0, nthreads);
}

/*
 * The error scale of each output: D[b][i][j] = sum_k |alpha*a_ik*b_kj| + |beta*c0_ij|.
 * This is the denominator of the normalised error bound; it is the same loop as
 * oracle_gemm with absolute values taken term by term.
 */
int oracle_gemm_absden(int64_t batch, int64_t M, int64_t N, int64_t K, double alpha,
                       const void *A, int a_type, int64_t lda, int64_t strideA,
                       const void *B, int b_type, int64_t ldb, int64_t strideB, int op_b,
                       double beta, const void *C0, int c_type, int64_t ldc, int64_t strideC,
                       double *D, int64_t ldo, int64_t strideO, int nthreads) {
    return gemm_common(batch, M, N, K, alpha, A, a_type, lda, strideA, B, b_type, ldb, strideB,
                       op_b, beta, C0, c_type, ldc, strideC, D, ldo, strideO, 1, nthreads);
}

/*
 * Selected outputs only, one dot product each (for full-size problems whose
 * complete product would take the CPU too long).  For sample s the output is
 * C[bidx[s]][rows[s]][cols[s]] with its error scale in den[s].
 */
int oracle_gemm_entries(int64_t M, int64_t N, int64_t K, double alpha,
                        const void *A, int a_type, int64_t lda, int64_t strideA,
                        const void *B, int b_type, int64_t ldb, int64_t strideB, int op_b,
                        double beta, const void *C0, int c_type, int64_t ldc, int64_t strideC,
                        int64_t n, const int64_t *bidx, const int64_t *rows, const int64_t *cols,
                        double *out, double *den) {
    for (int64_t s = 0; s < n; ++s) {
        int64_t b = bidx ? bidx[s] : 0, i = rows[s], c = cols[s];
        if (i < 0 || i >= M || c < 0 || c >= N || b < 0) return -2;
        double acc = 0.0, absacc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = load_elem(A, a_type, b * strideA + i * lda + k);
            int64_t bi = op_b ? c * ldb + k : k * ldb + c;
            double w = load_elem(B, b_type, b * strideB + bi);
            acc += a * w;
            absacc += fabs(alpha * a * w);
        }
        double c0 = 0.0;
        if (beta != 0.0 && C0) c0 = load_elem(C0, c_type, b * strideC + i * ldc + c);
        out[s] = alpha * acc + beta * c0;
        if (den) den[s] = absacc + fabs(beta * c0);
    }
    return 0;
}

/*
 * Round-to-nearest-even of a double to bfloat16 (1 sign, 8 exponent, 7 stored
 * significand bits), written from the IEEE-754 rounding rule: among the two
 * neighbouring representable values pick the nearer, on a tie the one whose
 * last significand bit is 0; magnitudes at or beyond 2^128 * (1 - 2^-9) round
 * to infinity; NaN stays NaN (quiet, sign kept).  Subnormals are rounded at
 * the fixed quantum 2^-133.
 */
static uint16_t round_one_bf16(double x) {
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7FC0);
    if (isinf(x)) return (uint16_t)(sign | 0x7F80);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);               /* a = f * 2^e, f in [0.5, 1) */
    int exp_unb = e - 1;        /* a in [2^exp_unb, 2^(exp_unb+1)) */
    if (exp_unb < -126) exp_unb = -126;        /* subnormal range: fixed quantum */
    double quantum = ldexp(1.0, exp_unb - 7);  /* spacing of bf16 values there */
    double q = a / quantum;                    /* exact: scaling by a power of two */
    double fl = floor(q);
    double rem = q - fl;
    double r;
    if (rem > 0.5) r = fl + 1.0;
    else if (rem < 0.5) r = fl;
    else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double v = r * quantum;     /* exact */
    if (v >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    /* encode v */
    if (v < ldexp(1.0, -126)) {
        /* subnormal: v = m * 2^-133, m in [1, 127] */
        uint16_t m = (uint16_t)(v / ldexp(1.0, -133));
        return (uint16_t)(sign | m);
    }
    int ev;
    double fv = frexp(v, &ev);  /* v = fv * 2^ev, fv in [0.5,1) */
    int biased = ev - 1 + 127;
    uint16_t mant = (uint16_t)((fv * 2.0 - 1.0) * 128.0); /* 7 bits, exact */
    return (uint16_t)(sign | (uint16_t)(biased << 7) | mant);
}

void oracle_round_bf16(const double *x, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = round_one_bf16(x[i]);
}

/* Spacing of bfloat16 values at magnitude |x| (one unit in the last place):
 * 2^(floor(log2|x|) - 7) for normal magnitudes, 2^-133 below 2^-126. */
double oracle_ulp_bf16(double x) {
    double a = fabs(x);
    if (isnan(a) || isinf(a)) return a;
    if (a < ldexp(1.0, -126)) return ldexp(1.0, -133);
    int e;
    frexp(a, &e);
    return ldexp(1.0, e - 1 - 7);
}

void oracle_ulp_bf16_array(const double *x, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_ulp_bf16(x[i]);
}

/* Algorithmic FLOP count of one GEMM: one multiply and one add per (i,j,k)
 * ("Operator & Runtime", section 5.2.1, F_gemm = 2MKN). */
double oracle_gemm_flops(int64_t batch, int64_t M, int64_t N, int64_t K) {
    return 2.0 * (double)batch * (double)M * (double)N * (double)K;
}
