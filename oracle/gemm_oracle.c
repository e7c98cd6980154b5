/*
 * CPU oracle for the dense fp16 NT matrix multiply  C[M,N] = A[M,K] · B[N,K]ᵀ.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant with the
 * CUDA path.
 *
 * What it computes (the plain definition, no blocking, no reordering):
 *
 *     C_ref[m,n] = RNE_fp16( sum_{k=0}^{K-1} (double)A[m,k] * (double)B[n,k] )
 *
 *  - Operand layout: A is M rows of K halves (row m starts at A + m*lda), B is
 *    N rows of K halves (row n at B + n*ldb), and the product contracts the K
 *    axis of both, i.e. B enters transposed.  Source: Tilus matmul-hopper
 *    tutorial, "3. Warp Specialization", §The Full Kernel (global views
 *    ga[m_size,k_size], gb[n_size,k_size], the MMA on sa and sb.transpose()).
 *  - Accumulation: the pages accumulate in fp32 registers ("4. Pipeline
 *    Abstraction and Two Consumer Warp Groups", §The Full Kernel, the float32
 *    register tensors; "6. Register Reallocation, Multicast, and a Persistent
 *    Kernel", opening list, "keeps fp32 accumulation").  The oracle sums in
 *    fp64, sequentially in k, so that its only rounding that matters is the
 *    final one; the products of two fp16 values are exact in fp64.
 *  - Output: one cast to fp16.  The pages say only "cast" (same §The Full
 *    Kernel, cast(acc, float16)); the reading taken is IEEE-754
 *    round-to-nearest-even, with overflow to ±inf.  The rounding below is
 *    written from the IEEE-754 binary16 definition (1 sign bit, 5 exponent
 *    bits with bias 15, 10 fraction bits, subnormals below 2^-14).
 *
 * Threads split the output by row blocks; each element's summation order is
 * the same whatever the thread count.
 *
 * The same product with bfloat16 operands and result (oracle_gemm_bf16_nt and
 * its helpers, at the end of this file) serves the bf16 variant of the
 * method: the sum is again a sequential fp64 sum, rounded once, to bf16.
 * oracle_gemm_f16_nt_acc16 serves the fp16-accumulation variant: the
 * accumulator is rounded to fp16 after every 16-wide k step (see dot_acc16).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- binary16 <-> binary64 from the IEEE-754 definition ---------------- */

double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int efield = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (efield == 0) {
        v = ldexp((double)frac, -24);                 /* subnormal: frac * 2^-24 */
    } else if (efield == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(frac | 0x400), efield - 25); /* 1.frac * 2^(e-15) */
    }
    return sign ? -v : v;
}

/*
 * Round a double to the nearest binary16 value, ties to the even significand.
 * For |x| in [2^E, 2^(E+1)) with E >= -14 the binary16 grid spacing is
 * 2^(E-10); below 2^-14 it is 2^-24 (subnormals).  q = |x| / spacing is exact
 * (a power-of-two scaling), r = RNE(q) is an integer in [0, 2048], and the
 * encoded value is r * spacing.
 */
uint16_t oracle_f64_to_f16(double x)
{
    if (isnan(x)) return 0x7e00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isinf(a)) return sign | 0x7c00;
    if (a == 0.0) return sign;

    int e2;
    (void)frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;               /* a in [2^E, 2^(E+1)) */
    if (E > 15) return sign | 0x7c00;
    if (E < -14) E = -14;

    double q = ldexp(a, 10 - E);  /* in [0, 2048) */
    double fl = floor(q);
    double rem = q - fl;          /* exact: q carries at most 53 significant bits */
    double r;
    if (rem > 0.5) {
        r = fl + 1.0;
    } else if (rem < 0.5) {
        r = fl;
    } else {
        r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    }
    long ri = (long)r;

    if (ri < 1024) {
        /* only possible when E == -14: a subnormal (or zero) result */
        return sign | (uint16_t)ri;
    }
    if (ri == 2048) {             /* rounded up into the next binade */
        ri = 1024;
        E += 1;
        if (E > 15) return sign | 0x7c00;
    }
    return sign | (uint16_t)(((E + 15) << 10) | (int)(ri - 1024));
}

/* ---- the GEMM ----------------------------------------------------------- */

static double g_f16_table[65536];
static pthread_once_t g_table_once = PTHREAD_ONCE_INIT;

static void build_table(void)
{
    for (uint32_t h = 0; h < 65536u; ++h) g_f16_table[h] = oracle_f16_to_f64((uint16_t)h);
}

/* The exact fp64 sum of one output element, k ascending. */
static double dot_f64(int64_t K, const uint16_t *a, const uint16_t *b)
{
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k) s += g_f16_table[a[k]] * g_f16_table[b[k]];
    return s;
}

/*
 * fp16 accumulation, the variant the pages set against fp32 accumulation
 * ("6. Register Reallocation, Multicast, and a Persistent Kernel",
 * §Shared-Memory Epilogue, the Note on an earlier version that accumulated
 * with wgmma f16.f16.f16, and its error over a K = 8192 reduction).  The pages do not say how the fp16
 * accumulator is rounded.  The reading taken: the tensor-core instruction adds
 * one 16-wide k step at a time (K = 16 for 16-bit operands), and the
 * accumulator is a binary16 value after every step:
 *
 *     acc_0 = +0,   acc_{j+1} = RNE_fp16( acc_j + sum_{k=16j}^{min(16j+16,K)-1} A[m,k]·B[n,k] ),
 *
 * C[m,n] = acc after the last step, each step's sum in fp64, k ascending.
 */
#define ORACLE_ACC16_STEP 16

static uint16_t dot_acc16(int64_t K, const uint16_t *a, const uint16_t *b)
{
    uint16_t acc = 0;
    for (int64_t k0 = 0; k0 < K; k0 += ORACLE_ACC16_STEP) {
        int64_t k1 = k0 + ORACLE_ACC16_STEP < K ? k0 + ORACLE_ACC16_STEP : K;
        double s = g_f16_table[acc];
        for (int64_t k = k0; k < k1; ++k) s += g_f16_table[a[k]] * g_f16_table[b[k]];
        acc = oracle_f64_to_f16(s);
    }
    return acc;
}

typedef struct {
    int64_t m0, m1, N, K;
    const uint16_t *A; int64_t lda;
    const uint16_t *B; int64_t ldb;
    uint16_t *C; int64_t ldc;       /* rounded output, or NULL */
    double *S; int64_t lds;         /* unrounded output, or NULL */
    int acc16;                      /* fp16 accumulation instead of one final rounding */
} rows_job;

static void *rows_worker(void *p)
{
    rows_job *j = (rows_job *)p;
    for (int64_t m = j->m0; m < j->m1; ++m) {
        for (int64_t n = 0; n < j->N; ++n) {
            if (j->acc16) {
                j->C[m * j->ldc + n] = dot_acc16(j->K, j->A + m * j->lda, j->B + n * j->ldb);
                continue;
            }
            double s = dot_f64(j->K, j->A + m * j->lda, j->B + n * j->ldb);
            if (j->C) j->C[m * j->ldc + n] = oracle_f64_to_f16(s);
            if (j->S) j->S[m * j->lds + n] = s;
        }
    }
    return NULL;
}

static void run_rows(int64_t M, int64_t N, int64_t K,
                     const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                     uint16_t *C, int64_t ldc, double *S, int64_t lds, int acc16, int nthreads)
{
    pthread_once(&g_table_once, build_table);
    if (M <= 0 || N <= 0) return;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = (int)M;
    if (nthreads > 256) nthreads = 256;
    pthread_t tid[256];
    int created[256];
    rows_job job[256];
    int64_t per = (M + nthreads - 1) / nthreads;
    int njobs = 0;
    for (int t = 0; t < nthreads; ++t) {
        int64_t m0 = t * per, m1 = m0 + per;
        if (m0 >= M) break;
        if (m1 > M) m1 = M;
        job[t] = (rows_job){m0, m1, N, K, A, lda, B, ldb, C, ldc, S, lds, acc16};
        created[t] = 0;
        njobs = t + 1;
    }
    for (int t = 1; t < njobs; ++t)
        created[t] = (pthread_create(&tid[t], NULL, rows_worker, &job[t]) == 0);
    rows_worker(&job[0]);
    for (int t = 1; t < njobs; ++t) {
        if (created[t]) pthread_join(tid[t], NULL);
        else rows_worker(&job[t]);   /* run inline if a thread could not start */
    }
}

/* C[m*ldc+n] = RNE_fp16(sum_k A[m,k]·B[n,k]) for all m < M, n < N.  Entries of
 * C outside that M×N window (columns N..ldc-1) are not touched. */
void oracle_gemm_f16_nt(int64_t M, int64_t N, int64_t K,
                        const uint16_t *A, int64_t lda,
                        const uint16_t *B, int64_t ldb,
                        uint16_t *C, int64_t ldc, int nthreads)
{
    run_rows(M, N, K, A, lda, B, ldb, C, ldc, NULL, 0, 0, nthreads);
}

/* The same sums before the final rounding, S[m*lds+n] (fp64). */
void oracle_gemm_f16_nt_f64(int64_t M, int64_t N, int64_t K,
                            const uint16_t *A, int64_t lda,
                            const uint16_t *B, int64_t ldb,
                            double *S, int64_t lds, int nthreads)
{
    run_rows(M, N, K, A, lda, B, ldb, NULL, 0, S, lds, 0, nthreads);
}

/* Selected elements only: out[i] = C_ref[rows[i], cols[i]], one by one.  For
 * full-size problems whose whole product is too slow on the host. */
void oracle_gemm_f16_nt_points(int64_t K,
                               const uint16_t *A, int64_t lda,
                               const uint16_t *B, int64_t ldb,
                               int64_t npts, const int64_t *rows, const int64_t *cols,
                               uint16_t *out, double *out_f64)
{
    pthread_once(&g_table_once, build_table);
    for (int64_t i = 0; i < npts; ++i) {
        double s = dot_f64(K, A + rows[i] * lda, B + cols[i] * ldb);
        if (out) out[i] = oracle_f64_to_f16(s);
        if (out_f64) out_f64[i] = s;
    }
}

/* C[m*ldc+n] = acc after the last 16-wide step of the fp16-accumulation
 * recurrence above, for all m < M, n < N. */
void oracle_gemm_f16_nt_acc16(int64_t M, int64_t N, int64_t K,
                              const uint16_t *A, int64_t lda,
                              const uint16_t *B, int64_t ldb,
                              uint16_t *C, int64_t ldc, int nthreads)
{
    run_rows(M, N, K, A, lda, B, ldb, C, ldc, NULL, 0, 1, nthreads);
}

/* Selected elements of the fp16-accumulation variant, one by one. */
void oracle_gemm_f16_nt_acc16_points(int64_t K,
                                     const uint16_t *A, int64_t lda,
                                     const uint16_t *B, int64_t ldb,
                                     int64_t npts, const int64_t *rows, const int64_t *cols,
                                     uint16_t *out)
{
    pthread_once(&g_table_once, build_table);
    for (int64_t i = 0; i < npts; ++i) out[i] = dot_acc16(K, A + rows[i] * lda, B + cols[i] * ldb);
}

/* Vectorised conversions for the tests. */
void oracle_f64_to_f16_array(int64_t n, const double *x, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_f16(x[i]);
}

void oracle_f16_to_f64_array(int64_t n, const uint16_t *h, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f64(h[i]);
}

/* ---- bfloat16 (the same product with bf16 operands and result) ------------
 *
 * bfloat16: 1 sign bit, 8 exponent bits with bias 127, 7 fraction bits,
 * subnormals below 2^-126 (spacing 2^-133), largest finite (2 - 2^-7)·2^127.
 * The sum is the same sequential fp64 sum; the one final rounding is to the
 * nearest bf16, ties to the even significand, overflowing to ±inf.
 */

double oracle_bf16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int efield = (h >> 7) & 0xff;
    int frac = h & 0x7f;
    double v;
    if (efield == 0) {
        v = ldexp((double)frac, -133);                 /* subnormal: frac * 2^-133 */
    } else if (efield == 255) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(frac | 0x80), efield - 134); /* 1.frac * 2^(e-127) */
    }
    return sign ? -v : v;
}

/* For |x| in [2^E, 2^(E+1)) with E >= -126 the bf16 grid spacing is 2^(E-7);
 * below 2^-126 it is 2^-133.  q = |x| / spacing is exact, r = RNE(q) lies in
 * [0, 256], and the result is r * spacing. */
uint16_t oracle_f64_to_bf16(double x)
{
    if (isnan(x)) return 0x7fc0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isinf(a)) return sign | 0x7f80;
    if (a == 0.0) return sign;

    int e2;
    (void)frexp(a, &e2);
    int E = e2 - 1;
    if (E > 127) return sign | 0x7f80;
    if (E < -126) E = -126;

    double q = ldexp(a, 7 - E);   /* in [0, 256) */
    double fl = floor(q);
    double rem = q - fl;
    double r;
    if (rem > 0.5) {
        r = fl + 1.0;
    } else if (rem < 0.5) {
        r = fl;
    } else {
        r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    }
    long ri = (long)r;

    if (ri < 128) {
        /* only possible when E == -126: a subnormal (or zero) result */
        return sign | (uint16_t)ri;
    }
    if (ri == 256) {
        ri = 128;
        E += 1;
        if (E > 127) return sign | 0x7f80;
    }
    return sign | (uint16_t)(((E + 127) << 7) | (int)(ri - 128));
}

static double g_bf16_table[65536];
static pthread_once_t g_bf16_once = PTHREAD_ONCE_INIT;

static void build_bf16_table(void)
{
    for (uint32_t h = 0; h < 65536u; ++h) g_bf16_table[h] = oracle_bf16_to_f64((uint16_t)h);
}

static double dot_bf16(int64_t K, const uint16_t *a, const uint16_t *b)
{
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k) s += g_bf16_table[a[k]] * g_bf16_table[b[k]];
    return s;
}

typedef struct {
    int64_t m0, m1, N, K;
    const uint16_t *A; int64_t lda;
    const uint16_t *B; int64_t ldb;
    uint16_t *C; int64_t ldc;
} bf16_job;

static void *bf16_worker(void *p)
{
    bf16_job *j = (bf16_job *)p;
    for (int64_t m = j->m0; m < j->m1; ++m)
        for (int64_t n = 0; n < j->N; ++n)
            j->C[m * j->ldc + n] = oracle_f64_to_bf16(dot_bf16(j->K, j->A + m * j->lda, j->B + n * j->ldb));
    return NULL;
}

/* C[m*ldc+n] = RNE_bf16(sum_k A[m,k]·B[n,k]) for all m < M, n < N (bf16 bit
 * patterns in and out). */
void oracle_gemm_bf16_nt(int64_t M, int64_t N, int64_t K,
                         const uint16_t *A, int64_t lda,
                         const uint16_t *B, int64_t ldb,
                         uint16_t *C, int64_t ldc, int nthreads)
{
    pthread_once(&g_bf16_once, build_bf16_table);
    if (M <= 0 || N <= 0) return;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > M) nthreads = (int)M;
    if (nthreads > 256) nthreads = 256;
    pthread_t tid[256];
    int created[256];
    bf16_job job[256];
    int64_t per = (M + nthreads - 1) / nthreads;
    int njobs = 0;
    for (int t = 0; t < nthreads; ++t) {
        int64_t m0 = t * per, m1 = m0 + per;
        if (m0 >= M) break;
        if (m1 > M) m1 = M;
        job[t] = (bf16_job){m0, m1, N, K, A, lda, B, ldb, C, ldc};
        created[t] = 0;
        njobs = t + 1;
    }
    for (int t = 1; t < njobs; ++t)
        created[t] = (pthread_create(&tid[t], NULL, bf16_worker, &job[t]) == 0);
    bf16_worker(&job[0]);
    for (int t = 1; t < njobs; ++t) {
        if (created[t]) pthread_join(tid[t], NULL);
        else bf16_worker(&job[t]);
    }
}

/* Selected elements, one by one (bf16). */
void oracle_gemm_bf16_nt_points(int64_t K,
                                const uint16_t *A, int64_t lda,
                                const uint16_t *B, int64_t ldb,
                                int64_t npts, const int64_t *rows, const int64_t *cols,
                                uint16_t *out)
{
    pthread_once(&g_bf16_once, build_bf16_table);
    for (int64_t i = 0; i < npts; ++i)
        out[i] = oracle_f64_to_bf16(dot_bf16(K, A + rows[i] * lda, B + cols[i] * ldb));
}

void oracle_f64_to_bf16_array(int64_t n, const double *x, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_bf16(x[i]);
}

void oracle_bf16_to_f64_array(int64_t n, const uint16_t *h, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f64(h[i]);
}
