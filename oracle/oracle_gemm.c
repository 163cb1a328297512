/*
 * CPU oracle for single-precision dense matrix multiply.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; it shares no header, helper, constant or build flag with the
 * CUDA path.  Only the test suite, the smoke check and the benchmark's CPU
 * baseline leg load it.
 *
 * What it computes is the plain definition of the product, nothing more:
 *
 *     C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j]
 *
 * as stated in "Hardware acceleration: optimising the memory access pattern of
 * CUDA kernels for matrix multiply", section "computational characteristics of
 * matrix multiplication" (the C_{i,j} summation equation), with the row-major
 * indexing A[row*K+k], B[k*N+col], C[row*N+col] of that page's basic kernel
 * listing, generalised to leading dimensions lda/ldb/ldc.  The CPU reference of
 * "[infra] 03: writing CUDA kernels, from vector add to matrix multiply"
 * (matMulCPU, experiments 2-4) sums over k in ascending order for each (i,j);
 * this oracle keeps exactly that per-element summation order and changes only
 * the accumulator from float to double.
 *
 * Why double: the product of two binary32 values is exact in binary64
 * (24 + 24 significant bits < 53), so the only rounding left is in the K-term
 * double sum, at least 2^29 times finer than any float32 result.
 *
 * Alongside C the oracle returns bound[i][j] = sum_k |A[i][k]| * |B[k][j]|,
 * the scale against which a float32 result is judged.
 *
 * Loop order is i -> k -> j with a double row accumulator; for every (i,j) the
 * k-terms still enter in ascending k, so the result is bit-identical to the
 * i -> j -> k triple loop (a test checks this).  Rows are split over POSIX
 * threads; each thread owns whole rows, so the threading changes no sum.
 *
 * The general form (oracle_gemm_general_f64) computes the BLAS-style
 *
 *     C_out[i][j] = alpha * sum_k op(A)[i][k] * op(B)[k][j] + beta * C_in[i][j]
 *
 * where op(X) is X or its transpose (row-major storage: op(A)[i][k] is
 * A[k][i] when A is stored transposed, K x M), and C_in is not read when
 * beta == 0 (so NaN or uninitialised memory there has no effect).  The pages
 * define only the plain product; scaling, accumulation into C and transposed
 * storage are the standard GEMM interface (the "Column-major" remark of the
 * optimisation-summary page is the pages' only mention of another layout).
 * The k sum is formed exactly as for the plain product (ascending k, double
 * accumulator, exact float products); then alpha * sum + beta * C_in in
 * double.  Its bound is |alpha| * sum_k |a||b| + |beta| * |C_in|.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -fPIC -shared -pthread
 * (no contraction into fused multiply-add, no reassociation).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t N, K;
    const float *A;
    int64_t lda;
    const float *B;
    int64_t ldb;
    double *C;          /* nrows x ldc */
    int64_t ldc;
    double *bound;      /* nrows x ldbound, may be NULL */
    int64_t ldbound;
    const int64_t *rows; /* row indices into A; NULL = 0..nrows-1 */
    int64_t row_begin, row_end; /* range of output rows this worker owns */
    /* general form only (general != 0) */
    int general, transa, transb;
    float alpha, beta;
    const float *Cin;
    int64_t ldcin;
} oracle_job;

/* One output row: C[r][:] = sum_k A[i][k] * B[k][:], k ascending. */
static void oracle_one_row(const oracle_job *jb, int64_t r)
{
    const int64_t i = jb->rows ? jb->rows[r] : r;
    double *crow = jb->C + r * jb->ldc;
    double *brow = jb->bound ? jb->bound + r * jb->ldbound : NULL;
    for (int64_t j = 0; j < jb->N; ++j) crow[j] = 0.0;
    if (brow)
        for (int64_t j = 0; j < jb->N; ++j) brow[j] = 0.0;
    const float *arow = jb->A + i * jb->lda;
    for (int64_t k = 0; k < jb->K; ++k) {
        const double a = (double)arow[k];
        const float *bk = jb->B + k * jb->ldb;
        for (int64_t j = 0; j < jb->N; ++j) crow[j] += a * (double)bk[j];
        if (brow) {
            const double aa = fabs(a);
            for (int64_t j = 0; j < jb->N; ++j) brow[j] += aa * fabs((double)bk[j]);
        }
    }
}

/* One output row of the general form.  op(A)[i][k] and op(B)[k][j] are read
 * through the storage order of each operand; k ascending as above. */
static void oracle_general_row(const oracle_job *jb, int64_t r)
{
    const int64_t i = jb->rows ? jb->rows[r] : r;
    double *out = jb->C + r * jb->ldc;
    double *bnd = jb->bound ? jb->bound + r * jb->ldbound : NULL;
    for (int64_t j = 0; j < jb->N; ++j) {
        out[j] = 0.0;
        if (bnd) bnd[j] = 0.0;
    }
    for (int64_t k = 0; k < jb->K; ++k) {
        const double aik = (double)(jb->transa ? jb->A[k * jb->lda + i] : jb->A[i * jb->lda + k]);
        for (int64_t j = 0; j < jb->N; ++j) {
            const double bkj = (double)(jb->transb ? jb->B[j * jb->ldb + k] : jb->B[k * jb->ldb + j]);
            out[j] += aik * bkj;
            if (bnd) bnd[j] += fabs(aik) * fabs(bkj);
        }
    }
    const double alpha = (double)jb->alpha, beta = (double)jb->beta;
    for (int64_t j = 0; j < jb->N; ++j) {
        double v = alpha * out[j];
        double vb = bnd ? fabs(alpha) * bnd[j] : 0.0;
        if (jb->beta != 0.0f) { /* beta == 0: C_in is not read */
            const double c = (double)jb->Cin[i * jb->ldcin + j];
            v += beta * c;
            vb += fabs(beta) * fabs(c);
        }
        out[j] = v;
        if (bnd) bnd[j] = vb;
    }
}

static void *oracle_worker(void *arg)
{
    const oracle_job *jb = (const oracle_job *)arg;
    for (int64_t r = jb->row_begin; r < jb->row_end; ++r) {
        if (jb->general)
            oracle_general_row(jb, r);
        else
            oracle_one_row(jb, r);
    }
    return NULL;
}

static int oracle_run(oracle_job base, int64_t nrows, int threads)
{
    if (nrows <= 0) return 0;
    if (threads < 1) threads = 1;
    if (threads > nrows) threads = (int)nrows;
    if (threads == 1) {
        base.row_begin = 0;
        base.row_end = nrows;
        oracle_worker(&base);
        return 0;
    }
    pthread_t *tid = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    oracle_job *jobs = (oracle_job *)calloc((size_t)threads, sizeof(oracle_job));
    if (!tid || !jobs) {
        free(tid);
        free(jobs);
        return -2;
    }
    int started = 0;
    for (int t = 0; t < threads; ++t) {
        jobs[t] = base;
        jobs[t].row_begin = nrows * t / threads;
        jobs[t].row_end = nrows * (t + 1) / threads;
        if (pthread_create(&tid[t], NULL, oracle_worker, &jobs[t]) != 0) {
            /* fall back to running this share on the calling thread */
            oracle_worker(&jobs[t]);
            tid[t] = 0;
            continue;
        }
        ++started;
    }
    for (int t = 0; t < threads; ++t)
        if (tid[t]) pthread_join(tid[t], NULL);
    (void)started;
    free(tid);
    free(jobs);
    return 0;
}

static int oracle_check_dims(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                             const float *B, int64_t ldb)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (lda < K || ldb < N) return -1;
    if (M > 0 && K > 0 && !A) return -1;
    if (K > 0 && N > 0 && !B) return -1;
    return 0;
}

/*
 * Full product.  C (M x ldc doubles) receives the exact-product, double-summed
 * result; bound (M x ldbound, may be NULL) receives sum_k |a||b|.
 * Returns 0 on success, -1 on invalid arguments, -2 if out of host memory.
 */
int oracle_sgemm_f64(int64_t M, int64_t N, int64_t K,
                     const float *A, int64_t lda,
                     const float *B, int64_t ldb,
                     double *C, int64_t ldc,
                     double *bound, int64_t ldbound,
                     int threads)
{
    if (oracle_check_dims(M, N, K, A, lda, B, ldb)) return -1;
    if (ldc < N || (M > 0 && N > 0 && !C)) return -1;
    if (bound && ldbound < N) return -1;
    oracle_job jb;
    memset(&jb, 0, sizeof(jb));
    jb.N = N; jb.K = K; jb.A = A; jb.lda = lda; jb.B = B; jb.ldb = ldb;
    jb.C = C; jb.ldc = ldc; jb.bound = bound; jb.ldbound = ldbound; jb.rows = NULL;
    return oracle_run(jb, M, threads);
}

/*
 * Selected rows only: row r of the output (nrows x N, dense) is row rows[r] of
 * the full product.  Used to check large products on a sample of whole rows.
 */
int oracle_sgemm_rows_f64(int64_t M, int64_t N, int64_t K,
                          const float *A, int64_t lda,
                          const float *B, int64_t ldb,
                          const int64_t *rows, int64_t nrows,
                          double *C, double *bound, int threads)
{
    if (oracle_check_dims(M, N, K, A, lda, B, ldb)) return -1;
    if (nrows < 0 || (nrows > 0 && (!rows || !C))) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return -1;
    oracle_job jb;
    memset(&jb, 0, sizeof(jb));
    jb.N = N; jb.K = K; jb.A = A; jb.lda = lda; jb.B = B; jb.ldb = ldb;
    jb.C = C; jb.ldc = N; jb.bound = bound; jb.ldbound = N; jb.rows = rows;
    return oracle_run(jb, nrows, threads);
}

/*
 * Single entries, one by one: c[t] = C[ii[t]][jj[t]], summed over ascending k
 * exactly as above.  Used for spot checks (corners, tile edges) of products
 * too large to recompute whole.
 */
int oracle_sgemm_entries_f64(int64_t M, int64_t N, int64_t K,
                             const float *A, int64_t lda,
                             const float *B, int64_t ldb,
                             const int64_t *ii, const int64_t *jj, int64_t n,
                             double *c, double *bound)
{
    if (oracle_check_dims(M, N, K, A, lda, B, ldb)) return -1;
    if (n < 0 || (n > 0 && (!ii || !jj || !c))) return -1;
    for (int64_t t = 0; t < n; ++t) {
        const int64_t i = ii[t], j = jj[t];
        if (i < 0 || i >= M || j < 0 || j >= N) return -1;
        double s = 0.0, sb = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = (double)A[i * lda + k];
            const double b = (double)B[k * ldb + j];
            s += a * b;
            sb += fabs(a) * fabs(b);
        }
        c[t] = s;
        if (bound) bound[t] = sb;
    }
    return 0;
}

/*
 * General form, C_out = alpha * op(A) op(B) + beta * C_in (see the header).
 * op(A) is M x K: A is stored M x K (lda >= K), or K x M (lda >= M) when
 * transa != 0.  op(B) is K x N: B is stored K x N (ldb >= N), or N x K
 * (ldb >= K) when transb != 0.  C_in is M x N with ldcin >= N (read only when
 * beta != 0).  With rows != NULL, output row r (C, bound: nrows x ldc /
 * ldbound) is row rows[r] of the result; with rows == NULL, nrows must be M.
 */
int oracle_gemm_general_f64(int transa, int transb, int64_t M, int64_t N, int64_t K,
                            float alpha,
                            const float *A, int64_t lda,
                            const float *B, int64_t ldb,
                            float beta,
                            const float *Cin, int64_t ldcin,
                            const int64_t *rows, int64_t nrows,
                            double *C, int64_t ldc,
                            double *bound, int64_t ldbound,
                            int threads)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
    if (lda < (transa ? M : K) || ldb < (transb ? K : N)) return -1;
    if (M > 0 && K > 0 && !A) return -1;
    if (K > 0 && N > 0 && !B) return -1;
    if (beta != 0.0f && M > 0 && N > 0 && (!Cin || ldcin < N)) return -1;
    if (ldc < N || (nrows > 0 && N > 0 && !C)) return -1;
    if (bound && ldbound < N) return -1;
    if (!rows && nrows != M) return -1;
    if (rows)
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= M) return -1;
    oracle_job jb;
    memset(&jb, 0, sizeof(jb));
    jb.N = N; jb.K = K; jb.A = A; jb.lda = lda; jb.B = B; jb.ldb = ldb;
    jb.C = C; jb.ldc = ldc; jb.bound = bound; jb.ldbound = ldbound; jb.rows = rows;
    jb.general = 1; jb.transa = transa != 0; jb.transb = transb != 0;
    jb.alpha = alpha; jb.beta = beta; jb.Cin = Cin; jb.ldcin = ldcin;
    return oracle_run(jb, nrows, threads);
}
