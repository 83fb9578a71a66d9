/*
 * Plain CPU oracle for the fp32 GEMM  C = alpha * A * B + beta * C_old.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (the definition, written out):
 *   C_ref[i][j] = alpha * sum_{k=0}^{K-1} A[i][k] * B[k][j] + beta * C_old[i][j]
 * for 0 <= i < M, 0 <= j < N, with every matrix row-major:
 *   A[i][k] = A[i*lda + k],  B[k][j] = B[k*ldb + j],  C[i][j] = C[i*ldc + j].
 * Source: the `matmul` kernel listing of the "@cluster" attribute page
 * (phobos-lang.dev, "What the cluster compiler accepts": acc summed over the
 * K loop, then C = alpha * acc + beta * c_old) and the "Matrix Multiplication"
 * section of "Show HN: Phobos - A tiny scale-free kernel language with tile-DAG
 * support" (C = alpha A B + beta C, A is M x K, B is K x N).
 *
 * Arithmetic: every fp32 input is widened to double.  A product of two fp32
 * values is exact in double (24 + 24 significant bits <= 53), so the only
 * rounding is the double-precision running sum, taken over k in ascending
 * order; the result is deterministic and independent of the thread count.
 *
 * Beside the value the oracle returns the error scale of each entry,
 *   den[i][j] = |alpha| * sum_k |A[i][k]| * |B[k][j]| + |beta| * |C_old[i][j]|,
 * against which the GPU result is judged (max |C - C_ref| / den).
 *
 * beta == 0 means C_old is not read (the init leaf of the cluster split
 * "zeroes the output super-tile, or scales it by beta"; read as the BLAS rule),
 * so a NaN in C_old with beta == 0 does not reach the result.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared -pthread (no fast-math; the
 * contraction switch keeps alpha*s + beta*c two roundings on every host).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARGS 1
#define ORACLE_ERR_NOMEM 2

/* ---------------------------------------------------------------- full mode */

typedef struct {
  int64_t M, N, K;
  double alpha, beta;
  const float *A, *B, *C_old;
  int64_t lda, ldb, ldc;
  double *ref, *den; /* M x N, row-major, leading dimension N */
  int64_t row_begin, row_end;
  int status;
} full_job_t;

/* One output row i: s[j] = sum_k A[i][k] B[k][j], a[j] = sum_k |A[i][k]||B[k][j]|. */
static void *full_rows(void *arg) {
  full_job_t *job = (full_job_t *)arg;
  const int64_t N = job->N, K = job->K;
  double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
  double *a = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
  if (!s || !a) {
    free(s);
    free(a);
    job->status = ORACLE_ERR_NOMEM;
    return NULL;
  }
  for (int64_t i = job->row_begin; i < job->row_end; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      s[j] = 0.0;
      a[j] = 0.0;
    }
    for (int64_t k = 0; k < K; ++k) {
      const double aik = (double)job->A[i * job->lda + k];
      const double abs_aik = fabs(aik);
      const float *brow = job->B + k * job->ldb;
      for (int64_t j = 0; j < N; ++j) {
        const double bkj = (double)brow[j];
        s[j] += aik * bkj;
        a[j] += abs_aik * fabs(bkj);
      }
    }
    for (int64_t j = 0; j < N; ++j) {
      double value = job->alpha * s[j];
      double scale = fabs(job->alpha) * a[j];
      if (job->beta != 0.0) {
        const double c = (double)job->C_old[i * job->ldc + j];
        value += job->beta * c;
        scale += fabs(job->beta) * fabs(c);
      }
      job->ref[i * N + j] = value;
      if (job->den) job->den[i * N + j] = scale;
    }
  }
  free(s);
  free(a);
  job->status = ORACLE_OK;
  return NULL;
}

static int check_args(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                      int64_t ldc, const float *A, const float *B,
                      const float *C_old, double beta) {
  if (M < 0 || N < 0 || K < 0) return ORACLE_ERR_ARGS;
  if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
    return ORACLE_ERR_ARGS;
  if (M > 0 && K > 0 && !A) return ORACLE_ERR_ARGS;
  if (K > 0 && N > 0 && !B) return ORACLE_ERR_ARGS;
  if (beta != 0.0 && M > 0 && N > 0 && !C_old) return ORACLE_ERR_ARGS;
  return ORACLE_OK;
}

/*
 * Full oracle.  ref (and den, if not NULL) are caller-owned M x N double arrays
 * with leading dimension N.  nthreads <= 0 means one thread.  Returns 0 on
 * success, 1 on bad arguments, 2 when a row buffer cannot be allocated.
 */
int oracle_sgemm(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                 int64_t lda, const float *B, int64_t ldb, float beta,
                 const float *C_old, int64_t ldc, double *ref, double *den,
                 int nthreads) {
  int st = check_args(M, N, K, lda, ldb, ldc, A, B, C_old, (double)beta);
  if (st != ORACLE_OK) return st;
  if (M == 0 || N == 0) return ORACLE_OK;
  if (!ref) return ORACLE_ERR_ARGS;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > M) nthreads = (int)M;

  full_job_t *jobs = (full_job_t *)calloc((size_t)nthreads, sizeof(full_job_t));
  pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !tids) {
    free(jobs);
    free(tids);
    return ORACLE_ERR_NOMEM;
  }
  int64_t per = M / nthreads, extra = M % nthreads, row = 0;
  for (int t = 0; t < nthreads; ++t) {
    full_job_t *j = &jobs[t];
    j->M = M; j->N = N; j->K = K;
    j->alpha = (double)alpha; j->beta = (double)beta;
    j->A = A; j->B = B; j->C_old = C_old;
    j->lda = lda; j->ldb = ldb; j->ldc = ldc;
    j->ref = ref; j->den = den;
    j->row_begin = row;
    row += per + (t < extra ? 1 : 0);
    j->row_end = row;
  }
  int spawned = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&tids[t], NULL, full_rows, &jobs[t]) != 0) break;
    spawned = t;
  }
  /* rows of threads that failed to spawn run here, in order */
  full_rows(&jobs[0]);
  for (int t = spawned + 1; t < nthreads; ++t) full_rows(&jobs[t]);
  for (int t = 1; t <= spawned; ++t) pthread_join(tids[t], NULL);
  st = ORACLE_OK;
  for (int t = 0; t < nthreads; ++t)
    if (jobs[t].status != ORACLE_OK) st = jobs[t].status;
  free(jobs);
  free(tids);
  return st;
}

/* ------------------------------------------------------------- sampled mode */

typedef struct {
  int64_t K;
  double alpha, beta;
  const float *A, *B, *C_old;
  int64_t lda, ldb, ldc;
  const int64_t *rows, *cols;
  double *ref, *den;
  int64_t begin, end;
} entry_job_t;

/* The same sum as full mode for one (i, j), k ascending: bit-identical. */
static void *entry_range(void *arg) {
  entry_job_t *job = (entry_job_t *)arg;
  for (int64_t e = job->begin; e < job->end; ++e) {
    const int64_t i = job->rows[e], j = job->cols[e];
    double s = 0.0, a = 0.0;
    for (int64_t k = 0; k < job->K; ++k) {
      const double aik = (double)job->A[i * job->lda + k];
      const double bkj = (double)job->B[k * job->ldb + j];
      s += aik * bkj;
      a += fabs(aik) * fabs(bkj);
    }
    double value = job->alpha * s;
    double scale = fabs(job->alpha) * a;
    if (job->beta != 0.0) {
      const double c = (double)job->C_old[i * job->ldc + j];
      value += job->beta * c;
      scale += fabs(job->beta) * fabs(c);
    }
    job->ref[e] = value;
    if (job->den) job->den[e] = scale;
  }
  return NULL;
}

/*
 * Sampled oracle: entries (rows[e], cols[e]) for e < count, written to ref[e]
 * (and den[e] if not NULL).  Indices outside [0,M) x [0,N) are an argument error.
 */
int oracle_sgemm_entries(int64_t M, int64_t N, int64_t K, float alpha,
                         const float *A, int64_t lda, const float *B,
                         int64_t ldb, float beta, const float *C_old,
                         int64_t ldc, const int64_t *rows, const int64_t *cols,
                         int64_t count, double *ref, double *den, int nthreads) {
  int st = check_args(M, N, K, lda, ldb, ldc, A, B, C_old, (double)beta);
  if (st != ORACLE_OK) return st;
  if (count < 0) return ORACLE_ERR_ARGS;
  if (count == 0) return ORACLE_OK;
  if (!rows || !cols || !ref) return ORACLE_ERR_ARGS;
  for (int64_t e = 0; e < count; ++e)
    if (rows[e] < 0 || rows[e] >= M || cols[e] < 0 || cols[e] >= N)
      return ORACLE_ERR_ARGS;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > count) nthreads = (int)count;

  entry_job_t *jobs = (entry_job_t *)calloc((size_t)nthreads, sizeof(entry_job_t));
  pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !tids) {
    free(jobs);
    free(tids);
    return ORACLE_ERR_NOMEM;
  }
  int64_t per = count / nthreads, extra = count % nthreads, at = 0;
  for (int t = 0; t < nthreads; ++t) {
    entry_job_t *j = &jobs[t];
    j->K = K;
    j->alpha = (double)alpha; j->beta = (double)beta;
    j->A = A; j->B = B; j->C_old = C_old;
    j->lda = lda; j->ldb = ldb; j->ldc = ldc;
    j->rows = rows; j->cols = cols; j->ref = ref; j->den = den;
    j->begin = at;
    at += per + (t < extra ? 1 : 0);
    j->end = at;
  }
  int spawned = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&tids[t], NULL, entry_range, &jobs[t]) != 0) break;
    spawned = t;
  }
  entry_range(&jobs[0]);
  for (int t = spawned + 1; t < nthreads; ++t) entry_range(&jobs[t]);
  for (int t = 1; t <= spawned; ++t) pthread_join(tids[t], NULL);
  free(jobs);
  free(tids);
  return ORACLE_OK;
}
