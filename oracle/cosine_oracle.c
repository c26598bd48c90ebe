/*
 * CPU oracle for exact bulk cosine similarity over CSR sparse embeddings.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  The CUDA library
 * shares no code, header, table or helper with it.
 *
 * What it computes follows the blog post "Engineering practice for bulk
 * similarity calculation over sparse embeddings":
 *   - section 3.1, cosine definition: cos(u, v) = u.v / (|u|_2 |v|_2);
 *   - section 3.1, sparse dot product: u.v is summed only over the indices
 *     present in both supports, supp(u) and supp(v);
 *   - section 3.1, two-pointer merge: walk both ascending index lists at once
 *     and multiply-add only where the two indices are equal;
 *   - section 5.2 ("detail one"), norms: square and sum only the stored
 *     nonzeros of a row, then take the square root;
 *   - section 2.3: the result is the full (n_query x n_item) float32 matrix.
 *
 * Precision: every product and sum is taken in double (a product of two
 * floats is exact in double), the norms are double, and the cosine
 * acc / (|q| |v|) is rounded once to float (round to nearest even).
 *
 * Readings where the post is silent (each is listed with the design notes):
 *   - a row with no nonzeros (or all-zero values) has norm 0, and every cosine
 *     that involves it is 0, never NaN;
 *   - indices must be strictly increasing within a row (the merge's
 *     precondition); oracle_check_csr reports rows that break it;
 *   - no clamp to [-1, 1] is applied.
 *
 * Build: gcc -O2 -std=c11 -pthread -shared -fPIC (no -ffast-math: the double
 * arithmetic must stay IEEE).
 *
 * A mutant build (-DORACLE_MUTANT=k, k > 0) plants one deliberate mistake so
 * that the pin tests can show that they catch it; k = 0 is the oracle.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* Sparse dot product of two sorted index lists by the two-pointer merge. */
static double merge_dot(const int32_t *ia, const float *va, int64_t na,
                        const int32_t *ib, const float *vb, int64_t nb) {
  double acc = 0.0;
  int64_t a = 0, b = 0;
  while (a < na && b < nb) {
    int32_t ka = ia[a], kb = ib[b];
    if (ka < kb) {
      ++a;
    } else if (ka > kb) {
      ++b;
    } else {
#if ORACLE_MUTANT == 1 /* mutant: drops the last shared index of each pair */
      if (a + 1 == na || b + 1 == nb) { ++a; ++b; continue; }
#endif
#if ORACLE_MUTANT == 2 /* mutant: wrong sign on one operand */
      acc -= (double)va[a] * (double)vb[b];
#else
      acc += (double)va[a] * (double)vb[b];
#endif
      ++a;
      ++b;
    }
#if ORACLE_MUTANT == 3 /* mutant: advances both lists on any mismatch */
    if (ka != kb) { a += (ka > kb); b += (ka < kb); }
#endif
  }
  return acc;
}

/* Euclidean norm of one row over its stored values, in double. */
static double row_norm(const float *v, int64_t n) {
  double s = 0.0;
  for (int64_t j = 0; j < n; ++j) s += (double)v[j] * (double)v[j];
#if ORACLE_MUTANT == 4 /* mutant: forgets the square root */
  return s;
#else
  return sqrt(s);
#endif
}

/* norms[r] = sqrt(sum_j values[j]^2) over row r's stored values. */
int oracle_row_norms(int64_t n_rows, const int64_t *indptr, const float *values,
                     double *norms) {
  if (n_rows < 0 || (n_rows > 0 && (!indptr || !norms))) return 1;
  for (int64_t r = 0; r < n_rows; ++r)
    norms[r] = row_norm(values + indptr[r], indptr[r + 1] - indptr[r]);
  return 0;
}

/* Returns the first row that breaks the CSR rules (indptr non-decreasing,
 * indices strictly increasing and in [0, dim)), or -1 when all rows are valid. */
int64_t oracle_check_csr(int64_t n_rows, const int64_t *indptr, const int32_t *indices,
                         int64_t dim) {
  if (n_rows > 0 && indptr[0] != 0) return 0;
  for (int64_t r = 0; r < n_rows; ++r) {
    if (indptr[r + 1] < indptr[r]) return r;
    for (int64_t j = indptr[r]; j < indptr[r + 1]; ++j) {
      if (indices[j] < 0 || indices[j] >= dim) return r;
      if (j > indptr[r] && indices[j] <= indices[j - 1]) return r;
    }
  }
  return -1;
}

typedef struct {
  const int64_t *q_indptr;
  const int32_t *q_indices;
  const float *q_values;
  const int64_t *i_indptr;
  const int32_t *i_indices;
  const float *i_values;
  const int64_t *q_rows; /* selected query rows, or NULL for 0..n_sel-1 */
  int64_t n_sel;
  int64_t i_begin, i_end;
  const double *q_norm; /* per selected query row */
  const double *i_norm; /* per item in [i_begin, i_end) */
  double *out_f64;      /* [n_sel][i_end - i_begin] or NULL */
  float *out_f32;       /* [n_sel][i_end - i_begin] or NULL */
  int64_t next;         /* next selected row to take (under lock) */
  pthread_mutex_t lock;
} cosine_job;

static void cosine_row(cosine_job *job, int64_t s) {
  int64_t q = job->q_rows ? job->q_rows[s] : s;
  const int32_t *iq = job->q_indices + job->q_indptr[q];
  const float *vq = job->q_values + job->q_indptr[q];
  int64_t nq = job->q_indptr[q + 1] - job->q_indptr[q];
  int64_t width = job->i_end - job->i_begin;
  double nrm_q = job->q_norm[s];
  for (int64_t c = 0; c < width; ++c) {
    int64_t i = job->i_begin + c;
    int64_t p0 = job->i_indptr[i];
    double dot = merge_dot(iq, vq, nq, job->i_indices + p0, job->i_values + p0,
                           job->i_indptr[i + 1] - p0);
    double den = nrm_q * job->i_norm[c];
    double cosv = (den > 0.0) ? dot / den : 0.0;
#if ORACLE_MUTANT == 5 /* mutant: divides by the query norm only */
    cosv = (nrm_q > 0.0) ? dot / nrm_q : 0.0;
#endif
#if ORACLE_MUTANT == 6 /* mutant: writes the output transposed */
    int64_t o = (width == job->n_sel) ? c * width + s : s * width + c;
#else
    int64_t o = s * width + c;
#endif
    if (job->out_f64) job->out_f64[o] = cosv;
    if (job->out_f32) job->out_f32[o] = (float)cosv;
  }
}

static void *cosine_worker(void *arg) {
  cosine_job *job = (cosine_job *)arg;
  for (;;) {
    pthread_mutex_lock(&job->lock);
    int64_t s = job->next++;
    pthread_mutex_unlock(&job->lock);
    if (s >= job->n_sel) break;
    cosine_row(job, s);
  }
  return NULL;
}

/*
 * S[s][c] = cos(Q[q_rows[s]], I[i_begin + c]) for s < n_sel, c < i_end - i_begin.
 * q_rows may be NULL (then rows 0..n_sel-1).  Either output may be NULL.
 * Returns 0 on success, nonzero on a bad argument or an allocation failure.
 */
int oracle_cosine(const int64_t *q_indptr, const int32_t *q_indices, const float *q_values,
                  int64_t n_q, const int64_t *i_indptr, const int32_t *i_indices,
                  const float *i_values, int64_t n_i, const int64_t *q_rows, int64_t n_sel,
                  int64_t i_begin, int64_t i_end, double *out_f64, float *out_f32,
                  int n_threads) {
  if (n_sel < 0 || i_begin < 0 || i_end < i_begin || i_end > n_i) return 1;
  if (!q_rows && n_sel > n_q) return 1;
  for (int64_t s = 0; q_rows && s < n_sel; ++s)
    if (q_rows[s] < 0 || q_rows[s] >= n_q) return 1;
  int64_t width = i_end - i_begin;
  if (n_sel == 0 || width == 0) return 0;
  double *q_norm = (double *)malloc(sizeof(double) * (size_t)n_sel);
  double *i_norm = (double *)malloc(sizeof(double) * (size_t)width);
  if (!q_norm || !i_norm) {
    free(q_norm);
    free(i_norm);
    return 2;
  }
  for (int64_t s = 0; s < n_sel; ++s) {
    int64_t q = q_rows ? q_rows[s] : s;
    q_norm[s] = row_norm(q_values + q_indptr[q], q_indptr[q + 1] - q_indptr[q]);
  }
  for (int64_t c = 0; c < width; ++c) {
    int64_t i = i_begin + c;
    i_norm[c] = row_norm(i_values + i_indptr[i], i_indptr[i + 1] - i_indptr[i]);
  }
  cosine_job job = {q_indptr, q_indices, q_values, i_indptr, i_indices, i_values, q_rows,
                    n_sel,    i_begin,   i_end,    q_norm,   i_norm,    out_f64,  out_f32, 0};
  pthread_mutex_init(&job.lock, NULL);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 1024) n_threads = 1024;
  if ((int64_t)n_threads > n_sel) n_threads = (int)n_sel;
  if (n_threads == 1) {
    cosine_worker(&job);
  } else {
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    int started = 0;
    if (tid)
      for (; started < n_threads; ++started)
        if (pthread_create(&tid[started], NULL, cosine_worker, &job) != 0) break;
    if (started == 0) cosine_worker(&job);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    free(tid);
  }
  pthread_mutex_destroy(&job.lock);
  free(q_norm);
  free(i_norm);
  return 0;
}

/* Unnormalised sparse dot products D[s][c] = Q[q_rows[s]] . I[i_begin + c]. */
int oracle_dot(const int64_t *q_indptr, const int32_t *q_indices, const float *q_values,
               int64_t n_q, const int64_t *i_indptr, const int32_t *i_indices,
               const float *i_values, int64_t n_i, const int64_t *q_rows, int64_t n_sel,
               int64_t i_begin, int64_t i_end, double *out) {
  if (n_sel < 0 || i_begin < 0 || i_end < i_begin || i_end > n_i || !out) return 1;
  int64_t width = i_end - i_begin;
  for (int64_t s = 0; s < n_sel; ++s) {
    int64_t q = q_rows ? q_rows[s] : s;
    if (q < 0 || q >= n_q) return 1;
    for (int64_t c = 0; c < width; ++c) {
      int64_t i = i_begin + c;
      out[s * width + c] =
          merge_dot(q_indices + q_indptr[q], q_values + q_indptr[q], q_indptr[q + 1] - q_indptr[q],
                    i_indices + i_indptr[i], i_values + i_indptr[i], i_indptr[i + 1] - i_indptr[i]);
    }
  }
  return 0;
}

int oracle_mutant_id(void) { return ORACLE_MUTANT; }
