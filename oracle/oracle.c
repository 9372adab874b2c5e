/*
 * CPU oracle for the W4A16 mixed-precision GEMM.  TEST INFRASTRUCTURE ONLY:
 * the tests, the smoke check and the benchmark's CPU-baseline leg call it;
 * the product path never does.
 *
 * What it computes (plain definition, fp64, no blocking or reordering):
 *
 *   dequant(w)[k][n] = (q[k][n] - z[k/g][n]) * s[k/g][n]
 *     -- the dequantisation rule of "LMDeploy Guide: Fast Mixed-Precision
 *        LLM Inference Engine", section 3 "Instruction-Level Parallelism (ILP)
 *        for Zero-Overhead Dequantization": the 4-bit code less its zero
 *        point, times its scale.  One scale (and one zero) serves a group of
 *        g consecutive weights along K ("LMDeploy, in depth", section
 *        "Quantization: AWQ weights and KV cache": 4-bit groups of 128, one
 *        scale each).
 *
 *   Y[m][n] = sum_{k=0}^{K-1} X[m][k] * dequant(w)[k][n]
 *     -- the mixed-precision GEMM of the same guide, "Pipeline A:
 *        Hardware-Aware GEMM"; summed in ascending k.
 *
 * fp16 inputs are read as exact values (decoded from the IEEE 754 binary16
 * bit pattern below); every product (q - z) * s is exact in fp64 and the sums
 * are fp64.  The result is fp64, never rounded to fp16.
 *
 * The oracle knows nothing of the packed weight format or of any GPU layout.
 * Threads (POSIX) split the output columns into blocks; each (m, n) sum is
 * still taken in the plain order above, so the thread count does not change
 * a single bit of the result.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* IEEE 754 binary16 -> double, from the format's definition:
 * sign bit, 5-bit biased exponent (bias 15), 10-bit fraction;
 * exponent 0 = zero/subnormal (2^-14 * f/1024), 31 = inf/NaN. */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24); /* 2^-14 * f / 2^10 */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp(1024.0 + (double)f, e - 25); /* 2^(e-15) * (1 + f/2^10) */
  }
  return sign ? -v : v;
}

/* Dequantise the whole K x N weight matrix into W (row-major, fp64). */
void oracle_dequant(const uint8_t* q, const uint8_t* z, const uint16_t* s, int K, int N, int g,
                    double* W) {
  for (int k = 0; k < K; ++k) {
    int grp = k / g;
    for (int n = 0; n < N; ++n) {
      double qv = (double)q[(size_t)k * N + n];
      double zv = (double)z[(size_t)grp * N + n];
      double sv = oracle_half_to_double(s[(size_t)grp * N + n]);
      W[(size_t)k * N + n] = (qv - zv) * sv;
    }
  }
}

typedef struct {
  const uint16_t* X;
  const uint8_t* q;
  const uint8_t* z;
  const uint16_t* s;
  int M, K, N, g;
  const int* rows;
  int nrows;
  double* Y;
  int n0, n1;
  int status;
} job_t;

static void* run_block(void* arg) {
  job_t* j = (job_t*)arg;
  int nb = j->n1 - j->n0;
  if (nb <= 0) return NULL;
  int K = j->K, N = j->N, g = j->g;
  /* Step 1: dequantise this block of columns (all k). */
  double* W = (double*)malloc(sizeof(double) * (size_t)K * nb);
  double* xrow = (double*)malloc(sizeof(double) * (size_t)K);
  if (!W || !xrow) {
    free(W);
    free(xrow);
    j->status = 1;
    return NULL;
  }
  for (int k = 0; k < K; ++k) {
    int grp = k / g;
    for (int c = 0; c < nb; ++c) {
      int n = j->n0 + c;
      double qv = (double)j->q[(size_t)k * N + n];
      double zv = (double)j->z[(size_t)grp * N + n];
      double sv = oracle_half_to_double(j->s[(size_t)grp * N + n]);
      W[(size_t)k * nb + c] = (qv - zv) * sv;
    }
  }
  /* Step 2: for every requested row m, Y[m][n] = sum over k in ascending order. */
  for (int r = 0; r < j->nrows; ++r) {
    int m = j->rows ? j->rows[r] : r;
    for (int k = 0; k < K; ++k) xrow[k] = oracle_half_to_double(j->X[(size_t)m * K + k]);
    double* y = j->Y + (size_t)r * N + j->n0;
    for (int c = 0; c < nb; ++c) y[c] = 0.0;
    for (int k = 0; k < K; ++k) {
      double xv = xrow[k];
      const double* w = W + (size_t)k * nb;
      for (int c = 0; c < nb; ++c) y[c] += xv * w[c];
    }
  }
  free(W);
  free(xrow);
  return NULL;
}

/*
 * Y[r][n] for the rows listed in `rows` (all M rows when rows == NULL, then
 * nrows must equal M).  X: fp16 bits [M][K]; q: codes [K][N] (one per byte);
 * z: codes [K/g][N]; s: fp16 bits [K/g][N]; Y: fp64 [nrows][N].
 * Returns 0 on success, 1 on allocation failure, 2 on bad arguments,
 * 3 when a code is above 15.
 */
int oracle_gemm(const uint16_t* X, const uint8_t* q, const uint8_t* z, const uint16_t* s, int M,
                int K, int N, int g, const int* rows, int nrows, double* Y, int nthreads) {
  if (M < 0 || K <= 0 || N <= 0 || g <= 0 || K % g || nrows < 0) return 2;
  if (!rows && nrows != M) return 2;
  for (int r = 0; r < nrows; ++r)
    if (rows && (rows[r] < 0 || rows[r] >= M)) return 2;
  for (size_t i = 0; i < (size_t)K * N; ++i)
    if (q[i] > 15) return 3;
  for (size_t i = 0; i < (size_t)(K / g) * N; ++i)
    if (z[i] > 15) return 3;
  if (nrows == 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > N) nthreads = N;
  job_t* jobs = (job_t*)calloc((size_t)nthreads, sizeof(job_t));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return 1;
  }
  int per = (N + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    job_t* j = &jobs[t];
    j->X = X; j->q = q; j->z = z; j->s = s;
    j->M = M; j->K = K; j->N = N; j->g = g;
    j->rows = rows; j->nrows = nrows; j->Y = Y;
    j->n0 = t * per;
    j->n1 = (t + 1) * per < N ? (t + 1) * per : N;
    j->status = 0;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, run_block, &jobs[t]);
  run_block(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  int st = 0;
  for (int t = 0; t < nthreads; ++t) st |= jobs[t].status;
  free(jobs);
  free(th);
  return st ? 1 : 0;
}
