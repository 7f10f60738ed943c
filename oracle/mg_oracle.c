/*
 * mg_oracle.c -- fp64 CPU oracle for multi-head scaled-dot-product attention,
 * forward and backward.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library. The product path (the CUDA
 * library and its Python binding) never calls, links or imports it, and it
 * shares no code, header, table or helper with that path.
 *
 * What it computes. "Meganeura: Portable GPU Training and Inference through
 * Vulkan and Metal" names attention as one graph node with its own derivative
 * rule (Section 3.1) and lowers it to three kernel archetypes: tiled attention
 * forward, dQ, and fused dK+dV (Section 3.3; Section 8 on the fused dK+dV
 * invariant). The pages print no formula for attention, so this file writes out
 * the textbook definition of scaled dot-product attention and its chain-rule
 * gradient, per head, for Q,K,V,dO of shape [L][D]:
 *
 *   s_ij   = scale * sum_d Q_id K_jd          allowed(i,j) = (j <= i) if causal
 *   LSE_i  = ln sum_{j allowed} exp(s_ij)     (natural log of the scaled logits)
 *   P_ij   = exp(s_ij - LSE_i) if allowed, else 0
 *   O_i    = sum_j P_ij V_j
 *   Dvec_i = sum_d dO_id O_id
 *   dP_ij  = sum_d dO_id V_jd
 *   dS_ij  = P_ij (dP_ij - Dvec_i)
 *   dV_j   = sum_i P_ij dO_i
 *   dQ_i   = scale * sum_j dS_ij K_j
 *   dK_j   = scale * sum_i dS_ij Q_i
 *
 * Everything is fp64. The backward stays in full precision as the pages require
 * for derivative regions (Sections 3.1 and 4.2). LSE is evaluated as
 * max + ln sum exp(s - max), which is the same number as ln sum exp(s) and does
 * not overflow. No L x L matrix is held: one query row (or one key column) of
 * scores is formed at a time, so the largest shapes fit in host memory.
 *
 * Threads: OpenMP over (head, row) pairs; results do not depend on the thread
 * count because every output element is written by exactly one loop iteration
 * with a fixed summation order.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#include <omp.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NOMEM 2

static inline int allowed(long i, long j, int causal) { return !causal || j <= i; }

static inline double dot(const double *a, const double *b, int D) {
  double acc = 0.0;
  for (int d = 0; d < D; ++d) acc += a[d] * b[d];
  return acc;
}

/* Scores of query row i against every key; masked entries are -inf.
 * Returns LSE_i. */
static double score_row(const double *q, const double *K, long L, int D,
                        int causal, long i, double scale, double *s) {
  double m = -INFINITY;
  for (long j = 0; j < L; ++j) {
    if (allowed(i, j, causal)) {
      s[j] = scale * dot(q, K + j * D, D);
      if (s[j] > m) m = s[j];
    } else {
      s[j] = -INFINITY;
    }
  }
  double sum = 0.0;
  for (long j = 0; j < L; ++j)
    if (allowed(i, j, causal)) sum += exp(s[j] - m);
  return m + log(sum);
}

static int check(long BH, long L, int D, double scale) {
  if (BH < 1 || L < 1 || D < 1) return ORACLE_ERR_ARG;
  if (!(scale > 0.0) || !isfinite(scale)) return ORACLE_ERR_ARG;
  return ORACLE_OK;
}

/* Forward over BH independent heads laid out [BH][L][D]; LSE is [BH][L]. */
int oracle_attn_fwd(const double *Q, const double *K, const double *V,
                    double *O, double *LSE, long BH, long L, int D, int causal,
                    double scale, int nthreads) {
  int rc = check(BH, L, D, scale);
  if (rc) return rc;
  if (nthreads < 1) nthreads = omp_get_max_threads();
  int failed = 0;
#pragma omp parallel num_threads(nthreads)
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)L);
    if (!s) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for collapse(2) schedule(dynamic, 8)
    for (long h = 0; h < BH; ++h) {
      for (long i = 0; i < L; ++i) {
        if (!s) continue;
        const double *Qh = Q + h * L * D, *Kh = K + h * L * D, *Vh = V + h * L * D;
        double lse = score_row(Qh + i * D, Kh, L, D, causal, i, scale, s);
        double *o = O + (h * L + i) * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (long j = 0; j < L; ++j) {
          if (!allowed(i, j, causal)) continue;
          double p = exp(s[j] - lse);
          for (int d = 0; d < D; ++d) o[d] += p * Vh[j * D + d];
        }
        LSE[h * L + i] = lse;
      }
    }
    free(s);
  }
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* Forward for a chosen set of query rows of ONE head ([L][D] inputs).
 * rows[r] in [0,L); O_rows is [nrows][D], LSE_rows is [nrows]. */
int oracle_attn_fwd_rows(const double *Q, const double *K, const double *V,
                         const long *rows, long nrows, double *O_rows,
                         double *LSE_rows, long L, int D, int causal,
                         double scale, int nthreads) {
  int rc = check(1, L, D, scale);
  if (rc) return rc;
  for (long r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= L) return ORACLE_ERR_ARG;
  if (nthreads < 1) nthreads = omp_get_max_threads();
  int failed = 0;
#pragma omp parallel num_threads(nthreads)
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)L);
    if (!s) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (long r = 0; r < nrows; ++r) {
      if (!s) continue;
      long i = rows[r];
      double lse = score_row(Q + i * D, K, L, D, causal, i, scale, s);
      double *o = O_rows + r * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      for (long j = 0; j < L; ++j) {
        if (!allowed(i, j, causal)) continue;
        double p = exp(s[j] - lse);
        for (int d = 0; d < D; ++d) o[d] += p * V[j * D + d];
      }
      LSE_rows[r] = lse;
    }
    free(s);
  }
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* Backward over BH heads. Computes its own fp64 forward (O, LSE) first and
 * returns it together with Dvec and the three gradients. All arrays [BH][L][D]
 * except LSE and Dvec, which are [BH][L].
 *
 * Pass 1, one query row i at a time: LSE_i, O_i, Dvec_i, then the row of dS and
 * dQ_i. Pass 2, one key row j at a time: the column of P and dS is formed again
 * from LSE and Dvec, and dK_j, dV_j are summed over the allowed queries. Both
 * passes follow the definitions in the header literally. */
int oracle_attn_bwd(const double *Q, const double *K, const double *V,
                    const double *dO, double *O, double *LSE, double *Dvec,
                    double *dQ, double *dK, double *dV, long BH, long L, int D,
                    int causal, double scale, int nthreads) {
  int rc = check(BH, L, D, scale);
  if (rc) return rc;
  if (nthreads < 1) nthreads = omp_get_max_threads();
  int failed = 0;
#pragma omp parallel num_threads(nthreads)
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)L);
    if (!s) {
#pragma omp atomic write
      failed = 1;
    }
    /* pass 1: rows */
#pragma omp for collapse(2) schedule(dynamic, 8)
    for (long h = 0; h < BH; ++h) {
      for (long i = 0; i < L; ++i) {
        if (!s) continue;
        const long base = h * L * D;
        const double *Qh = Q + base, *Kh = K + base, *Vh = V + base, *dOh = dO + base;
        double lse = score_row(Qh + i * D, Kh, L, D, causal, i, scale, s);
        double *o = O + base + i * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (long j = 0; j < L; ++j) {
          if (!allowed(i, j, causal)) continue;
          double p = exp(s[j] - lse);
          for (int d = 0; d < D; ++d) o[d] += p * Vh[j * D + d];
        }
        LSE[h * L + i] = lse;
        double dv = dot(dOh + i * D, o, D);
        Dvec[h * L + i] = dv;
        double *dq = dQ + base + i * D;
        for (int d = 0; d < D; ++d) dq[d] = 0.0;
        for (long j = 0; j < L; ++j) {
          if (!allowed(i, j, causal)) continue;
          double p = exp(s[j] - lse);
          double dp = dot(dOh + i * D, Vh + j * D, D);
          double ds = p * (dp - dv);
          for (int d = 0; d < D; ++d) dq[d] += ds * Kh[j * D + d];
        }
        for (int d = 0; d < D; ++d) dq[d] *= scale;
      }
    }
    /* implicit barrier: LSE and Dvec of every row are final here */
    /* pass 2: key rows */
#pragma omp for collapse(2) schedule(dynamic, 8)
    for (long h = 0; h < BH; ++h) {
      for (long j = 0; j < L; ++j) {
        const long base = h * L * D;
        const double *Qh = Q + base, *Kh = K + base, *Vh = V + base, *dOh = dO + base;
        double *dk = dK + base + j * D, *dvv = dV + base + j * D;
        for (int d = 0; d < D; ++d) { dk[d] = 0.0; dvv[d] = 0.0; }
        for (long i = 0; i < L; ++i) {
          if (!allowed(i, j, causal)) continue;
          double sij = scale * dot(Qh + i * D, Kh + j * D, D);
          double p = exp(sij - LSE[h * L + i]);
          double dp = dot(dOh + i * D, Vh + j * D, D);
          double ds = p * (dp - Dvec[h * L + i]);
          for (int d = 0; d < D; ++d) {
            dvv[d] += p * dOh[i * D + d];
            dk[d] += ds * Qh[i * D + d];
          }
        }
        for (int d = 0; d < D; ++d) dk[d] *= scale;
      }
    }
    free(s);
  }
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

int oracle_max_threads(void) { return omp_get_max_threads(); }
