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
 * Queries and keys may differ in number (Lq query rows, Lk key rows; cross
 * attention). The mask is one of: none (every key allowed); causal aligned at
 * the top left, allowed(i,j) = (j <= i); causal aligned at the bottom right,
 * allowed(i,j) = (j <= i + Lk - Lq), so that the last query sees every key. A
 * query row with no allowed key (bottom-right alignment with Lq > Lk) has an
 * empty softmax: its output row is 0, its LSE is -inf and it contributes
 * nothing to any gradient. With Lq = Lk both causal alignments coincide.
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

#define ORACLE_MASK_NONE 0
#define ORACLE_MASK_CAUSAL 1             /* top-left aligned: j <= i */
#define ORACLE_MASK_CAUSAL_BOTTOM_RIGHT 2 /* j <= i + (Lk - Lq) */

/* off = Lk - Lq (used by the bottom-right alignment only) */
static inline int allowed(long i, long j, int mask, long off) {
  if (mask == ORACLE_MASK_CAUSAL) return j <= i;
  if (mask == ORACLE_MASK_CAUSAL_BOTTOM_RIGHT) return j <= i + off;
  return 1;
}

static inline double dot(const double *a, const double *b, int D) {
  double acc = 0.0;
  for (int d = 0; d < D; ++d) acc += a[d] * b[d];
  return acc;
}

/* Scores of query row i against the Lk keys; masked entries are -inf.
 * Returns LSE_i, or -inf when the row has no allowed key. */
static double score_row(const double *q, const double *K, long Lk, int D, int mask,
                        long off, long i, double scale, double *s) {
  double m = -INFINITY;
  for (long j = 0; j < Lk; ++j) {
    if (allowed(i, j, mask, off)) {
      s[j] = scale * dot(q, K + j * D, D);
      if (s[j] > m) m = s[j];
    } else {
      s[j] = -INFINITY;
    }
  }
  if (m == -INFINITY) return -INFINITY;
  double sum = 0.0;
  for (long j = 0; j < Lk; ++j)
    if (allowed(i, j, mask, off)) sum += exp(s[j] - m);
  return m + log(sum);
}

static int check(long BH, long Lq, long Lk, int D, int mask, double scale) {
  if (BH < 1 || Lq < 1 || Lk < 1 || D < 1) return ORACLE_ERR_ARG;
  if (mask < ORACLE_MASK_NONE || mask > ORACLE_MASK_CAUSAL_BOTTOM_RIGHT) return ORACLE_ERR_ARG;
  if (!(scale > 0.0) || !isfinite(scale)) return ORACLE_ERR_ARG;
  return ORACLE_OK;
}

/* Forward over BH independent heads: Q, O [BH][Lq][D], K, V [BH][Lk][D],
 * LSE [BH][Lq]. */
int oracle_attn_fwd_ex(const double *Q, const double *K, const double *V,
                       double *O, double *LSE, long BH, long Lq, long Lk, int D,
                       int mask, double scale, int nthreads) {
  int rc = check(BH, Lq, Lk, D, mask, scale);
  if (rc) return rc;
  if (nthreads < 1) nthreads = omp_get_max_threads();
  const long off = Lk - Lq;
  int failed = 0;
#pragma omp parallel num_threads(nthreads)
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)Lk);
    if (!s) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for collapse(2) schedule(dynamic, 8)
    for (long h = 0; h < BH; ++h) {
      for (long i = 0; i < Lq; ++i) {
        if (!s) continue;
        const double *Qh = Q + h * Lq * D, *Kh = K + h * Lk * D, *Vh = V + h * Lk * D;
        double lse = score_row(Qh + i * D, Kh, Lk, D, mask, off, i, scale, s);
        double *o = O + (h * Lq + i) * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (lse != -INFINITY) {
          for (long j = 0; j < Lk; ++j) {
            if (!allowed(i, j, mask, off)) continue;
            double p = exp(s[j] - lse);
            for (int d = 0; d < D; ++d) o[d] += p * Vh[j * D + d];
          }
        }
        LSE[h * Lq + i] = lse;
      }
    }
    free(s);
  }
  return failed ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/* Self-attention form: Lq = Lk = L, causal selects the (top-left) causal mask. */
int oracle_attn_fwd(const double *Q, const double *K, const double *V,
                    double *O, double *LSE, long BH, long L, int D, int causal,
                    double scale, int nthreads) {
  return oracle_attn_fwd_ex(Q, K, V, O, LSE, BH, L, L, D,
                            causal ? ORACLE_MASK_CAUSAL : ORACLE_MASK_NONE, scale, nthreads);
}

/* Forward for a chosen set of query rows of ONE head ([L][D] inputs).
 * rows[r] in [0,L); O_rows is [nrows][D], LSE_rows is [nrows]. */
int oracle_attn_fwd_rows(const double *Q, const double *K, const double *V,
                         const long *rows, long nrows, double *O_rows,
                         double *LSE_rows, long L, int D, int causal,
                         double scale, int nthreads) {
  const int mask = causal ? ORACLE_MASK_CAUSAL : ORACLE_MASK_NONE;
  int rc = check(1, L, L, D, mask, scale);
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
      double lse = score_row(Q + i * D, K, L, D, mask, 0, i, scale, s);
      double *o = O_rows + r * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      for (long j = 0; j < L; ++j) {
        if (!allowed(i, j, mask, 0)) continue;
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
 * returns it together with Dvec and the three gradients. Q, dO, O, dQ are
 * [BH][Lq][D], K, V, dK, dV are [BH][Lk][D], LSE and Dvec are [BH][Lq].
 *
 * Pass 1, one query row i at a time: LSE_i, O_i, Dvec_i, then the row of dS and
 * dQ_i. Pass 2, one key row j at a time: the column of P and dS is formed again
 * from LSE and Dvec, and dK_j, dV_j are summed over the allowed queries. Both
 * passes follow the definitions in the header literally; rows with an empty
 * softmax (LSE = -inf) contribute nothing. */
int oracle_attn_bwd_ex(const double *Q, const double *K, const double *V,
                       const double *dO, double *O, double *LSE, double *Dvec,
                       double *dQ, double *dK, double *dV, long BH, long Lq, long Lk,
                       int D, int mask, double scale, int nthreads) {
  int rc = check(BH, Lq, Lk, D, mask, scale);
  if (rc) return rc;
  if (nthreads < 1) nthreads = omp_get_max_threads();
  const long off = Lk - Lq;
  int failed = 0;
#pragma omp parallel num_threads(nthreads)
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)Lk);
    if (!s) {
#pragma omp atomic write
      failed = 1;
    }
    /* pass 1: query rows */
#pragma omp for collapse(2) schedule(dynamic, 8)
    for (long h = 0; h < BH; ++h) {
      for (long i = 0; i < Lq; ++i) {
        if (!s) continue;
        const long bq = h * Lq * D, bk = h * Lk * D;
        const double *Qh = Q + bq, *Kh = K + bk, *Vh = V + bk, *dOh = dO + bq;
        double lse = score_row(Qh + i * D, Kh, Lk, D, mask, off, i, scale, s);
        double *o = O + bq + i * D;
        double *dq = dQ + bq + i * D;
        for (int d = 0; d < D; ++d) { o[d] = 0.0; dq[d] = 0.0; }
        LSE[h * Lq + i] = lse;
        if (lse == -INFINITY) {
          Dvec[h * Lq + i] = 0.0;
          continue;
        }
        for (long j = 0; j < Lk; ++j) {
          if (!allowed(i, j, mask, off)) continue;
          double p = exp(s[j] - lse);
          for (int d = 0; d < D; ++d) o[d] += p * Vh[j * D + d];
        }
        double dv = dot(dOh + i * D, o, D);
        Dvec[h * Lq + i] = dv;
        for (long j = 0; j < Lk; ++j) {
          if (!allowed(i, j, mask, off)) continue;
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
      for (long j = 0; j < Lk; ++j) {
        const long bq = h * Lq * D, bk = h * Lk * D;
        const double *Qh = Q + bq, *Kh = K + bk, *Vh = V + bk, *dOh = dO + bq;
        double *dk = dK + bk + j * D, *dvv = dV + bk + j * D;
        for (int d = 0; d < D; ++d) { dk[d] = 0.0; dvv[d] = 0.0; }
        for (long i = 0; i < Lq; ++i) {
          if (!allowed(i, j, mask, off) || LSE[h * Lq + i] == -INFINITY) continue;
          double sij = scale * dot(Qh + i * D, Kh + j * D, D);
          double p = exp(sij - LSE[h * Lq + i]);
          double dp = dot(dOh + i * D, Vh + j * D, D);
          double ds = p * (dp - Dvec[h * Lq + i]);
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

/* Self-attention form: Lq = Lk = L, causal selects the (top-left) causal mask. */
int oracle_attn_bwd(const double *Q, const double *K, const double *V,
                    const double *dO, double *O, double *LSE, double *Dvec,
                    double *dQ, double *dK, double *dV, long BH, long L, int D,
                    int causal, double scale, int nthreads) {
  return oracle_attn_bwd_ex(Q, K, V, dO, O, LSE, Dvec, dQ, dK, dV, BH, L, L, D,
                            causal ? ORACLE_MASK_CAUSAL : ORACLE_MASK_NONE, scale, nthreads);
}

int oracle_max_threads(void) { return omp_get_max_threads(); }
