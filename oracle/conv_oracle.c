/*
 * conv_oracle.c -- fp64 CPU oracle for the two derivatives of a 2-D convolution
 * (input gradient and weight gradient).
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library. The product path (the CUDA
 * library and its Python binding) never calls, links or imports it, and it
 * shares no code, header, table or helper with that path.
 *
 * What it computes. "Meganeura: Portable GPU Training and Inference through
 * Vulkan and Metal" lists convolution input and weight derivatives among the
 * backward-only graph nodes (Section 3.1) and names the three derivative
 * kernels that own its ResNet-50 training gap (Section 7.3, "Convolution
 * derivatives own the ResNet gap": a weight-gradient GEMM, its small-output
 * variant, and an input-gradient GEMM). The pages print no formula, so this
 * file writes out the textbook definition of a 2-D convolution as deep-learning
 * frameworks define it (cross-correlation, zero padding, equal stride and
 * padding on both spatial axes, no dilation, one group) and its chain rule.
 * Layouts are channels-last: X [N][H][W][C], weights Wt [K][R][S][C],
 * Y and dY [N][P][Q][K] with P = (H + 2 pad - R) / stride + 1 and
 * Q = (W + 2 pad - S) / stride + 1 (integer division):
 *
 *   Y[n,p,q,k]   = sum_{r,s,c} X[n, p*stride - pad + r, q*stride - pad + s, c] Wt[k,r,s,c]
 *                  (X read as 0 outside [0,H) x [0,W))
 *   dX[n,h,w,c]  = sum over (p,q,k,r,s) with p*stride - pad + r = h and
 *                  q*stride - pad + s = w of dY[n,p,q,k] Wt[k,r,s,c]
 *   dW[k,r,s,c]  = sum_{n,p,q} dY[n,p,q,k] X[n, p*stride - pad + r, q*stride - pad + s, c]
 *
 * dX is written as the literal adjoint of the forward: every term of the
 * forward sum adds dY * Wt into the input element it read. The sampled forms
 * (_at) evaluate single elements by gathering the same terms; the tests check
 * that both forms agree, that the three functions satisfy the adjoint identity
 * <Y(X,Wt), G> = <X, dX(G,Wt)> = <Wt, dW(X,G)>, finite differences, 1x1
 * convolutions as plain matrix products and torch's float64 convolution.
 *
 * Threads: OpenMP over batch images (forward, dX) or output channels (dW);
 * every output element is written by one iteration in a fixed order, so results
 * do not depend on the thread count.
 */
#include <stdlib.h>
#include <string.h>
#include <omp.h>

#define CONV_OK 0
#define CONV_ERR_ARG 1

static int check(long N, long H, long W, long C, long K, long R, long S, long st, long pad,
                 long *P, long *Q) {
  if (N < 1 || H < 1 || W < 1 || C < 1 || K < 1 || R < 1 || S < 1 || st < 1 || pad < 0)
    return CONV_ERR_ARG;
  if (H + 2 * pad < R || W + 2 * pad < S) return CONV_ERR_ARG;
  *P = (H + 2 * pad - R) / st + 1;
  *Q = (W + 2 * pad - S) / st + 1;
  return CONV_OK;
}

static inline void set_threads(int nthreads) {
  if (nthreads > 0) omp_set_num_threads(nthreads);
}

int conv_oracle_fwd(const double *X, const double *Wt, double *Y, long N, long H, long W, long C,
                    long K, long R, long S, long st, long pad, int nthreads) {
  long P, Q;
  if (check(N, H, W, C, K, R, S, st, pad, &P, &Q)) return CONV_ERR_ARG;
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
  for (long n = 0; n < N; ++n)
    for (long p = 0; p < P; ++p)
      for (long q = 0; q < Q; ++q)
        for (long k = 0; k < K; ++k) {
          double acc = 0.0;
          for (long r = 0; r < R; ++r) {
            const long h = p * st - pad + r;
            if (h < 0 || h >= H) continue;
            for (long s = 0; s < S; ++s) {
              const long w = q * st - pad + s;
              if (w < 0 || w >= W) continue;
              const double *x = X + ((n * H + h) * W + w) * C;
              const double *wt = Wt + ((k * R + r) * S + s) * C;
              for (long c = 0; c < C; ++c) acc += x[c] * wt[c];
            }
          }
          Y[((n * P + p) * Q + q) * K + k] = acc;
        }
  return CONV_OK;
}

int conv_oracle_grad_input(const double *dY, const double *Wt, double *dX, long N, long H,
                           long W, long C, long K, long R, long S, long st, long pad,
                           int nthreads) {
  long P, Q;
  if (check(N, H, W, C, K, R, S, st, pad, &P, &Q)) return CONV_ERR_ARG;
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
  for (long n = 0; n < N; ++n) {
    double *dx = dX + n * H * W * C;
    memset(dx, 0, sizeof(double) * H * W * C);
    for (long p = 0; p < P; ++p)
      for (long q = 0; q < Q; ++q)
        for (long k = 0; k < K; ++k) {
          const double g = dY[((n * P + p) * Q + q) * K + k];
          for (long r = 0; r < R; ++r) {
            const long h = p * st - pad + r;
            if (h < 0 || h >= H) continue;
            for (long s = 0; s < S; ++s) {
              const long w = q * st - pad + s;
              if (w < 0 || w >= W) continue;
              const double *wt = Wt + ((k * R + r) * S + s) * C;
              double *o = dx + (h * W + w) * C;
              for (long c = 0; c < C; ++c) o[c] += g * wt[c];
            }
          }
        }
  }
  return CONV_OK;
}

int conv_oracle_grad_weight(const double *X, const double *dY, double *dW, long N, long H,
                            long W, long C, long K, long R, long S, long st, long pad,
                            int nthreads) {
  long P, Q;
  if (check(N, H, W, C, K, R, S, st, pad, &P, &Q)) return CONV_ERR_ARG;
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
  for (long k = 0; k < K; ++k) {
    double *dw = dW + k * R * S * C;
    memset(dw, 0, sizeof(double) * R * S * C);
    for (long n = 0; n < N; ++n)
      for (long p = 0; p < P; ++p)
        for (long q = 0; q < Q; ++q) {
          const double g = dY[((n * P + p) * Q + q) * K + k];
          for (long r = 0; r < R; ++r) {
            const long h = p * st - pad + r;
            if (h < 0 || h >= H) continue;
            for (long s = 0; s < S; ++s) {
              const long w = q * st - pad + s;
              if (w < 0 || w >= W) continue;
              const double *x = X + ((n * H + h) * W + w) * C;
              double *o = dw + (r * S + s) * C;
              for (long c = 0; c < C; ++c) o[c] += g * x[c];
            }
          }
        }
  }
  return CONV_OK;
}

/* dX at npts points idx[4i .. 4i+3] = (n, h, w, c): the terms of the forward
 * that read input element (n, h, w, c), gathered. */
int conv_oracle_grad_input_at(const double *dY, const double *Wt, const long *idx, long npts,
                              double *out, long N, long H, long W, long C, long K, long R,
                              long S, long st, long pad, int nthreads) {
  long P, Q;
  if (check(N, H, W, C, K, R, S, st, pad, &P, &Q)) return CONV_ERR_ARG;
  for (long i = 0; i < npts; ++i) {
    const long *t = idx + 4 * i;
    if (t[0] < 0 || t[0] >= N || t[1] < 0 || t[1] >= H || t[2] < 0 || t[2] >= W || t[3] < 0 ||
        t[3] >= C)
      return CONV_ERR_ARG;
  }
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
  for (long i = 0; i < npts; ++i) {
    const long n = idx[4 * i], h = idx[4 * i + 1], w = idx[4 * i + 2], c = idx[4 * i + 3];
    double acc = 0.0;
    for (long r = 0; r < R; ++r) {
      const long ph = h + pad - r; /* = p * st for the output row p that read h */
      if (ph < 0 || ph % st) continue;
      const long p = ph / st;
      if (p >= P) continue;
      for (long s = 0; s < S; ++s) {
        const long qw = w + pad - s;
        if (qw < 0 || qw % st) continue;
        const long q = qw / st;
        if (q >= Q) continue;
        for (long k = 0; k < K; ++k)
          acc += dY[((n * P + p) * Q + q) * K + k] * Wt[((k * R + r) * S + s) * C + c];
      }
    }
    out[i] = acc;
  }
  return CONV_OK;
}

/* dW at npts points idx[4i .. 4i+3] = (k, r, s, c). */
int conv_oracle_grad_weight_at(const double *X, const double *dY, const long *idx, long npts,
                               double *out, long N, long H, long W, long C, long K, long R,
                               long S, long st, long pad, int nthreads) {
  long P, Q;
  if (check(N, H, W, C, K, R, S, st, pad, &P, &Q)) return CONV_ERR_ARG;
  for (long i = 0; i < npts; ++i) {
    const long *t = idx + 4 * i;
    if (t[0] < 0 || t[0] >= K || t[1] < 0 || t[1] >= R || t[2] < 0 || t[2] >= S || t[3] < 0 ||
        t[3] >= C)
      return CONV_ERR_ARG;
  }
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
  for (long i = 0; i < npts; ++i) {
    const long k = idx[4 * i], r = idx[4 * i + 1], s = idx[4 * i + 2], c = idx[4 * i + 3];
    double acc = 0.0;
    for (long n = 0; n < N; ++n)
      for (long p = 0; p < P; ++p) {
        const long h = p * st - pad + r;
        if (h < 0 || h >= H) continue;
        for (long q = 0; q < Q; ++q) {
          const long w = q * st - pad + s;
          if (w < 0 || w >= W) continue;
          acc += dY[((n * P + p) * Q + q) * K + k] * X[((n * H + h) * W + w) * C + c];
        }
      }
    out[i] = acc;
  }
  return CONV_OK;
}
