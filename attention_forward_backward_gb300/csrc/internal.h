// internal.h -- host-side declarations shared by the library's translation
// units (launchers of each kernel family). Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

// One attention problem. L is the number of query rows (Lq), Lk the number of
// key rows. With causal set, query i may see key j iff j <= i + off, where off
// is 0 for the top-left alignment and Lk - Lq for the bottom-right one.
struct MgProblem {
  int B, H, L, D;
  int causal;
  float scale;
  int Lk;
  int off;
  // Per-batch key padding (device array of B lengths, or null): batch element
  // b keeps only its first kv_len[b] key rows. br marks the bottom-right causal
  // alignment, whose offset then follows the batch element's own key count.
  const int *kv_len = nullptr;
  int br = 0;
  // ACCEL precision variants: f16 = 1 for f16 Q, K, V, dO (P and dS rounded to
  // f16 as MMA operands) instead of bf16; out16 = 1 to store O, dQ, dK, dV in that
  // 16-bit type instead of f32 (LSE stays f32).
  int f16 = 0;
  int out16 = 0;
  // Derivative-precision policy: hilo = 1 splits dS into a 16-bit hi part and
  // a 16-bit lo part (dS - hi) and accumulates both products for dK and dQ.
  int hilo = 0;
};

// Key rows that one head (bh = b * H + h) attends to, and its causal offset:
// all Lk rows and `off` without padding; with padding the first kv_len[b] rows
// (clamped into [0, Lk]) and, for the bottom-right alignment, the offset
// kv_len[b] - Lq. Rows past the length are masked exactly like rows past Lk.
struct MgKeys {
  int len;
  int off;
};
#ifdef __CUDACC__
__device__ __forceinline__ MgKeys mg_keys(const int *kv_len, int bh, int H, int Lq, int Lk,
                                          int off, int br) {
  if (!kv_len) return MgKeys{Lk, off};
  int n = __ldg(kv_len + bh / H);
  n = n < 0 ? 0 : (n > Lk ? Lk : n);
  return MgKeys{n, br ? n - Lq : off};
}
#endif

// Kernel ids, in the order mg_attn_kernel_name() reports them.
enum MgKernelId {
  MGK_STRICT_FWD = 0,
  MGK_STRICT_DVEC = 1,
  MGK_STRICT_DKDV = 2,
  MGK_ACCEL_FWD = 3,
  MGK_ACCEL_DVEC = 4,
  MGK_ACCEL_DKDV_DQ = 5,  // fused dK/dV kernel that also adds dQ (atomic mode)
  MGK_DQ_ZERO = 6,
  MGK_ACCEL_DKDV = 7,     // dK/dV kernel of the two-pass backward
  MGK_ACCEL_DQ = 8,       // dQ pass of the two-pass backward
  MGK_DECODE_FWD = 9,     // split-key forward for a few query rows (partials + merge)
  MGK_DQ_ROUND = 10,      // f32 dQ accumulator rounded to the 16-bit output type
  MGK_CONV_DGRAD = 11,    // convolution input gradient
  MGK_CONV_WGRAD = 12,    // convolution weight gradient (after zeroing dW)
  MGK_COUNT = 13
};

// Device error codes written into the device error word by bounded waits.
enum MgDeviceError : unsigned int {
  MG_DEVERR_NONE = 0,
  MG_DEVERR_TIMEOUT = 1
};

// STRICT_F32 (FFMA) kernels.
cudaError_t mg_launch_strict_fwd(const float *Q, const float *K, const float *V, float *O,
                                 float *LSE, const MgProblem &p, cudaStream_t st);
cudaError_t mg_launch_strict_dkdv(const float *Q, const float *K, const float *V,
                                  const float *dO, const float *LSE, const float *Dvec,
                                  float *dQ, float *dK, float *dV, const MgProblem &p,
                                  cudaStream_t st);

// Dvec = rowsum(dO * O): STRICT (f32 O and dO).
cudaError_t mg_launch_dvec_f32(const float *O, const float *dO, float *Dvec, const MgProblem &p,
                               cudaStream_t st);
// ACCEL variants: dO bf16 or f16 (p.f16), O f32 or of dO's 16-bit type (p.out16).
cudaError_t mg_launch_dvec_16(const void *O, const void *dO, float *Dvec, const MgProblem &p,
                              cudaStream_t st);

// ACCEL_BF16 (tcgen05 / TMEM / TMA) kernels. `err` is the device error word.
// mg_launch_accel_dkdv: the fused kernel; it computes dK and dV and adds dQ
// into a zeroed dQ (dQ must not be null).
// Q, K, V (and dO) are bf16 or f16 (p.f16); O is f32 or 16-bit (p.out16).
cudaError_t mg_launch_accel_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                const MgProblem &p, unsigned int *err, cudaStream_t st);
// dQ is always f32 here (the caller's dQ, or an f32 accumulator for 16-bit
// outputs); dK, dV are f32 or 16-bit (p.out16).
cudaError_t mg_launch_accel_dkdv(const void *Q, const void *K, const void *V, const void *dO,
                                 const float *LSE, const float *Dvec, float *dQ, void *dK,
                                 void *dV, const MgProblem &p, unsigned int *err,
                                 cudaStream_t st);

// dK/dV kernel of the two-pass backward: two query blocks in flight per CTA.
cudaError_t mg_launch_accel_dkdv_pp(const void *Q, const void *K, const void *V, const void *dO,
                                    const float *LSE, const float *Dvec, void *dK, void *dV,
                                    const MgProblem &p, unsigned int *err, cudaStream_t st);

// Limit of every bounded wait in the tensor-core kernels, in ns: the environment
// variable MG_WAIT_TIMEOUT_MS (read once per process, at least 1 ms), else 4 s.
uint64_t mg_wait_limit_ns();

// Split-key forward for at most mg_decode_max_rows() query rows (decoding). The
// partial records need mg_decode_workspace_floats() floats of scratch.
int mg_decode_max_rows();
void mg_decode_split(const MgProblem &p, int *S, int *chunk, bool tc);
size_t mg_decode_workspace_floats(const MgProblem &p, bool tc);
cudaError_t mg_launch_decode_fwd(const void *Q, const void *K, const void *V, float *O,
                                 float *LSE, float *part, const MgProblem &p, int in_type,
                                 unsigned int *err, cudaStream_t st);

// The argument checks every compute call starts with (sizes, mask, scale,
// contract, head dim), in the same order: MG_OK or the mg_status_t to return.
int mg_check_args(int B, int H, int Lq, int Lk, int D, int mask, float scale, int contract);

// Number of SMs of the current device, read once per device (152 on a GB300;
// 152 is also the answer if the device cannot be queried).
int mg_sm_count();

// Opt a kernel into more than 48 KB of dynamic shared memory once per device.
cudaError_t mg_set_smem_attr(const void *func, int bytes, int slot);

// ACCEL dQ pass (one CTA per 128-row query block; dQ stored, not reduced: f32
// or 16-bit by p.out16).
cudaError_t mg_launch_accel_dq(const void *Q, const void *K, const void *V, const void *dO,
                               const float *LSE, const float *Dvec, void *dQ, const MgProblem &p,
                               unsigned int *err, cudaStream_t st);

// dst (16-bit, bf16 or f16 by `f16`) = src (f32), n elements (n % 4 == 0).
cudaError_t mg_launch_f32_to_16(const float *src, void *dst, size_t n, bool f16,
                                cudaStream_t st);

// A channels-last 2-D convolution: X [N][H][W][C], Wt [K][R][S][C], Y and dY
// [N][P][Q][K] with P = (H + 2 pad - R) / stride + 1, Q likewise; f16 = 1 for f16
// operands (else bf16). Shapes are validated by the caller.
struct MgConvProblem {
  int N, H, W, C, K, R, S, stride, pad, P, Q;
  int f16;
};

// dX (f32, overwritten) from dY and Wt.
cudaError_t mg_launch_conv_dgrad(const void *dY, const void *Wt, float *dX,
                                 const MgConvProblem &p, unsigned int *err, cudaStream_t st);
// dW += the weight gradient from X and dY (f32; the caller zeroes dW first).
cudaError_t mg_launch_conv_wgrad(const void *X, const void *dY, float *dW,
                                 const MgConvProblem &p, unsigned int *err, cudaStream_t st);

// Partial records of the split-key forward with both products on the tensor
// cores (16-bit inputs; the split from mg_decode_split(..., true)).
cudaError_t mg_launch_decode_tc_partial(const void *Q, const void *K, const void *V, float *part,
                                        const MgProblem &p, int S, int chunk, unsigned int *err,
                                        cudaStream_t st);
