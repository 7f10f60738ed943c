/*
 * mg_attn.h -- C ABI of libmgattn.so: multi-head scaled-dot-product attention,
 * forward and backward, as one training step on one GB300 GPU (sm_103a).
 *
 * The operation. "Meganeura: Portable GPU Training and Inference through Vulkan
 * and Metal" treats attention as one graph node with its own derivative rule
 * (Section 3.1) and lowers it to three kernel archetypes: tiled attention
 * forward, dQ, and fused dK+dV (Section 3.3; Section 8 makes the fused dK+dV
 * kernel an invariant). The pages print no formula; the functions below compute
 * the textbook definition, per (batch b, head h):
 *
 *   s_ij = scale * Q_i . K_j,  allowed(i,j) = (j <= i) when causal (top-left)
 *   LSE_i = ln sum_{allowed j} exp(s_ij)          (natural log, scaled logits)
 *   P_ij = exp(s_ij - LSE_i) on allowed pairs, else 0;   O_i = sum_j P_ij V_j
 *   Dvec_i = dO_i . O_i;  dS_ij = P_ij (dO_i . V_j - Dvec_i)
 *   dV_j = sum_i P_ij dO_i;  dQ_i = scale sum_j dS_ij K_j;  dK_j = scale sum_i dS_ij Q_i
 *
 * No L x L matrix is ever stored: the kernels tile the key axis and keep a
 * running max and sum (forward) or recompute P from LSE (backward).
 *
 * Arithmetic contracts (Section 4.2 separates a strict-f32 contract from an
 * accelerated one whose forward inputs are rounded to a 16-bit format with f32
 * accumulation and f32 stores; Section 10: strict governs permissions, not the
 * order of operations):
 *   MG_CONTRACT_STRICT_F32  every tensor f32; FP32 CUDA cores only (FFMA, no
 *                           TF32, no tensor cores). Results are not bitwise
 *                           reproducible across runs (dQ uses f32 atomics).
 *   MG_CONTRACT_ACCEL_BF16  Q, K, V, dO are bf16; O, dQ, dK, dV are f32; LSE f32.
 *                           Products run on tcgen05 tensor cores with f32
 *                           accumulation in tensor memory; P (forward and dV)
 *                           and dS (dK, dQ) are rounded to bf16 (RNE) as MMA
 *                           operands, everything else stays f32.
 *   MG_CONTRACT_ACCEL_F16   the same with f16 in place of bf16: the 16-bit
 *                           format the pages' accelerated path rounds its matrix
 *                           inputs to (Section 4.2). f16 has 10 mantissa bits
 *                           (bf16: 7) but a narrow range: P and dS below 2^-24
 *                           round to zero as MMA operands, the underflow that
 *                           the pages' precision bit guards derivative regions
 *                           against (Section 3.1); ACCEL_BF16, with f32's
 *                           range, cannot underflow there.
 * Flags OR-ed into an ACCEL contract:
 *   MG_OUT_16               O, dQ, dK, dV are stored in the inputs' 16-bit type
 *                           (bf16 or f16, RNE) instead of f32; LSE stays f32, and
 *                           every accumulation stays f32 (dQ's reductions add
 *                           into an f32 accumulator in the backward's workspace,
 *                           rounded once at the end). The backward then reads
 *                           O in that 16-bit type. Not valid with STRICT_F32
 *                           (MG_ERR_UNSUPPORTED), the decode forward or the
 *                           no-allocation backward.
 *   MG_DS_HILO              derivative-precision policy of the backward (the
 *                           pages attach a precision bit to derivative regions
 *                           so that the 16-bit promotion does not round small
 *                           gradient operands, Section 3.1): dS is split into
 *                           hi = round16(dS) and lo = round16(dS - hi), and dK
 *                           and dQ accumulate both products (dS_hi + dS_lo)
 *                           with f32 accumulation, so that the dS operand keeps
 *                           about twice the 16-bit type's mantissa (bf16: 16
 *                           bits, f16: 22) at twice the dK and dQ tensor work.
 *                           The split widens the mantissa, not the exponent
 *                           range (with f16, dS below 2^-24 still flushes). P
 *                           (forward, dV) stays one 16-bit operand. Runs in
 *                           the two-pass backward (a dK/dV kernel and a dQ
 *                           pass). No effect on the forward calls; not valid
 *                           with STRICT_F32 (MG_ERR_UNSUPPORTED).
 *
 * Layout. Q, K, V, O, dO, dQ, dK, dV are dense row-major [B][H][L][D] (D
 * innermost, no padding, no strides). LSE (and the workspace's Dvec) are
 * [B][H][L] f32. The self-attention calls take Lq = Lk = L; the _ex calls take
 * Q, O, dO, dQ as [B][H][Lq][D], K, V, dK, dV as [B][H][Lk][D] and LSE as
 * [B][H][Lq] (cross attention), with a mask of mg_mask_t:
 *   MG_MASK_NONE                 every key allowed
 *   MG_MASK_CAUSAL               allowed(i,j) = (j <= i)           (top-left)
 *   MG_MASK_CAUSAL_BOTTOM_RIGHT  allowed(i,j) = (j <= i + Lk - Lq) (the last
 *                                query sees every key)
 * A query row with no allowed key (bottom-right with Lq > Lk) has an empty
 * softmax: O row 0, LSE -inf, and no contribution to any gradient.
 *
 * Ownership. The caller owns every buffer (device memory, e.g. from PyTorch).
 * The library never allocates or frees device memory on these calls; the
 * backward's scratch is the caller-provided workspace. All compute calls are
 * asynchronous on `stream` (a cudaStream_t; NULL is the legacy default stream)
 * and return after the launches are queued.
 *
 * Errors. Every call returns an mg_status_t synchronously. Argument errors are
 * detected on the host before anything is launched (nothing is written).
 * A failed launch is MG_ERR_CUDA. A kernel that gives up on a bounded wait sets
 * a device error word; mg_get_device_error() reports it as MG_ERR_TIMEOUT.
 * Nothing aborts the process.
 *
 * Device state. The library looks up, once per device, the device addresses of
 * its own module variables (the device error word, the no-allocation scratch)
 * and caches them. They belong to the device's context: after cudaDeviceReset
 * on a device the library has used, the cached addresses are stale, so do not
 * call the library on a device reset since its first call there.
 *
 * Preconditions checked: pointers non-NULL and 16-byte aligned; B, H, L >= 1;
 * B*H <= 2^24, L (Lq, Lk) <= 2^20; D in {32, 64, 128} (else
 * MG_ERR_UNSUPPORTED); causal in {0, 1} (mask one of mg_mask_t); scale finite
 * and > 0; contract valid; no output buffer overlaps an input buffer or
 * another output.
 */
#ifndef MG_ATTN_H
#define MG_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MG_CONTRACT_STRICT_F32 = 0,
  MG_CONTRACT_ACCEL_BF16 = 1,
  MG_CONTRACT_ACCEL_F16 = 2,
  MG_CONTRACT_BASE_MASK = 0xff, /* the base contract is contract & MG_CONTRACT_BASE_MASK */
  MG_OUT_16 = 0x100,            /* flag: 16-bit O, dQ, dK, dV (see above) */
  MG_DS_HILO = 0x200            /* flag: hi/lo split of dS in the backward (see above) */
} mg_contract_t;

typedef enum {
  MG_MASK_NONE = 0,
  MG_MASK_CAUSAL = 1,              /* j <= i (top-left aligned) */
  MG_MASK_CAUSAL_BOTTOM_RIGHT = 2  /* j <= i + Lk - Lq */
} mg_mask_t;

typedef enum {
  MG_OK = 0,
  MG_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, aliasing, bad scale */
  MG_ERR_UNSUPPORTED = 2, /* D not in {32,64,128}; Lq > 8 for the decode forward */
  MG_ERR_WORKSPACE = 3,   /* workspace missing or smaller than the query says */
  MG_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  MG_ERR_TIMEOUT = 5      /* a kernel gave up on a bounded wait (device error word) */
} mg_status_t;

/*
 * Forward: O = softmax(scale * Q K^T + causal mask) V and LSE (natural log).
 * Tiled attention forward archetype (Section 3.3 of the paper).
 *   Q, K, V  in   [B][H][L][D]; f32 (STRICT), bf16 or f16 (ACCEL_BF16, ACCEL_F16)
 *   O        out  [B][H][L][D] f32 (16-bit with MG_OUT_16), overwritten
 *   LSE      out  [B][H][L] f32, overwritten; the backward requires it
 */
int mg_attn_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
                int B, int H, int L, int D, int causal, float scale, int contract,
                void *stream);

/*
 * Forward with Lq query rows and Lk key rows (cross attention) and a mask of
 * mg_mask_t. Q, O [B][H][Lq][D]; K, V [B][H][Lk][D]; LSE [B][H][Lq]. Same
 * contracts, ownership and errors as mg_attn_fwd, which is this call with
 * Lq = Lk = L and mask = causal ? MG_MASK_CAUSAL : MG_MASK_NONE.
 */
int mg_attn_fwd_ex(const void *Q, const void *K, const void *V, void *O, float *LSE,
                   int B, int H, int Lq, int Lk, int D, int mask, float scale, int contract,
                   void *stream);

/* Bytes of device workspace mg_attn_bwd needs for this shape and contract:
 * Dvec, [B][H][L] f32, rounded up to 256 bytes; with MG_OUT_16 also an f32 dQ
 * accumulator [B][H][L][D], rounded up to 256 bytes. 0 for invalid arguments. */
size_t mg_attn_bwd_workspace_bytes(int B, int H, int L, int D, int contract);

/*
 * Backward: dQ, dK, dV of loss = sum(dO * O), given the forward's O and LSE.
 * dQ and fused dK+dV archetypes (Sections 3.3 and 8 of the paper); the
 * derivative region keeps f32 accumulation (Sections 3.1 and 4.2).
 *   Q, K, V, dO  in   [B][H][L][D]; f32 (STRICT), bf16 or f16 (ACCEL_BF16, ACCEL_F16)
 *   O            in   [B][H][L][D] as written by mg_attn_fwd (f32, or 16-bit with
 *                     MG_OUT_16)
 *   LSE          in   [B][H][L] f32, as written by mg_attn_fwd
 *   dQ, dK, dV   out  [B][H][L][D] f32 (16-bit with MG_OUT_16), overwritten (never
 *                     accumulated into)
 *   workspace    scratch of at least mg_attn_bwd_workspace_bytes() bytes,
 *                16-byte aligned; its contents on entry do not matter
 * Steps on the stream: Dvec = rowsum(dO * O) into the workspace; then one
 * kernel per key block recomputes P from Q, K, LSE and accumulates dK, dV.
 * STRICT and the default ACCEL mode add each key block's dQ contribution into
 * a zeroed dQ with f32 reductions (results not bitwise reproducible); with the
 * environment variable MG_DQ_MODE=pass (read once per process) ACCEL instead
 * runs a dK/dV kernel and a separate dQ pass over query blocks that stores dQ
 * without atomics (bitwise reproducible; slower on GB300 at long sequences).
 */
int mg_attn_bwd(const void *Q, const void *K, const void *V, const void *O,
                const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                int B, int H, int L, int D, int causal, float scale, int contract,
                void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes for mg_attn_bwd_ex (Dvec is [B][H][Lq] f32, and with
 * MG_OUT_16 a [B][H][Lq][D] f32 dQ accumulator, each rounded up to 256 bytes).
 * 0 for invalid arguments. */
size_t mg_attn_bwd_workspace_bytes_ex(int B, int H, int Lq, int Lk, int D, int contract);

/*
 * Backward with Lq query rows and Lk key rows and a mask of mg_mask_t, given
 * the O and LSE of mg_attn_fwd_ex with the same arguments. Q, O, dO, dQ
 * [B][H][Lq][D]; K, V, dK, dV [B][H][Lk][D]; LSE [B][H][Lq]; workspace of at
 * least mg_attn_bwd_workspace_bytes_ex() bytes. Same contracts, steps,
 * ownership and errors as mg_attn_bwd, which is this call with Lq = Lk = L and
 * mask = causal ? MG_MASK_CAUSAL : MG_MASK_NONE. Key rows that no query may
 * see get dK = dV = 0; query rows with an empty softmax get dQ = 0.
 */
int mg_attn_bwd_ex(const void *Q, const void *K, const void *V, const void *O,
                   const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                   int B, int H, int Lq, int Lk, int D, int mask, float scale, int contract,
                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * Per-batch key padding (cross attention of a batch whose key sequences differ
 * in length, e.g. text conditioning padded to a common Lk; the diffusion
 * workload's text cross-attention in "Meganeura: Portable GPU Training and
 * Inference through Vulkan and Metal", Section 4.1 "Matched workloads"; the
 * pages print no mask convention for it, so this is the plain reading): batch
 * element b has kv_len[b] real key rows, 0 <= kv_len[b] <= Lk, and the rows of
 * K and V at or past kv_len[b] are padding. Batch element b is then exactly the
 * problem of mg_attn_fwd_ex / mg_attn_bwd_ex with Lk = kv_len[b] keys: the
 * bottom-right causal alignment uses its own offset kv_len[b] - Lq, a query row
 * that sees no key has an empty softmax (O row 0, LSE -inf, dQ row 0), and the
 * padding rows of dK and dV are written as 0.
 *   kv_len  device array of B int32 lengths, 4-byte aligned, not overlapping any
 *           output; NULL means no padding (then these calls are mg_attn_fwd_ex
 *           and mg_attn_bwd_ex). The kernels clamp each length into [0, Lk]:
 *           the host cannot read device memory without synchronising, so a
 *           length outside that range is not reported as an error.
 * Padding rows of K and V need not hold meaningful values, but under
 * ACCEL_BF16 they must be finite: the tensor cores read whole 128-row tiles, and
 * a NaN or infinity there would reach the outputs through a product with a zero
 * probability. STRICT_F32 never reads them. Layouts, contracts, workspace
 * (mg_attn_bwd_workspace_bytes_ex), ownership and errors as the _ex calls; the
 * backward needs the O and LSE of mg_attn_fwd_padded with the same kv_len.
 */
int mg_attn_fwd_padded(const void *Q, const void *K, const void *V, void *O, float *LSE,
                       const int *kv_len, int B, int H, int Lq, int Lk, int D, int mask,
                       float scale, int contract, void *stream);
int mg_attn_bwd_padded(const void *Q, const void *K, const void *V, const void *O,
                       const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                       const int *kv_len, int B, int H, int Lq, int Lk, int D, int mask,
                       float scale, int contract, void *workspace, size_t workspace_bytes,
                       void *stream);

/*
 * mg_attn_bwd without a workspace, for callers that cannot allocate device
 * memory at all (a plugin whose host runtime owns every device allocation and
 * offers no scratch, a service that fixes its memory budget at start-up, a
 * caller that cannot afford cudaMalloc's implicit synchronisation). The paper
 * has no counterpart: its runtime plans every buffer itself.
 * Same arguments, results and errors as mg_attn_bwd minus the workspace (its
 * argument checks run first, in the same order). The Dvec scratch is a fixed
 * device array inside the library (4 MiB, held by every GPU that loads the
 * library until the process exits), so B*H*L must not exceed 1,048,576 rows;
 * larger problems with otherwise valid arguments return MG_ERR_WORKSPACE before
 * anything is launched. Nothing is allocated or freed.
 * The first call on each device looks up the array's device address (make it
 * before any stream capture). All calls on a device share the array: calls
 * whose kernels overlap on the GPU race, calls ordered on one stream do not.
 * No part of the array needs to start at zero.
 */
int mg_attn_bwd_noalloc(const void *Q, const void *K, const void *V, const void *O,
                        const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                        int B, int H, int L, int D, int causal, float scale, int contract,
                        void *stream);

/* Workspace bytes for mg_attn_fwd_decode (one partial record of D + 4 f32 per
 * head, key split and query row, rounded up to 256 bytes). 0 for invalid
 * arguments or Lq > 8. */
size_t mg_attn_fwd_decode_workspace_bytes(int B, int H, int Lq, int Lk, int D, int contract);

/*
 * Forward for a few query rows against a long key axis (decoding: Lq <= 8
 * rows per head, e.g. the newest tokens against a key/value cache). Computes
 * exactly what mg_attn_fwd_ex computes for the same arguments, with a different
 * schedule: the key axis is split over many CTAs, each of which keeps the
 * running max, sum and unnormalised output of its keys (the online softmax of
 * the tiled forward archetype, Section 3.3 of the paper), and a second kernel
 * merges the splits. The split count depends on (B, H, Lk), the contract
 * family (f32 or 16-bit) and the device's SM count only.
 *   Q, O       [B][H][Lq][D] (Q f32, bf16 or f16 by contract, O f32), Lq in [1, 8]
 *   K, V       [B][H][Lk][D]
 *   LSE        out [B][H][Lq] f32
 *   mask       mg_mask_t; rows with no allowed key get O = 0, LSE = -inf
 *   workspace  scratch of at least mg_attn_fwd_decode_workspace_bytes() bytes,
 *              16-byte aligned, not overlapping any tensor; contents on entry do
 *              not matter
 * The work is one pass over K and V, bound by HBM. STRICT_F32 computes in f32
 * on the CUDA cores (FFMA). The ACCEL contracts compute S = Q K^T and P V on the
 * tensor cores: keys on the MMA's M axis, the query rows padded to N = 16, f32
 * accumulation, P rounded to the 16-bit input type as the operand (as in
 * mg_attn_fwd), the softmax in f32. Lq > 8 returns MG_ERR_UNSUPPORTED (use
 * mg_attn_fwd_ex). Other preconditions, ownership and errors as mg_attn_fwd_ex;
 * a bounded wait that gives up is reported by mg_get_device_error().
 */
int mg_attn_fwd_decode(const void *Q, const void *K, const void *V, void *O, float *LSE,
                       int B, int H, int Lq, int Lk, int D, int mask, float scale,
                       int contract, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Convolution derivatives ("Meganeura: Portable GPU Training and Inference
 * through Vulkan and Metal", Section 3.1 lists convolution input and weight
 * derivatives among the backward nodes; Section 7.3, "Convolution derivatives
 * own the ResNet gap", names the input-gradient GEMM and the weight-gradient
 * GEMM with its small-output variant). The forward is a 2-D convolution as
 * deep-learning frameworks define it (cross-correlation, zero padding, the same
 * stride and padding on both spatial axes, no dilation, one group), channels
 * last:
 *   X [N][H][W][C], Wt [K][R][S][C], Y and dY [N][P][Q][K],
 *   P = (H + 2 pad - R) / stride + 1,  Q = (W + 2 pad - S) / stride + 1,
 *   Y[n,p,q,k] = sum_{r,s,c} X[n, p*stride - pad + r, q*stride - pad + s, c] Wt[k,r,s,c]
 * and its derivatives are
 *   dX[n,h,w,c] = sum over p*stride - pad + r = h, q*stride - pad + s = w of
 *                 dY[n,p,q,k] Wt[k,r,s,c]
 *   dW[k,r,s,c] = sum_{n,p,q} dY[n,p,q,k] X[n, p*stride - pad + r, q*stride - pad + s, c]
 * Contract: ACCEL_BF16 (X, Wt, dY bf16) or ACCEL_F16 (f16); products on the
 * tcgen05 tensor cores with f32 accumulation; dX and dW are f32 and are
 * overwritten. Only the order of the f32 additions differs from exact
 * arithmetic on the 16-bit inputs; dW adds per-CTA partial sums with f32
 * atomics, so it is not bitwise reproducible across runs (nor is dX when there
 * are too few output tiles to fill the GPU and each tile's reduction is split).
 * Preconditions checked: pointers non-NULL, 16-byte aligned, outputs not
 * overlapping inputs; N, H, W, C, K, R, S >= 1; H, W <= 65535; R, S, pad in
 * [0, 64] with H + 2 pad >= R and W + 2 pad >= S; every tensor below 2^31
 * elements (else MG_ERR_INVALID_ARG); stride 1 or 2, C and K multiples of 8,
 * ceil(K/128) * ceil(C/64) <= 65535, contract ACCEL_BF16 or ACCEL_F16 without
 * flags (else MG_ERR_UNSUPPORTED: STRICT_F32 has no convolution derivatives).
 * Asynchronous on `stream`; no allocation and no synchronising call, so a
 * sequence of these calls can be captured in a CUDA graph (the host cost of one
 * call, argument checks, tensor-map encoding and the launch, is comparable to the
 * kernel time of small layers). The environment variable MG_CONV_MAX_N=128 or 64
 * (read once per process) caps the accumulator width, which is otherwise 256
 * channels of C for C >= 256. Kernel names in the profile: "conv_dgrad",
 * "conv_wgrad".
 */
int mg_conv2d_grad_input(const void *dY, const void *Wt, float *dX, int N, int H, int W, int C,
                         int K, int R, int S, int stride, int pad, int contract, void *stream);
int mg_conv2d_grad_weight(const void *X, const void *dY, float *dW, int N, int H, int W, int C,
                          int K, int R, int S, int stride, int pad, int contract, void *stream);

/* Static, human-readable name of a status code. Never NULL. */
const char *mg_status_string(int status);

/* Synchronises `stream`, then reads and clears the current device's error word.
 * MG_OK if no kernel has reported a give-up since the last call, MG_ERR_TIMEOUT
 * if one has, MG_ERR_CUDA if the synchronisation itself failed. */
int mg_get_device_error(void *stream);

/*
 * Kernel timing for benchmarks. While enabled, every kernel launch made by the
 * calls above is bracketed by two CUDA events recorded on the call's stream.
 * mg_attn_profile_enable(1) (re)creates the event pool (capacity launches) and
 * zeroes the counters; (0) stops recording and frees the events. These are the
 * only entry points that create CUDA objects.
 * mg_attn_profile_read() synchronises on the recorded events and returns, for
 * kernel id `kernel` (0 <= kernel < mg_attn_kernel_count()), the number of
 * recorded launches and their summed device time in milliseconds.
 */
int mg_attn_profile_enable(int enable, int capacity);
int mg_attn_profile_read(int kernel, int *launches, double *total_ms);
int mg_attn_kernel_count(void);
const char *mg_attn_kernel_name(int kernel);

#ifdef __cplusplus
}
#endif

#endif /* MG_ATTN_H */
