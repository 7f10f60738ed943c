// api.cu -- the C ABI of libmgattn.so (declared in include/mg_attn.h):
// argument validation, dispatch on (contract, D), the per-device error word
// and the optional per-kernel event timing used by benchmarks.
//
// The pages ("Meganeura: Portable GPU Training and Inference through Vulkan and
// Metal", Sections 3.5 and 5.6) keep every buffer owned by a static plan and
// allocate nothing while a step runs; the calls here follow the same rule:
// they validate, then enqueue kernels on the caller's stream.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "../../include/mg_attn.h"
#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSlots = 64;

// Device error word: bounded waits in the ACCEL kernels write a code here
// instead of trapping. One copy per device (module globals are per context).
__device__ unsigned int g_mg_device_error;

std::mutex g_mu;
unsigned int *g_err_ptr[kMaxDevices] = {};
bool g_smem_done[kMaxDevices][kMaxSlots] = {};

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

// Device address of the error word for the current device (looked up once).
unsigned int *device_error_word() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_mg_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned int *>(p);
  }
  return g_err_ptr[dev];
}

// ---------------------------------------------------------------- profiling
struct ProfState {
  bool enabled = false;
  int capacity = 0;
  int used = 0;
  cudaEvent_t *ev = nullptr;  // 2 * capacity
  int *kid = nullptr;         // kernel id of each pair
};
ProfState g_prof;

struct ProfScope {
  int pair = -1;
  cudaStream_t st;
  ProfScope(int kernel, cudaStream_t s) : st(s) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_prof.enabled || g_prof.used >= g_prof.capacity) return;
    pair = g_prof.used++;
    g_prof.kid[pair] = kernel;
    cudaEventRecord(g_prof.ev[2 * pair], st);
  }
  ~ProfScope() {
    if (pair >= 0) cudaEventRecord(g_prof.ev[2 * pair + 1], st);
  }
};

void prof_free() {
  if (g_prof.ev) {
    for (int i = 0; i < 2 * g_prof.capacity; ++i) cudaEventDestroy(g_prof.ev[i]);
    delete[] g_prof.ev;
    delete[] g_prof.kid;
  }
  g_prof = ProfState();
}

const char *const kKernelNames[MGK_COUNT] = {
    "strict_fwd", "strict_dvec", "strict_dkdv_dq", "accel_fwd",     "accel_dvec",
    "accel_dkdv_dq", "dq_zero",  "accel_dkdv",    "accel_dq",    "decode_fwd",
    "dq_round", "conv_dgrad", "conv_wgrad"};

// How the ACCEL backward produces dQ: f32 TMA reductions from the fused dK/dV
// kernel (default, measured faster on GB300) or a separate dQ pass that
// recomputes S and dP per query block (MG_DQ_MODE=pass). Read once.
bool accel_dq_atomic() {
  static const bool v = [] {
    const char *e = getenv("MG_DQ_MODE");
    return !(e && strcmp(e, "pass") == 0);
  }();
  return v;
}

// ---------------------------------------------------------------- validation
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
  uintptr_t lo, hi;
};
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

int check_common(int B, int H, int Lq, int Lk, int D, int mask, float scale, int contract) {
  if (B < 1 || H < 1 || Lq < 1 || Lk < 1) return MG_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > (1LL << 24) || Lq > (1 << 20) || Lk > (1 << 20))
    return MG_ERR_INVALID_ARG;
  if (mask != MG_MASK_NONE && mask != MG_MASK_CAUSAL && mask != MG_MASK_CAUSAL_BOTTOM_RIGHT)
    return MG_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return MG_ERR_INVALID_ARG;
  const int base = contract & MG_CONTRACT_BASE_MASK, flags = contract & ~MG_CONTRACT_BASE_MASK;
  if (base != MG_CONTRACT_STRICT_F32 && base != MG_CONTRACT_ACCEL_BF16 &&
      base != MG_CONTRACT_ACCEL_F16)
    return MG_ERR_INVALID_ARG;
  if (flags & ~(MG_OUT_16 | MG_DS_HILO)) return MG_ERR_INVALID_ARG;
  // STRICT_F32 is f32 end to end: no 16-bit outputs, no 16-bit dS to split
  if (flags && base == MG_CONTRACT_STRICT_F32) return MG_ERR_UNSUPPORTED;
  if (D != 32 && D != 64 && D != 128) return MG_ERR_UNSUPPORTED;
  return MG_OK;
}

MgProblem make_problem(int B, int H, int Lq, int Lk, int D, int mask, float scale,
                       const int *kv_len = nullptr, int contract = 0) {
  MgProblem p{B, H, Lq, D, mask != MG_MASK_NONE ? 1 : 0, scale, Lk, 0};
  if (mask == MG_MASK_CAUSAL_BOTTOM_RIGHT) p.off = Lk - Lq;
  p.kv_len = kv_len;
  p.br = mask == MG_MASK_CAUSAL_BOTTOM_RIGHT ? 1 : 0;
  p.f16 = (contract & MG_CONTRACT_BASE_MASK) == MG_CONTRACT_ACCEL_F16 ? 1 : 0;
  p.out16 = (contract & MG_OUT_16) ? 1 : 0;
  p.hilo = (contract & MG_DS_HILO) ? 1 : 0;
  return p;
}

bool is_strict(int contract) {
  return (contract & MG_CONTRACT_BASE_MASK) == MG_CONTRACT_STRICT_F32;
}
// Bytes per element of the inputs Q, K, V, dO and of the outputs O, dQ, dK, dV.
size_t in_bytes(int contract) { return is_strict(contract) ? 4 : 2; }
size_t out_bytes(int contract) { return (contract & MG_OUT_16) ? 2 : 4; }

// kv_len (device array of B int32, may be null) must be 4-byte aligned and must
// not overlap any output.
int check_kv_len(const int *kv_len) {
  return (kv_len && (reinterpret_cast<uintptr_t>(kv_len) & 3u) != 0) ? MG_ERR_INVALID_ARG
                                                                     : MG_OK;
}

int check_ptrs(const void *const *ptrs, int n) {
  for (int i = 0; i < n; ++i)
    if (!ptrs[i] || !aligned16(ptrs[i])) return MG_ERR_INVALID_ARG;
  return MG_OK;
}

// Outputs must not overlap inputs or each other.
int check_alias(const Range *in, int nin, const Range *out, int nout) {
  for (int o = 0; o < nout; ++o) {
    for (int i = 0; i < nin; ++i)
      if (overlap(out[o], in[i])) return MG_ERR_INVALID_ARG;
    for (int p = o + 1; p < nout; ++p)
      if (overlap(out[o], out[p])) return MG_ERR_INVALID_ARG;
  }
  return MG_OK;
}

Range rng(const void *p, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Range{a, a + bytes};
}

int map_cuda(cudaError_t e) { return e == cudaSuccess ? MG_OK : MG_ERR_CUDA; }

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Backward workspace: Dvec [B][H][Lq] f32, then for 16-bit outputs an f32 dQ
// accumulator [B][H][Lq][D] (the reductions add in f32; one pass rounds it).
size_t dvec_ws_bytes(int B, int H, int L) {
  return round256(static_cast<size_t>(B) * H * L * sizeof(float));
}
size_t ws_bytes(int B, int H, int L, int D = 0, int contract = 0) {
  size_t b = dvec_ws_bytes(B, H, L);
  if (contract & MG_OUT_16) b += round256(static_cast<size_t>(B) * H * L * D * sizeof(float));
  return b;
}

}  // namespace

uint64_t mg_wait_limit_ns() {
  static const uint64_t v = [] {
    const char *e = getenv("MG_WAIT_TIMEOUT_MS");
    long long ms = e ? atoll(e) : 4000;
    if (ms < 1) ms = 1;
    return static_cast<uint64_t>(ms) * 1000000ull;
  }();
  return v;
}

int mg_check_args(int B, int H, int Lq, int Lk, int D, int mask, float scale, int contract) {
  return check_common(B, H, Lq, Lk, D, mask, scale, contract);
}

int mg_sm_count() {
  static int cached[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 152;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 152;
    cached[dev] = n;
  }
  return cached[dev];
}

cudaError_t mg_set_smem_attr(const void *func, int bytes, int slot) {
  const int dev = current_device();
  if (dev < 0) return cudaErrorNoDevice;
  if (dev >= kMaxDevices || slot < 0 || slot >= kMaxSlots)
    return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_smem_done[dev][slot]) return cudaSuccess;
  }
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_smem_done[dev][slot] = true;
  }
  return e;
}

// ---------------------------------------------------------------- convolution derivatives
namespace {

// Shape and contract checks shared by both convolution derivatives.
int conv_problem(int N, int H, int W, int C, int K, int R, int S, int stride, int pad,
                 int contract, MgConvProblem *p) {
  if (N < 1 || H < 1 || W < 1 || C < 1 || K < 1 || R < 1 || S < 1 || pad < 0)
    return MG_ERR_INVALID_ARG;
  if (H > 65535 || W > 65535 || R > 64 || S > 64 || pad > 64) return MG_ERR_INVALID_ARG;
  if (stride != 1 && stride != 2) return (stride < 1) ? MG_ERR_INVALID_ARG : MG_ERR_UNSUPPORTED;
  if (H + 2 * pad < R || W + 2 * pad < S) return MG_ERR_INVALID_ARG;
  const int base = contract & MG_CONTRACT_BASE_MASK, flags = contract & ~MG_CONTRACT_BASE_MASK;
  if (base != MG_CONTRACT_STRICT_F32 && base != MG_CONTRACT_ACCEL_BF16 &&
      base != MG_CONTRACT_ACCEL_F16)
    return MG_ERR_INVALID_ARG;
  if (flags & ~(MG_OUT_16 | MG_DS_HILO)) return MG_ERR_INVALID_ARG;
  // tensor cores only, f32 results; channel counts in whole 16-byte rows
  if (base == MG_CONTRACT_STRICT_F32 || flags) return MG_ERR_UNSUPPORTED;
  if (C % 8 != 0 || K % 8 != 0) return MG_ERR_UNSUPPORTED;
  const int P = (H + 2 * pad - R) / stride + 1, Q = (W + 2 * pad - S) / stride + 1;
  const long long lim = 0x7fffffffLL;
  if (static_cast<long long>(N) * H * W * C > lim || static_cast<long long>(N) * P * Q * K > lim ||
      static_cast<long long>(K) * R * S * C > lim)
    return MG_ERR_INVALID_ARG;
  // grid limits of the weight gradient (R*S taps, K/128 x C/64 channel blocks)
  if (static_cast<long long>((K + 127) / 128) * ((C + 63) / 64) > 65535) return MG_ERR_UNSUPPORTED;
  *p = MgConvProblem{N, H, W, C, K, R, S, stride, pad, P, Q,
                     base == MG_CONTRACT_ACCEL_F16 ? 1 : 0};
  return MG_OK;
}

}  // namespace

extern "C" {

const char *mg_status_string(int status) {
  switch (status) {
    case MG_OK: return "MG_OK";
    case MG_ERR_INVALID_ARG: return "MG_ERR_INVALID_ARG: invalid argument";
    case MG_ERR_UNSUPPORTED: return "MG_ERR_UNSUPPORTED: head dim must be 32, 64 or 128";
    case MG_ERR_WORKSPACE: return "MG_ERR_WORKSPACE: workspace missing or too small";
    case MG_ERR_CUDA: return "MG_ERR_CUDA: CUDA runtime error";
    case MG_ERR_TIMEOUT: return "MG_ERR_TIMEOUT: a kernel gave up on a bounded wait";
    default: return "unknown mg_status_t";
  }
}

int mg_attn_fwd_padded(const void *Q, const void *K, const void *V, void *O, float *LSE,
                       const int *kv_len, int B, int H, int Lq, int Lk, int D, int mask,
                       float scale, int contract, void *stream) {
  int rc = check_common(B, H, Lq, Lk, D, mask, scale, contract);
  if (rc) return rc;
  const void *ptrs[] = {Q, K, V, O, LSE};
  if ((rc = check_ptrs(ptrs, 5))) return rc;
  if ((rc = check_kv_len(kv_len))) return rc;
  const size_t nq = static_cast<size_t>(B) * H * Lq * D;
  const size_t nk = static_cast<size_t>(B) * H * Lk * D;
  const size_t in_el = in_bytes(contract), out_el = out_bytes(contract);
  const Range in[] = {rng(Q, nq * in_el), rng(K, nk * in_el), rng(V, nk * in_el),
                      rng(kv_len, kv_len ? static_cast<size_t>(B) * 4 : 0)};
  const Range out[] = {rng(O, nq * out_el), rng(LSE, static_cast<size_t>(B) * H * Lq * 4)};
  if ((rc = check_alias(in, 4, out, 2))) return rc;

  const MgProblem p = make_problem(B, H, Lq, Lk, D, mask, scale, kv_len, contract);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (is_strict(contract)) {
    ProfScope ps(MGK_STRICT_FWD, st);
    e = mg_launch_strict_fwd(static_cast<const float *>(Q), static_cast<const float *>(K),
                             static_cast<const float *>(V), static_cast<float *>(O), LSE, p, st);
  } else {
    unsigned int *err = device_error_word();
    if (!err) return MG_ERR_CUDA;
    ProfScope ps(MGK_ACCEL_FWD, st);
    e = mg_launch_accel_fwd(Q, K, V, O, LSE, p, err, st);
  }
  return map_cuda(e);
}

int mg_attn_fwd_ex(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                   int H, int Lq, int Lk, int D, int mask, float scale, int contract,
                   void *stream) {
  return mg_attn_fwd_padded(Q, K, V, O, LSE, nullptr, B, H, Lq, Lk, D, mask, scale, contract,
                            stream);
}

int mg_attn_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                int L, int D, int causal, float scale, int contract, void *stream) {
  if (causal != 0 && causal != 1) return MG_ERR_INVALID_ARG;
  return mg_attn_fwd_ex(Q, K, V, O, LSE, B, H, L, L, D, causal ? MG_MASK_CAUSAL : MG_MASK_NONE,
                        scale, contract, stream);
}

size_t mg_attn_fwd_decode_workspace_bytes(int B, int H, int Lq, int Lk, int D, int contract) {
  if (check_common(B, H, Lq, Lk, D, MG_MASK_NONE, 1.f, contract) != MG_OK) return 0;
  if (Lq > mg_decode_max_rows()) return 0;
  const MgProblem p = make_problem(B, H, Lq, Lk, D, MG_MASK_NONE, 1.f);
  return (mg_decode_workspace_floats(p, !is_strict(contract)) * sizeof(float) + 255) &
         ~static_cast<size_t>(255);
}

int mg_attn_fwd_decode(const void *Q, const void *K, const void *V, void *O, float *LSE, int B,
                       int H, int Lq, int Lk, int D, int mask, float scale, int contract,
                       void *workspace, size_t workspace_bytes, void *stream) {
  int rc = check_common(B, H, Lq, Lk, D, mask, scale, contract);
  if (rc) return rc;
  if (Lq > mg_decode_max_rows()) return MG_ERR_UNSUPPORTED;
  if (contract & MG_OUT_16) return MG_ERR_UNSUPPORTED;  // O is f32 here
  const void *ptrs[] = {Q, K, V, O, LSE};
  if ((rc = check_ptrs(ptrs, 5))) return rc;
  const size_t need = mg_attn_fwd_decode_workspace_bytes(B, H, Lq, Lk, D, contract);
  if (!workspace || !aligned16(workspace) || workspace_bytes < need) return MG_ERR_WORKSPACE;
  const size_t nq = static_cast<size_t>(B) * H * Lq * D;
  const size_t nk = static_cast<size_t>(B) * H * Lk * D;
  const size_t in_el = in_bytes(contract);
  const Range in[] = {rng(Q, nq * in_el), rng(K, nk * in_el), rng(V, nk * in_el)};
  const Range out[] = {rng(O, nq * 4), rng(LSE, static_cast<size_t>(B) * H * Lq * 4),
                       rng(workspace, need)};
  if ((rc = check_alias(in, 3, out, 3))) return rc;
  const MgProblem p = make_problem(B, H, Lq, Lk, D, mask, scale, nullptr, contract);
  unsigned int *err = device_error_word();
  if (!err) return MG_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ProfScope ps(MGK_DECODE_FWD, st);
  return map_cuda(mg_launch_decode_fwd(Q, K, V, static_cast<float *>(O), LSE,
                                       static_cast<float *>(workspace), p,
                                       contract & MG_CONTRACT_BASE_MASK, err, st));
}

size_t mg_attn_bwd_workspace_bytes_ex(int B, int H, int Lq, int Lk, int D, int contract) {
  if (check_common(B, H, Lq, Lk, D, MG_MASK_NONE, 1.f, contract) != MG_OK) return 0;
  return ws_bytes(B, H, Lq, D, contract);
}

size_t mg_attn_bwd_workspace_bytes(int B, int H, int L, int D, int contract) {
  return mg_attn_bwd_workspace_bytes_ex(B, H, L, L, D, contract);
}

int mg_attn_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int L, int D,
                int causal, float scale, int contract, void *workspace, size_t workspace_bytes,
                void *stream) {
  if (causal != 0 && causal != 1) return MG_ERR_INVALID_ARG;
  return mg_attn_bwd_ex(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, L, L, D,
                        causal ? MG_MASK_CAUSAL : MG_MASK_NONE, scale, contract, workspace,
                        workspace_bytes, stream);
}

int mg_attn_bwd_ex(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                   const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int Lq, int Lk,
                   int D, int mask, float scale, int contract, void *workspace,
                   size_t workspace_bytes, void *stream) {
  return mg_attn_bwd_padded(Q, K, V, O, dO, LSE, dQ, dK, dV, nullptr, B, H, Lq, Lk, D, mask,
                            scale, contract, workspace, workspace_bytes, stream);
}

int mg_attn_bwd_padded(const void *Q, const void *K, const void *V, const void *O,
                       const void *dO, const float *LSE, void *dQ, void *dK, void *dV,
                       const int *kv_len, int B, int H, int Lq, int Lk, int D, int mask,
                       float scale, int contract, void *workspace, size_t workspace_bytes,
                       void *stream) {
  int rc = check_common(B, H, Lq, Lk, D, mask, scale, contract);
  if (rc) return rc;
  const void *ptrs[] = {Q, K, V, O, dO, LSE, dQ, dK, dV};
  if ((rc = check_ptrs(ptrs, 9))) return rc;
  if ((rc = check_kv_len(kv_len))) return rc;
  const size_t need = ws_bytes(B, H, Lq, D, contract);
  if (!workspace || !aligned16(workspace) || workspace_bytes < need) return MG_ERR_WORKSPACE;
  const size_t n = static_cast<size_t>(B) * H * Lq * D;   // Q, O, dO, dQ
  const size_t nk = static_cast<size_t>(B) * H * Lk * D;  // K, V, dK, dV
  const size_t rows = static_cast<size_t>(B) * H * Lq;
  const size_t in_el = in_bytes(contract), out_el = out_bytes(contract);
  const Range in[] = {rng(Q, n * in_el), rng(K, nk * in_el), rng(V, nk * in_el),
                      rng(dO, n * in_el), rng(O, n * out_el), rng(LSE, rows * 4),
                      rng(kv_len, kv_len ? static_cast<size_t>(B) * 4 : 0)};
  const Range out[] = {rng(dQ, n * out_el), rng(dK, nk * out_el), rng(dV, nk * out_el),
                       rng(workspace, need)};
  if ((rc = check_alias(in, 7, out, 4))) return rc;

  const MgProblem p = make_problem(B, H, Lq, Lk, D, mask, scale, kv_len, contract);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float *Dvec = static_cast<float *>(workspace);
  cudaError_t e;
  if (is_strict(contract)) {
    {
      ProfScope ps(MGK_STRICT_DVEC, st);
      e = mg_launch_dvec_f32(static_cast<const float *>(O), static_cast<const float *>(dO), Dvec,
                             p, st);
    }
    if (e != cudaSuccess) return MG_ERR_CUDA;
    {
      ProfScope ps(MGK_DQ_ZERO, st);
      e = cudaMemsetAsync(dQ, 0, n * 4, st);
    }
    if (e != cudaSuccess) return MG_ERR_CUDA;
    ProfScope ps(MGK_STRICT_DKDV, st);
    e = mg_launch_strict_dkdv(static_cast<const float *>(Q), static_cast<const float *>(K),
                              static_cast<const float *>(V), static_cast<const float *>(dO), LSE,
                              Dvec, static_cast<float *>(dQ), static_cast<float *>(dK),
                              static_cast<float *>(dV), p, st);
  } else {
    unsigned int *err = device_error_word();
    if (!err) return MG_ERR_CUDA;
    {
      ProfScope ps(MGK_ACCEL_DVEC, st);
      e = mg_launch_dvec_16(O, dO, Dvec, p, st);
    }
    if (e != cudaSuccess) return MG_ERR_CUDA;
    // the hi/lo dS policy runs in the two-pass backward, where both parts of dS
    // are tensor-memory operands of the dK and dQ products
    if (accel_dq_atomic() && !p.hilo) {
      // the reductions add into f32: the caller's dQ, or for 16-bit outputs an
      // f32 accumulator in the workspace that one pass rounds into dQ at the end
      float *dq_acc = p.out16 ? reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                                          dvec_ws_bytes(B, H, Lq))
                              : static_cast<float *>(dQ);
      {
        ProfScope ps(MGK_DQ_ZERO, st);
        e = cudaMemsetAsync(dq_acc, 0, n * 4, st);
      }
      if (e != cudaSuccess) return MG_ERR_CUDA;
      {
        ProfScope ps(MGK_ACCEL_DKDV_DQ, st);
        e = mg_launch_accel_dkdv(Q, K, V, dO, LSE, Dvec, dq_acc, dK, dV, p, err, st);
      }
      if (e != cudaSuccess || !p.out16) return map_cuda(e);
      ProfScope ps(MGK_DQ_ROUND, st);
      e = mg_launch_f32_to_16(dq_acc, dQ, n, p.f16 != 0, st);
    } else {
      {
        ProfScope ps(MGK_ACCEL_DKDV, st);
        e = mg_launch_accel_dkdv_pp(Q, K, V, dO, LSE, Dvec, dK, dV, p, err, st);
      }
      if (e != cudaSuccess) return MG_ERR_CUDA;
      ProfScope ps(MGK_ACCEL_DQ, st);
      e = mg_launch_accel_dq(Q, K, V, dO, LSE, Dvec, dQ, p, err, st);
    }
  }
  return map_cuda(e);
}

int mg_get_device_error(void *stream) {
  unsigned int *err = device_error_word();
  if (!err) return MG_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned int h = 0;
  if (cudaMemcpyAsync(&h, err, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MG_ERR_CUDA;
  if (cudaMemsetAsync(err, 0, sizeof(h), st) != cudaSuccess) return MG_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MG_ERR_CUDA;
  return h == MG_DEVERR_NONE ? MG_OK : MG_ERR_TIMEOUT;
}

int mg_attn_profile_enable(int enable, int capacity) {
  std::lock_guard<std::mutex> lk(g_mu);
  prof_free();
  if (!enable) return MG_OK;
  if (capacity < 1 || capacity > (1 << 20)) return MG_ERR_INVALID_ARG;
  g_prof.ev = new cudaEvent_t[2 * static_cast<size_t>(capacity)];
  g_prof.kid = new int[capacity];
  for (int i = 0; i < 2 * capacity; ++i) {
    if (cudaEventCreate(&g_prof.ev[i]) != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(g_prof.ev[j]);
      delete[] g_prof.ev;
      delete[] g_prof.kid;
      g_prof = ProfState();
      return MG_ERR_CUDA;
    }
  }
  g_prof.capacity = capacity;
  g_prof.enabled = true;
  return MG_OK;
}

int mg_attn_profile_read(int kernel, int *launches, double *total_ms) {
  if (kernel < 0 || kernel >= MGK_COUNT || !launches || !total_ms) return MG_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  int cnt = 0;
  double ms = 0.0;
  for (int i = 0; i < g_prof.used; ++i) {
    if (g_prof.kid[i] != kernel) continue;
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess) return MG_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess)
      return MG_ERR_CUDA;
    ++cnt;
    ms += t;
  }
  *launches = cnt;
  *total_ms = ms;
  return MG_OK;
}

// ---------------------------------------------------------------- convolution derivatives
int mg_conv2d_grad_input(const void *dY, const void *Wt, float *dX, int N, int H, int W, int C,
                         int K, int R, int S, int stride, int pad, int contract, void *stream) {
  MgConvProblem p;
  int rc = conv_problem(N, H, W, C, K, R, S, stride, pad, contract, &p);
  if (rc) return rc;
  const void *ptrs[] = {dY, Wt, dX};
  if ((rc = check_ptrs(ptrs, 3))) return rc;
  const Range in[] = {rng(dY, static_cast<size_t>(N) * p.P * p.Q * K * 2),
                      rng(Wt, static_cast<size_t>(K) * R * S * C * 2)};
  const Range out[] = {rng(dX, static_cast<size_t>(N) * H * W * C * 4)};
  if ((rc = check_alias(in, 2, out, 1))) return rc;
  unsigned int *err = device_error_word();
  if (!err) return MG_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ProfScope ps(MGK_CONV_DGRAD, st);
  return map_cuda(mg_launch_conv_dgrad(dY, Wt, dX, p, err, st));
}

int mg_conv2d_grad_weight(const void *X, const void *dY, float *dW, int N, int H, int W, int C,
                          int K, int R, int S, int stride, int pad, int contract, void *stream) {
  MgConvProblem p;
  int rc = conv_problem(N, H, W, C, K, R, S, stride, pad, contract, &p);
  if (rc) return rc;
  const void *ptrs[] = {X, dY, dW};
  if ((rc = check_ptrs(ptrs, 3))) return rc;
  const size_t nw = static_cast<size_t>(K) * R * S * C;
  const Range in[] = {rng(X, static_cast<size_t>(N) * H * W * C * 2),
                      rng(dY, static_cast<size_t>(N) * p.P * p.Q * K * 2)};
  const Range out[] = {rng(dW, nw * 4)};
  if ((rc = check_alias(in, 2, out, 1))) return rc;
  unsigned int *err = device_error_word();
  if (!err) return MG_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ProfScope ps(MGK_CONV_WGRAD, st);
  cudaError_t e = cudaMemsetAsync(dW, 0, nw * 4, st);
  if (e == cudaSuccess) e = mg_launch_conv_wgrad(X, dY, dW, p, err, st);
  return map_cuda(e);
}

int mg_attn_kernel_count(void) { return MGK_COUNT; }

const char *mg_attn_kernel_name(int kernel) {
  if (kernel < 0 || kernel >= MGK_COUNT) return "unknown";
  return kKernelNames[kernel];
}

}  // extern "C"
