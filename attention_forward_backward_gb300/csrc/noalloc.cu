// noalloc.cu -- mg_attn_bwd_noalloc: the backward for callers that cannot
// allocate device memory at all, not even a workspace of their own.
//
// Some hosts of this library own every byte of device memory and hand out no
// scratch: a plugin inside another runtime whose allocator is closed to it, an
// embedded or real-time service that fixes its memory budget at start-up and
// forbids allocation afterwards, or a caller that must not pay the implicit
// device synchronisation of cudaMalloc. For them the Dvec scratch of the
// backward lives in a fixed, file-scope device array instead of a
// caller-provided workspace.
//
// The array is a module global: every GPU that loads the library keeps it
// (4 MiB) until the process exits. Every call on a device uses the same array,
// so two calls whose kernels overlap on that GPU (different streams, no
// ordering between them) race on it; calls on one stream, or otherwise
// ordered, are safe. The backward writes every Dvec entry it reads before
// reading it, so nothing in the array has to start at zero and the contents a
// previous call left behind do not matter.
//
// Host code cannot use the array's name as a device pointer (it names a host
// stand-in), so the first call on each device looks up the array's device
// address with cudaGetSymbolAddress while that device is current and caches
// it; that first call should therefore happen before any stream capture. The
// cached address belongs to the device's current context: after
// cudaDeviceReset on that device it is stale, so the library must not be used on
// a device that has been reset since its first call there.
//
// Argument errors are reported exactly as mg_attn_bwd reports them (same checks,
// same order); only then is B*H*L compared with the array's size.
#include <mutex>

#include "../../include/mg_attn.h"
#include "internal.h"

namespace {

constexpr long long kNoallocMaxRows = 1LL << 20;  // B*H*L <= 1,048,576 rows
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_dvec[kNoallocMaxRows];

std::mutex g_mu;
float *g_scratch[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per
// device). Returns nullptr if the device cannot be queried.
float *scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_dvec) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch[dev] = static_cast<float *>(p);
  }
  return g_scratch[dev];
}

}  // namespace

extern "C" int mg_attn_bwd_noalloc(const void *Q, const void *K, const void *V, const void *O,
                                   const void *dO, const float *LSE, void *dQ, void *dK,
                                   void *dV, int B, int H, int L, int D, int causal, float scale,
                                   int contract, void *stream) {
  // mg_attn_bwd's own checks first, in its order, so that every argument error
  // reports the same status as there; only then the limit of the fixed array.
  if (causal != 0 && causal != 1) return MG_ERR_INVALID_ARG;
  int rc = mg_check_args(B, H, L, L, D, causal ? MG_MASK_CAUSAL : MG_MASK_NONE, scale, contract);
  if (rc != MG_OK) return rc;
  // the fixed array holds Dvec only, not the f32 dQ accumulator of 16-bit outputs
  if (contract & MG_OUT_16) return MG_ERR_UNSUPPORTED;
  const void *ptrs[] = {Q, K, V, O, dO, LSE, dQ, dK, dV};
  for (const void *p : ptrs)
    if (!p || (reinterpret_cast<uintptr_t>(p) & 15u) != 0) return MG_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * H * L;
  if (rows > kNoallocMaxRows) return MG_ERR_WORKSPACE;  // beyond the fixed scratch
  float *scratch = scratch_on_current_device();
  if (!scratch) return MG_ERR_CUDA;
  return mg_attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, L, D, causal, scale, contract,
                     scratch, static_cast<size_t>(kNoallocMaxRows) * sizeof(float), stream);
}
