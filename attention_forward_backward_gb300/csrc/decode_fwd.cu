// decode_fwd.cu -- attention forward for a few query rows against a long key
// axis (decoding): the key axis is split over many CTAs, each producing a partial
// softmax (running max, sum and unnormalised output per query row), and a second
// kernel merges the partials into O and LSE.
//
// The computation is the forward of the attention node ("Meganeura: Portable GPU
// Training and Inference through Vulkan and Metal", Section 3.1) for Lq <= 8
// query rows. With so few rows the work is one pass over K and V, bound by HBM,
// and the generic kernels leave most SMs idle when there are few heads: splitting
// the keys lets every SM stream its share. Arithmetic is f32 on the CUDA cores for
// both contracts (bf16 inputs are widened on load); scores are in base 2 with
// scale * log2(e) folded into Q, and each split keeps the exact online-softmax
// state, so the merge is exact up to rounding:
//   m = max_s m_s,  l = sum_s l_s 2^(m_s - m),  O = sum_s O_s 2^(m_s - m) / l,
//   LSE = ln 2 (m + log2 l);  a row with no allowed key gets O = 0, LSE = -inf.
#include <math.h>

#include "internal.h"

namespace {

constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;
constexpr int kMaxLq = 8;   // query rows per head handled here
constexpr int kTile = 32;   // keys per shared-memory tile
constexpr int kThreads = 256;

__device__ __forceinline__ float load_in(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_in(const __nv_bfloat16 *p, size_t i) {
  return __bfloat162float(p[i]);
}

// Eight consecutive input elements as raw registers (16-byte loads): fetched one
// tile ahead, widened to f32 when stored to shared memory.
template <typename TIn> struct Raw8;
template <> struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float *p) {
    a = *reinterpret_cast<const float4 *>(p);
    b = *reinterpret_cast<const float4 *>(p + 4);
  }
  __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ void put(float *dst) const {
    dst[0] = a.x; dst[1] = a.y; dst[2] = a.z; dst[3] = a.w;
    dst[4] = b.x; dst[5] = b.y; dst[6] = b.z; dst[7] = b.w;
  }
};
template <> struct Raw8<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16 *p) {
    u = *reinterpret_cast<const uint4 *>(p);
  }
  __device__ __forceinline__ void zero() { u = make_uint4(0u, 0u, 0u, 0u); }
  __device__ __forceinline__ void put(float *dst) const {
    const unsigned w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // bf16 -> f32 is a 16-bit shift
      dst[2 * k] = __uint_as_float(w[k] << 16);
      dst[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One CTA: head bh, keys [k_begin, k_end). Partial record per (bh, split, q):
// [m (base 2), l, O_0 .. O_{D-1}] in `part`.
template <int D, typename TIn>
__global__ void __launch_bounds__(kThreads)
    decode_partial_kernel(const TIn *__restrict__ Q, const TIn *__restrict__ K,
                          const TIn *__restrict__ V, float *__restrict__ part, int Lq, int Lk,
                          int causal, int off, int S, int chunk, float scale_log2) {
  constexpr int KS = D + 1;                       // padded K row: conflict-free column reads
  constexpr int QPT = kMaxLq * D / kThreads;      // output (q, d) cells per thread
  constexpr int QSTEP = kThreads / D;             // q stride between a thread's cells
  constexpr int CH = kTile * D / 8;               // 8-element chunks per tile of K (and V)
  constexpr int CPT = (CH + kThreads - 1) / kThreads;
  static_assert(QPT >= 1 && kThreads % D == 0 && D % 8 == 0, "layout");
  __shared__ float sQ[kMaxLq][D];
  __shared__ float sK[kTile][KS];
  __shared__ float sV[kTile][D];
  __shared__ float sP[kMaxLq][kTile];
  __shared__ float sAlpha[kMaxLq];

  const int bh = blockIdx.x / S, s = blockIdx.x % S;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k_begin = s * chunk;
  const int k_end = min(Lk, k_begin + chunk);
  const size_t qbase = static_cast<size_t>(bh) * Lq * D;
  const size_t kbase = static_cast<size_t>(bh) * Lk * D;

  for (int i = tid; i < kMaxLq * D; i += kThreads) {
    const int q = i / D, d = i % D;
    sQ[q][d] = q < Lq ? load_in(Q, qbase + static_cast<size_t>(q) * D + d) * scale_log2 : 0.f;
  }
  // running state: warp q owns m, l of query q; thread owns O cells (q0 + j QSTEP, dd)
  float m = -INFINITY, l = 0.f;
  float o[QPT];
#pragma unroll
  for (int j = 0; j < QPT; ++j) o[j] = 0.f;
  const int dd = tid % D, q0 = tid / D;

  // K and V chunks of the next tile, in flight while the current one is used
  Raw8<TIn> rk[CPT], rv[CPT];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      const int i = tid + c * kThreads, r = i / (D / 8);
      if (i < CH && k0 + r < k_end) {
        const size_t g = kbase + static_cast<size_t>(k0 + r) * D + (i % (D / 8)) * 8;
        rk[c].load(K + g);
        rv[c].load(V + g);
      } else {
        rk[c].zero();
        rv[c].zero();
      }
    }
  };
  fetch(k_begin);

  for (int k0 = k_begin; k0 < k_end; k0 += kTile) {
    __syncthreads();  // previous tile fully consumed (and sQ written, first time)
    const int nk = min(kTile, k_end - k0);
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      const int i = tid + c * kThreads;
      if (i < CH) {
        const int r = i / (D / 8), d = (i % (D / 8)) * 8;
        rk[c].put(&sK[r][d]);
        rv[c].put(&sV[r][d]);
      }
    }
    if (k0 + kTile < k_end) fetch(k0 + kTile);
    __syncthreads();
    // scores: warp q (< Lq) -> query q, lane -> key k0 + lane
    if (warp < Lq) {
      const int q = warp, j = lane;
      float sc = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) sc = fmaf(sQ[q][d], sK[j][d], sc);
      const int kg = k0 + j;
      const bool allowed = j < nk && (!causal || kg <= q + off);
      sP[q][j] = allowed ? sc : -INFINITY;
    }
    __syncthreads();
    // online softmax: warp q updates query q's state over the tile's 32 keys
    if (warp < Lq) {
      const float x = sP[warp][lane];
      const float mt = warp_max(x);
      const float mn = fmaxf(m, mt);
      const float mu = mn == -INFINITY ? 0.f : mn;  // no allowed key yet: P = 0
      const float p = exp2f(x - mu);
      const float alpha = exp2f(m - mu);
      l = l * alpha + warp_sum(p);
      m = mn;
      sP[warp][lane] = p;
      if (lane == 0) sAlpha[warp] = alpha;
    }
    __syncthreads();
    // O[q][dd] = alpha_q O[q][dd] + sum_j P[q][j] V[j][dd]
#pragma unroll
    for (int jq = 0; jq < QPT; ++jq) {
      const int q = q0 + jq * QSTEP;
      if (q < Lq) {
        float acc = o[jq] * sAlpha[q];
#pragma unroll 8
        for (int j = 0; j < kTile; ++j) acc = fmaf(sP[q][j], sV[j][dd], acc);
        o[jq] = acc;
      }
    }
  }

  // partial record of this split
  float *rec = part + (static_cast<size_t>(bh) * S + s) * Lq * (D + 2);
  if (warp < Lq && lane == 0) {
    rec[warp * (D + 2)] = m;
    rec[warp * (D + 2) + 1] = l;
  }
#pragma unroll
  for (int jq = 0; jq < QPT; ++jq) {
    const int q = q0 + jq * QSTEP;
    if (q < Lq) rec[q * (D + 2) + 2 + dd] = o[jq];
  }
}

// One CTA of D threads per (bh, q): merge the S partial records.
template <int D>
__global__ void __launch_bounds__(128)
    decode_merge_kernel(const float *__restrict__ part, float *__restrict__ O,
                        float *__restrict__ LSE, int Lq, int S) {
  const int bh = blockIdx.x / Lq, q = blockIdx.x % Lq;
  const int d = threadIdx.x;
  const float *rec = part + static_cast<size_t>(bh) * S * Lq * (D + 2) + q * (D + 2);
  const size_t stride = static_cast<size_t>(Lq) * (D + 2);
  float mmax = -INFINITY;
  for (int s = 0; s < S; ++s) mmax = fmaxf(mmax, rec[s * stride]);
  float lsum = 0.f, acc = 0.f;
  if (mmax != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const float w = exp2f(rec[s * stride] - mmax);  // an empty split has m = -inf: w = 0
      lsum = fmaf(rec[s * stride + 1], w, lsum);
      acc = fmaf(rec[s * stride + 2 + d], w, acc);
    }
  }
  const size_t row = static_cast<size_t>(bh) * Lq + q;
  O[row * D + d] = lsum > 0.f ? acc / lsum : 0.f;
  if (d == 0) LSE[row] = lsum > 0.f ? (mmax + log2f(lsum)) * kLn2F : -INFINITY;
}

template <int D, typename TIn>
cudaError_t launch(const TIn *Q, const TIn *K, const TIn *V, float *O, float *LSE, float *part,
                   const MgProblem &p, int S, int chunk, cudaStream_t st) {
  const int BH = p.B * p.H;
  decode_partial_kernel<D, TIn><<<static_cast<unsigned>(static_cast<long long>(BH) * S),
                                  kThreads, 0, st>>>(Q, K, V, part, p.L, p.Lk, p.causal, p.off,
                                                     S, chunk, p.scale * kLog2eF);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_merge_kernel<D><<<static_cast<unsigned>(static_cast<long long>(BH) * p.L), D, 0, st>>>(
      part, O, LSE, p.L, S);
  return cudaGetLastError();
}

}  // namespace

int mg_decode_max_rows() { return kMaxLq; }

// Splits of the key axis: about four CTAs per SM of a 152-SM GB300, at least 256
// keys per split. Depends only on the shape (the workspace size uses it too).
void mg_decode_split(const MgProblem &p, int *S, int *chunk) {
  const long long BH = static_cast<long long>(p.B) * p.H;
  const int want = static_cast<int>((4LL * 152 + BH - 1) / BH);
  const int maxs = (p.Lk + 255) / 256;
  int s = want < 1 ? 1 : want;
  if (s > maxs) s = maxs;
  if (s > 256) s = 256;
  const int c = ((p.Lk + s - 1) / s + kTile - 1) / kTile * kTile;
  *S = (p.Lk + c - 1) / c;
  *chunk = c;
}

size_t mg_decode_workspace_floats(const MgProblem &p) {
  int S, chunk;
  mg_decode_split(p, &S, &chunk);
  return static_cast<size_t>(p.B) * p.H * S * p.L * (p.D + 2);
}

cudaError_t mg_launch_decode_fwd(const void *Q, const void *K, const void *V, float *O,
                                 float *LSE, float *part, const MgProblem &p, bool bf16,
                                 cudaStream_t st) {
  int S, chunk;
  mg_decode_split(p, &S, &chunk);
  if (bf16) {
    using T = __nv_bfloat16;
    const T *q = static_cast<const T *>(Q), *k = static_cast<const T *>(K),
            *v = static_cast<const T *>(V);
    switch (p.D) {
      case 32: return launch<32, T>(q, k, v, O, LSE, part, p, S, chunk, st);
      case 64: return launch<64, T>(q, k, v, O, LSE, part, p, S, chunk, st);
      case 128: return launch<128, T>(q, k, v, O, LSE, part, p, S, chunk, st);
      default: return cudaErrorInvalidValue;
    }
  }
  const float *q = static_cast<const float *>(Q), *k = static_cast<const float *>(K),
              *v = static_cast<const float *>(V);
  switch (p.D) {
    case 32: return launch<32, float>(q, k, v, O, LSE, part, p, S, chunk, st);
    case 64: return launch<64, float>(q, k, v, O, LSE, part, p, S, chunk, st);
    case 128: return launch<128, float>(q, k, v, O, LSE, part, p, S, chunk, st);
    default: return cudaErrorInvalidValue;
  }
}
