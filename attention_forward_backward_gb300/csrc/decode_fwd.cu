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
// both contracts (bf16 inputs are widened on load) with K, V and Q held in
// registers, never staged in shared memory; scores are in base 2 with
// scale * log2(e) folded into Q, and every partial state is the exact
// online-softmax state of its keys, so merging is exact up to rounding:
//   m = max_s m_s,  l = sum_s l_s 2^(m_s - m),  O = sum_s O_s 2^(m_s - m) / l,
//   LSE = ln 2 (m + log2 l);  a row with no allowed key gets O = 0, LSE = -inf.
#include <math.h>

#include <cuda_fp16.h>

#include "internal.h"

namespace {

constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;
constexpr int kMaxLq = 8;   // query rows per head handled here
constexpr int kTile = 32;   // split lengths are whole multiples of this many keys
constexpr int kThreads = 128;

__device__ __forceinline__ float load_in(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float load_in(const __nv_bfloat16 *p, size_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ float load_in(const __half *p, size_t i) { return __half2float(p[i]); }

// Eight consecutive input elements as raw registers (16-byte loads): fetched one
// step ahead, widened to f32 registers when the step uses them.
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

template <> struct Raw8<__half> {
  uint4 u;
  __device__ __forceinline__ void load(const __half *p) { u = *reinterpret_cast<const uint4 *>(p); }
  __device__ __forceinline__ void zero() { u = make_uint4(0u, 0u, 0u, 0u); }
  __device__ __forceinline__ void put(float *dst) const {
    const unsigned w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[k]));
      dst[2 * k] = f.x;
      dst[2 * k + 1] = f.y;
    }
  }
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One CTA of four warps: head bh, keys [k_begin, k_end). Nothing is staged in
// shared memory: a key row of D elements is spread over LPR = D / 8 lanes (eight
// consecutive elements each, one 16-byte load for bf16, two for f32), so a warp
// reads RPW = 32 / LPR whole rows per load, coalesced. Each group of LPR lanes
// keeps its own online-softmax state (m, l, O slice) for every query row; Q lives
// in registers. The next kUnroll rows per group are in flight while the current
// ones are used. At the end the CTA's G = 4 RPW states are combined in shared
// memory into one partial record per query row:
//   [O_0 .. O_{D-1} (unnormalised, relative to m), m (base 2), l, -, -].
template <int D, int LQ, typename TIn>
__global__ void __launch_bounds__(kThreads)
    decode_partial_kernel(const TIn *__restrict__ Q, const TIn *__restrict__ K,
                          const TIn *__restrict__ V, float *__restrict__ part, int Lq, int Lk,
                          int causal, int off, int S, int chunk, float scale_log2) {
  constexpr int LPR = D / 8;
  constexpr int RPW = 32 / LPR;
  constexpr int G = (kThreads / 32) * RPW;
  constexpr int U = LQ >= 8 ? 2 : 4;  // rows per group per step (register budget)
  constexpr int STEP = G * U;         // keys per CTA step
  __shared__ float sM[LQ][G], sL[LQ][G];
  __shared__ float sO[LQ][G][D];

  const int bh = blockIdx.x / S, s = blockIdx.x % S;
  const int tid = threadIdx.x, lane = tid & 31;
  const int c = lane % LPR;                          // elements 8c .. 8c+7 of a row
  const int grp = (tid >> 5) * RPW + lane / LPR;     // this lane's softmax state
  const int k_begin = s * chunk;
  const int k_end = min(Lk, k_begin + chunk);
  const TIn *Kb = K + static_cast<size_t>(bh) * Lk * D + c * 8;
  const TIn *Vb = V + static_cast<size_t>(bh) * Lk * D + c * 8;

  float qr[LQ][8], o[LQ][8], m[LQ], l[LQ];
#pragma unroll
  for (int q = 0; q < LQ; ++q) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      qr[q][e] = q < Lq
          ? load_in(Q, (static_cast<size_t>(bh) * Lq + q) * D + c * 8 + e) * scale_log2
          : 0.f;
      o[q][e] = 0.f;
    }
    m[q] = -INFINITY;
    l[q] = 0.f;
  }

  Raw8<TIn> rk[U], rv[U];
  auto fetch = [&](int kb) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int row = kb + u * G + grp;
      if (row < k_end) {
        rk[u].load(Kb + static_cast<size_t>(row) * D);
        rv[u].load(Vb + static_cast<size_t>(row) * D);
      } else {
        rk[u].zero();
        rv[u].zero();
      }
    }
  };
  fetch(k_begin);

  for (int kb = k_begin; kb < k_end; kb += STEP) {
    float kf[U][8], vf[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      rk[u].put(kf[u]);
      rv[u].put(vf[u]);
    }
    if (kb + STEP < k_end) fetch(kb + STEP);
    // scores (base 2): partial dot over this lane's 8 elements, summed over the
    // LPR lanes of the row (xor offsets below LPR stay inside the group)
    float sc[U][LQ];
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int q = 0; q < LQ; ++q) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) a = fmaf(qr[q][e], kf[u][e], a);
        sc[u][q] = a;
      }
    }
#pragma unroll
    for (int w = LPR / 2; w >= 1; w >>= 1) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int q = 0; q < LQ; ++q) sc[u][q] += __shfl_xor_sync(0xffffffffu, sc[u][q], w);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int key = kb + u * G + grp;
#pragma unroll
      for (int q = 0; q < LQ; ++q) {
        const bool allowed = key < k_end && q < Lq && (!causal || key <= q + off);
        if (!allowed) sc[u][q] = -INFINITY;
      }
    }
    // online softmax of each query row over this group's U keys
#pragma unroll
    for (int q = 0; q < LQ; ++q) {
      float mt = sc[0][q];
#pragma unroll
      for (int u = 1; u < U; ++u) mt = fmaxf(mt, sc[u][q]);
      const float mn = fmaxf(m[q], mt);
      const float mu = mn == -INFINITY ? 0.f : mn;  // no allowed key yet: P = 0
      const float alpha = exp2f(m[q] - mu);
      float ps = 0.f;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        sc[u][q] = exp2f(sc[u][q] - mu);
        ps += sc[u][q];
      }
      l[q] = l[q] * alpha + ps;
      m[q] = mn;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float a = o[q][e] * alpha;
#pragma unroll
        for (int u = 0; u < U; ++u) a = fmaf(sc[u][q], vf[u][e], a);
        o[q][e] = a;
      }
    }
  }

  // combine the CTA's G states: the lanes of a group hold the same m and l
#pragma unroll
  for (int q = 0; q < LQ; ++q) {
    if (c == 0) {
      sM[q][grp] = m[q];
      sL[q][grp] = l[q];
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) sO[q][grp][c * 8 + e] = o[q][e];
  }
  __syncthreads();
  float *rec = part + (static_cast<size_t>(bh) * S + s) * Lq * (D + 4);
  for (int i = tid; i < Lq * D; i += kThreads) {
    const int q = i / D, d = i % D;
    float mx = -INFINITY;
#pragma unroll 8
    for (int g = 0; g < G; ++g) mx = fmaxf(mx, sM[q][g]);
    float ls = 0.f, acc = 0.f;
    if (mx != -INFINITY) {
#pragma unroll 8
      for (int g = 0; g < G; ++g) {
        const float w = exp2f(sM[q][g] - mx);  // a state that saw no allowed key: w = 0
        ls = fmaf(sL[q][g], w, ls);
        acc = fmaf(sO[q][g][d], w, acc);
      }
    }
    rec[q * (D + 4) + d] = acc;
    if (d == 0) {
      rec[q * (D + 4) + D] = mx;
      rec[q * (D + 4) + D + 1] = ls;
    }
  }
}

// One CTA per (bh, q): merge the S partial records. Thread (slot, c4) adds the
// records of splits slot, slot + SLOTS, ... for elements 4 c4 .. 4 c4 + 3; the
// slots are summed in shared memory.
template <int D>
__global__ void __launch_bounds__(kThreads)
    decode_merge_kernel(const float *__restrict__ part, float *__restrict__ O,
                        float *__restrict__ LSE, int Lq, int S) {
  constexpr int TPR = D / 4;
  constexpr int SLOTS = kThreads / TPR;
  __shared__ float sRed[kThreads / 32];
  __shared__ float sAcc[SLOTS][D];
  __shared__ float sL[SLOTS];
  const int bh = blockIdx.x / Lq, q = blockIdx.x % Lq;
  const int tid = threadIdx.x, slot = tid / TPR, c4 = tid % TPR;
  const size_t rstride = static_cast<size_t>(Lq) * (D + 4);
  const float *rec0 = part + static_cast<size_t>(bh) * S * rstride + q * (D + 4);

  float mx = -INFINITY;
  for (int s = tid; s < S; s += kThreads) mx = fmaxf(mx, rec0[s * rstride + D]);
  mx = warp_max(mx);
  if ((tid & 31) == 0) sRed[tid >> 5] = mx;
  __syncthreads();
  mx = sRed[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) mx = fmaxf(mx, sRed[w]);

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float ls = 0.f;
  if (mx != -INFINITY) {
#pragma unroll 4
    for (int s = slot; s < S; s += SLOTS) {
      const float *r = rec0 + s * rstride;
      const float w = exp2f(r[D] - mx);  // a split with no allowed key has m = -inf: w = 0
      ls = fmaf(r[D + 1], w, ls);
      const float4 v = *reinterpret_cast<const float4 *>(r + 4 * c4);
      acc.x = fmaf(v.x, w, acc.x);
      acc.y = fmaf(v.y, w, acc.y);
      acc.z = fmaf(v.z, w, acc.z);
      acc.w = fmaf(v.w, w, acc.w);
    }
  }
  sAcc[slot][4 * c4] = acc.x;
  sAcc[slot][4 * c4 + 1] = acc.y;
  sAcc[slot][4 * c4 + 2] = acc.z;
  sAcc[slot][4 * c4 + 3] = acc.w;
  if (c4 == 0) sL[slot] = ls;
  __syncthreads();
  const size_t row = static_cast<size_t>(bh) * Lq + q;
  float lsum = 0.f;
#pragma unroll
  for (int k = 0; k < SLOTS; ++k) lsum += sL[k];
  for (int d = tid; d < D; d += kThreads) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < SLOTS; ++k) t += sAcc[k][d];
    O[row * D + d] = lsum > 0.f ? t / lsum : 0.f;
  }
  if (tid == 0) LSE[row] = lsum > 0.f ? (mx + log2f(lsum)) * kLn2F : -INFINITY;
}

template <int D, int LQ, typename TIn>
cudaError_t launch(const TIn *Q, const TIn *K, const TIn *V, float *O, float *LSE, float *part,
                   const MgProblem &p, int S, int chunk, cudaStream_t st) {
  const int BH = p.B * p.H;
  decode_partial_kernel<D, LQ, TIn>
      <<<static_cast<unsigned>(static_cast<long long>(BH) * S), kThreads, 0, st>>>(
          Q, K, V, part, p.L, p.Lk, p.causal, p.off, S, chunk, p.scale * kLog2eF);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_merge_kernel<D><<<static_cast<unsigned>(static_cast<long long>(BH) * p.L), kThreads, 0,
                           st>>>(part, O, LSE, p.L, S);
  return cudaGetLastError();
}

template <int D, typename TIn>
cudaError_t launch_rows(const TIn *Q, const TIn *K, const TIn *V, float *O, float *LSE,
                        float *part, const MgProblem &p, int S, int chunk, cudaStream_t st) {
  if (p.L <= 1) return launch<D, 1, TIn>(Q, K, V, O, LSE, part, p, S, chunk, st);
  if (p.L <= 2) return launch<D, 2, TIn>(Q, K, V, O, LSE, part, p, S, chunk, st);
  if (p.L <= 4) return launch<D, 4, TIn>(Q, K, V, O, LSE, part, p, S, chunk, st);
  return launch<D, 8, TIn>(Q, K, V, O, LSE, part, p, S, chunk, st);
}

}  // namespace

int mg_decode_max_rows() { return kMaxLq; }

// Splits of the key axis: about eight CTAs per SM of the current device (its SM
// count is read once per device), at least 256 keys per split. Depends only on
// the shape and the device, so the workspace query and the call agree.
void mg_decode_split(const MgProblem &p, int *S, int *chunk) {
  const long long BH = static_cast<long long>(p.B) * p.H;
  const int want = static_cast<int>((8LL * mg_sm_count() + BH - 1) / BH);
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
  return static_cast<size_t>(p.B) * p.H * S * p.L * (p.D + 4);
}

template <typename T>
cudaError_t dispatch_d(const void *Q, const void *K, const void *V, float *O, float *LSE,
                       float *part, const MgProblem &p, int S, int chunk, cudaStream_t st) {
  const T *q = static_cast<const T *>(Q), *k = static_cast<const T *>(K),
          *v = static_cast<const T *>(V);
  switch (p.D) {
    case 32: return launch_rows<32, T>(q, k, v, O, LSE, part, p, S, chunk, st);
    case 64: return launch_rows<64, T>(q, k, v, O, LSE, part, p, S, chunk, st);
    case 128: return launch_rows<128, T>(q, k, v, O, LSE, part, p, S, chunk, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t mg_launch_decode_fwd(const void *Q, const void *K, const void *V, float *O,
                                 float *LSE, float *part, const MgProblem &p, int in_type,
                                 cudaStream_t st) {
  int S, chunk;
  mg_decode_split(p, &S, &chunk);
  if (in_type == 1) return dispatch_d<__nv_bfloat16>(Q, K, V, O, LSE, part, p, S, chunk, st);
  if (in_type == 2) return dispatch_d<__half>(Q, K, V, O, LSE, part, p, S, chunk, st);
  return dispatch_d<float>(Q, K, V, O, LSE, part, p, S, chunk, st);
}
