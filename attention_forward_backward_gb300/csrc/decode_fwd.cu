// decode_fwd.cu -- attention forward for a few query rows against a long key
// axis (decoding): the key axis is split over many CTAs, each producing a partial
// softmax (running max, sum and unnormalised output per query row), and a second
// kernel merges the partials into O and LSE.
//
// The computation is the forward of the attention node ("Meganeura: Portable GPU
// Training and Inference through Vulkan and Metal", Section 3.1) for Lq <= 8
// query rows. With so few rows the work is one pass over K and V, bound by HBM,
// and the generic kernels leave most SMs idle when there are few heads: splitting
// the keys lets every SM stream its share. This file holds the STRICT_F32 partial
// kernel (f32 FFMA on the CUDA cores, K, V and Q in registers, never staged in
// shared memory), the merge shared by both contracts, and the split policy; the
// 16-bit contracts compute their partials on the tensor cores (decode_tc.cu).
// Scores are in base 2 with
// scale * log2(e) folded into Q, and every partial state is the exact
// online-softmax state of its keys, so merging is exact up to rounding:
//   m = max_s m_s,  l = sum_s l_s 2^(m_s - m),  O = sum_s O_s 2^(m_s - m) / l,
//   LSE = ln 2 (m + log2 l);  a row with no allowed key gets O = 0, LSE = -inf.
#include <math.h>

#include <algorithm>

#include "internal.h"

namespace {

constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;
constexpr int kMaxLq = 8;   // query rows per head handled here
constexpr int kTile = 32;   // split lengths are whole multiples of this many keys
constexpr int kThreads = 128;
constexpr int kMaxSplits = 256;  // the split policies never exceed this

__device__ __forceinline__ float load_in(const float *p, size_t i) { return p[i]; }
// Eight consecutive input elements as raw registers (16-byte loads): fetched one
// step ahead, copied to the f32 registers the step uses.
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

// One CTA of D threads per (bh, q) merges the S partial records in two passes
// (each a few memory round trips, not one per record): the threads read the
// splits' (m, l) pairs and reduce m = max_s m_s and l = sum_s l_s 2^(m_s - m),
// keeping the weights w_s = 2^(m_s - m) in shared memory; then thread d adds
// O_s[d] w_s over the splits, sixteen records in flight. Launched as a
// programmatic dependent of the partial kernel: it may be scheduled before the
// partials finish and waits for them here.
template <int D>
__global__ void __launch_bounds__(D)
    decode_merge_kernel(const float *__restrict__ part, float *__restrict__ O,
                        float *__restrict__ LSE, int Lq, int S) {
  constexpr int NW = D / 32;
  __shared__ float sW[kMaxSplits];
  __shared__ float sRed[NW];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int bh = blockIdx.x / Lq, q = blockIdx.x % Lq, d = threadIdx.x;
  const int lane = d & 31, wid = d >> 5;
  const size_t rstride = static_cast<size_t>(Lq) * (D + 4);
  const float *rec0 = part + static_cast<size_t>(bh) * S * rstride + q * (D + 4);
  // pass 1: maximum over the splits (a split with no allowed key has m = -inf)
  float mx = -INFINITY;
  for (int sp = d; sp < S; sp += D) {
    const float m = rec0[sp * rstride + D];
    sW[sp] = m;
    mx = fmaxf(mx, m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) sRed[wid] = mx;
  __syncthreads();
  mx = sRed[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) mx = fmaxf(mx, sRed[w]);
  __syncthreads();
  float ls = 0.f;
  for (int sp = d; sp < S; sp += D) {
    const float w = mx == -INFINITY ? 0.f : exp2f(sW[sp] - mx);  // m_s = -inf: 0
    sW[sp] = w;
    ls = fmaf(rec0[sp * rstride + D + 1], w, ls);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
  if (lane == 0) sRed[wid] = ls;
  __syncthreads();
  ls = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) ls += sRed[w];
  // pass 2: element d
  float acc = 0.f;
  for (int s0 = 0; s0 < S; s0 += 16) {
    float v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u)
      v[u] = s0 + u < S ? rec0[static_cast<size_t>(s0 + u) * rstride + d] : 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u)
      if (s0 + u < S) acc = fmaf(v[u], sW[s0 + u], acc);
  }
  const size_t row = static_cast<size_t>(bh) * Lq + q;
  O[row * D + d] = ls > 0.f ? acc / ls : 0.f;
  if (d == 0) LSE[row] = ls > 0.f ? (mx + log2f(ls)) * kLn2F : -INFINITY;
}

template <int D, int LQ, typename TIn>
cudaError_t launch(const TIn *Q, const TIn *K, const TIn *V, float *part, const MgProblem &p,
                   int S, int chunk, cudaStream_t st) {
  const int BH = p.B * p.H;
  decode_partial_kernel<D, LQ, TIn>
      <<<static_cast<unsigned>(static_cast<long long>(BH) * S), kThreads, 0, st>>>(
          Q, K, V, part, p.L, p.Lk, p.causal, p.off, S, chunk, p.scale * kLog2eF);
  return cudaGetLastError();
}

template <int D, typename TIn>
cudaError_t launch_rows(const TIn *Q, const TIn *K, const TIn *V, float *part, const MgProblem &p,
                        int S, int chunk, cudaStream_t st) {
  if (p.L <= 1) return launch<D, 1, TIn>(Q, K, V, part, p, S, chunk, st);
  if (p.L <= 2) return launch<D, 2, TIn>(Q, K, V, part, p, S, chunk, st);
  if (p.L <= 4) return launch<D, 4, TIn>(Q, K, V, part, p, S, chunk, st);
  return launch<D, 8, TIn>(Q, K, V, part, p, S, chunk, st);
}

// The merge, launched with programmatic stream serialisation so that its launch
// overlaps the end of the partial kernel (it waits for the partials itself).
template <int D>
cudaError_t merge(const float *part, float *O, float *LSE, const MgProblem &p, int S,
                  cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long long>(p.B) * p.H * p.L));
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel<D>, part, O, LSE, p.L, S);
}

template <int D>
cudaError_t partial_f32(const void *Q, const void *K, const void *V, float *part,
                        const MgProblem &p, int S, int chunk, cudaStream_t st) {
  return launch_rows<D, float>(static_cast<const float *>(Q), static_cast<const float *>(K),
                               static_cast<const float *>(V), part, p, S, chunk, st);
}

}  // namespace

int mg_decode_max_rows() { return kMaxLq; }

// Splits of the key axis. Depends only on the shape, the kernel family and the
// device (its SM count is read once per device), so the workspace query and the
// call agree.
// * CUDA-core kernel: about eight CTAs per SM, at least 256 keys per split,
//   split lengths in whole 32-key steps.
// * tensor-core kernel (one CTA per SM): the split count s minimising
//   waves(s) * (c0 + Lk / s), waves(s) = ceil(B H s / SMs), with c0 = 256 keys
//   standing for a CTA's fixed cost (set-up, pipeline fill, record); at least
//   512 keys per split, split lengths in whole 128-key tiles.
void mg_decode_split(const MgProblem &p, int *S, int *chunk, bool tc) {
  const long long BH = static_cast<long long>(p.B) * p.H;
  const int sms = mg_sm_count();
  int s, step;
  if (tc) {
    step = 128;
    const int maxs = std::max(1, std::min(kMaxSplits, (p.Lk + 511) / 512));
    double best = 0.0;
    s = 1;
    for (int t = 1; t <= maxs; ++t) {
      const long long waves = (BH * t + sms - 1) / sms;
      const double cost = static_cast<double>(waves) * (256.0 + static_cast<double>(p.Lk) / t);
      if (t == 1 || cost < best) {
        best = cost;
        s = t;
      }
    }
  } else {
    step = kTile;
    const int want = static_cast<int>((8LL * sms + BH - 1) / BH);
    const int maxs = (p.Lk + 255) / 256;
    s = want < 1 ? 1 : want;
    if (s > maxs) s = maxs;
    if (s > kMaxSplits) s = kMaxSplits;
  }
  const int c = ((p.Lk + s - 1) / s + step - 1) / step * step;
  *S = (p.Lk + c - 1) / c;
  *chunk = c;
}

size_t mg_decode_workspace_floats(const MgProblem &p, bool tc) {
  int S, chunk;
  mg_decode_split(p, &S, &chunk, tc);
  return static_cast<size_t>(p.B) * p.H * S * p.L * (p.D + 4);
}

cudaError_t mg_launch_decode_fwd(const void *Q, const void *K, const void *V, float *O,
                                 float *LSE, float *part, const MgProblem &p, int in_type,
                                 unsigned int *err, cudaStream_t st) {
  int S, chunk;
  cudaError_t e;
  if (in_type == 1 || in_type == 2) {
    // 16-bit inputs: both products on the tensor cores
    mg_decode_split(p, &S, &chunk, true);
    e = mg_launch_decode_tc_partial(Q, K, V, part, p, S, chunk, err, st);
  } else {
    mg_decode_split(p, &S, &chunk, false);
    switch (p.D) {
      case 32: e = partial_f32<32>(Q, K, V, part, p, S, chunk, st); break;
      case 64: e = partial_f32<64>(Q, K, V, part, p, S, chunk, st); break;
      case 128: e = partial_f32<128>(Q, K, V, part, p, S, chunk, st); break;
      default: return cudaErrorInvalidValue;
    }
  }
  if (e != cudaSuccess) return e;
  switch (p.D) {
    case 32: return merge<32>(part, O, LSE, p, S, st);
    case 64: return merge<64>(part, O, LSE, p, S, st);
    case 128: return merge<128>(part, O, LSE, p, S, st);
    default: return cudaErrorInvalidValue;
  }
}
