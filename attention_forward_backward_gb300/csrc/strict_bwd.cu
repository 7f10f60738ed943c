// strict_bwd.cu -- STRICT_F32 attention backward on FP32 CUDA cores: the Dvec
// pre-pass and the fused dK+dV kernel that also emits dQ through f32
// reductions.
//
// "Meganeura: Portable GPU Training and Inference through Vulkan and Metal"
// splits the attention derivative into a dQ kernel and one fused dK+dV kernel
// (Section 3.3; Section 8 makes fused dK+dV an invariant; Section 7.3 names the
// two as the dominant backward cost). Derivative regions stay f32 (Sections 3.1
// and 4.2). Here the dQ contribution of each key block is added into a zeroed
// f32 dQ with vector atomics instead of a second pass that would recompute S
// and dP per query block: at FFMA speed the atomic traffic is a few percent of
// the step, while a separate pass costs two extra L x L x D products.
//
// One CTA of 256 threads owns BC = 64 keys of one head and walks the query axis
// in tiles of BR = 64 rows (only tiles at or below the diagonal when causal).
// Per query tile: S^T = K Q^T and dP^T = V dO^T (64 x 64 each), P^T = exp2(S^T
// scale log2e - LSE log2e), dS^T = P^T (dP^T - Dvec); dV += P^T dO, dK += dS^T Q
// in registers; dQ_tile = scale dS K is added to global dQ. Thread (ty, tx)
// owns keys ty + 16 a (a < 4), queries tx + 16 b (b < 4) of the score tiles and
// output columns VW*tx + 16*VW*v of dK, dV and the dQ tile.
#include <cuda_fp16.h>

#include <type_traits>

#include "internal.h"
#include "strict_common.cuh"

namespace {

using namespace mg_strict;

template <int D>
struct BwdCfg {
  static constexpr int BR = 64, BC = 64, NT = 256;
  static constexpr int RS = D + 4;  // row stride of the K, V, Q, dO tiles (floats)
  static constexpr int TS = 64 + 16;  // row stride of the 64 x 64 score tiles
  static constexpr int DPT = D / 16;
  static constexpr int VW = DPT >= 4 ? 4 : DPT;
  static constexpr int NV = DPT / VW;
  static constexpr int SMEM_FLOATS = 4 * 64 * RS + 3 * 64 * TS + 2 * 64;
  static constexpr int SMEM_BYTES = SMEM_FLOATS * 4;
};

template <int D>
__global__ void __launch_bounds__(256, 1)
    strict_dkdv_kernel(const float *__restrict__ Q, const float *__restrict__ K,
                       const float *__restrict__ V, const float *__restrict__ dO,
                       const float *__restrict__ LSE, const float *__restrict__ Dvec,
                       float *__restrict__ dQ, float *__restrict__ dK, float *__restrict__ dV,
                       int BH, int L, int Lk_rows, int causal, int off0, float scale,
                       float scale_log2, const int *__restrict__ kv_len, int H, int br) {
  using C = BwdCfg<D>;
  using VecV = typename VecT<C::VW>::T;
  extern __shared__ float4 smem_f4[];
  float *sK = reinterpret_cast<float *>(smem_f4);
  float *sV = sK + 64 * C::RS;
  float *sQ = sV + 64 * C::RS;
  float *sdO = sQ + 64 * C::RS;
  float *sPT = sdO + 64 * C::RS;  // [key][query]
  float *sdST = sPT + 64 * C::TS; // [key][query]
  float *sdS = sdST + 64 * C::TS; // [query][key]
  float *sLse = sdS + 64 * C::TS; // LSE (natural) of the query tile
  float *sDv = sLse + 64;         // Dvec of the query tile

  const int kt = static_cast<int>(blockIdx.x / BH);  // heaviest (kt = 0) first
  const int bh = static_cast<int>(blockIdx.x % BH);
  const int k0 = kt * C::BC;
  // query rows L, key rows Lk (all Lk_rows rows, or the batch element's padded
  // length; rows past it are never staged and get dK = dV = 0); causal: query
  // i sees key j iff j <= i + off
  const MgKeys keys = mg_keys(kv_len, bh, H, L, Lk_rows, off0, br);
  const int Lk = keys.len, off = keys.off;
  const size_t head = static_cast<size_t>(bh) * L * D;
  const size_t khead = static_cast<size_t>(bh) * Lk_rows * D;
  const float *Qh = Q + head, *Kh = K + khead, *Vh = V + khead, *dOh = dO + head;
  const float *Lh = LSE + static_cast<size_t>(bh) * L, *Dh = Dvec + static_cast<size_t>(bh) * L;
  float *dQh = dQ + head;

  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  // query tiles holding a query that sees key k0 (none when the block starts
  // past the key count or past the last tile: dK = dV = 0 then)
  const int nqt = k0 >= Lk ? 0 : (L + C::BR - 1) / C::BR;
  const int qt0 = causal ? max(0, k0 - off) / C::BR : 0;

  stage_rows<D, 64, C::NT>(sK, C::RS, Kh, k0, Lk, tid);
  stage_rows<D, 64, C::NT>(sV, C::RS, Vh, k0, Lk, tid);
  stage_rows<D, 64, C::NT>(sQ, C::RS, Qh, qt0 * C::BR, L, tid);
  stage_rows<D, 64, C::NT>(sdO, C::RS, dOh, qt0 * C::BR, L, tid);
  stage_vec<64>(sLse, Lh, qt0 * C::BR, L, tid);
  stage_vec<64>(sDv, Dh, qt0 * C::BR, L, tid);
  cp_async_commit();

  float dk[4][C::DPT], dv[4][C::DPT];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < C::DPT; ++c) dk[a][c] = dv[a][c] = 0.f;

  for (int qt = qt0; qt < nqt; ++qt) {
    const int q0 = qt * C::BR;
    cp_async_wait<0>();
    __syncthreads();

    // ---- S^T = K Q^T and dP^T = V dO^T
    float st[4][4], dpt[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) st[a][b] = dpt[a][b] = 0.f;
#pragma unroll 2
    for (int k = 0; k < D; k += 4) {
      float4 qv[4], ov[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        qv[b] = *reinterpret_cast<const float4 *>(sQ + (tx + 16 * b) * C::RS + k);
        ov[b] = *reinterpret_cast<const float4 *>(sdO + (tx + 16 * b) * C::RS + k);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const float4 kv = *reinterpret_cast<const float4 *>(sK + (ty + 16 * a) * C::RS + k);
        const float4 vv = *reinterpret_cast<const float4 *>(sV + (ty + 16 * a) * C::RS + k);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          st[a][b] = fmaf(kv.x, qv[b].x, st[a][b]);
          st[a][b] = fmaf(kv.y, qv[b].y, st[a][b]);
          st[a][b] = fmaf(kv.z, qv[b].z, st[a][b]);
          st[a][b] = fmaf(kv.w, qv[b].w, st[a][b]);
          dpt[a][b] = fmaf(vv.x, ov[b].x, dpt[a][b]);
          dpt[a][b] = fmaf(vv.y, ov[b].y, dpt[a][b]);
          dpt[a][b] = fmaf(vv.z, ov[b].z, dpt[a][b]);
          dpt[a][b] = fmaf(vv.w, ov[b].w, dpt[a][b]);
        }
      }
    }

    // ---- P^T = exp(S^T scale - LSE), dS^T = P^T (dP^T - Dvec)
    const bool need_mask =
        (q0 + C::BR > L) || (k0 + C::BC > Lk) || (causal && q0 + off < k0 + C::BC - 1);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int ql = tx + 16 * b;
      const float lse2 = sLse[ql] * kLog2e;
      const float dvq = sDv[ql];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int kl = ty + 16 * a;
        float p = exp2f(fmaf(st[a][b], scale_log2, -lse2));
        if (need_mask) {
          const int qg = q0 + ql, kg = k0 + kl;
          if (qg >= L || kg >= Lk || (causal && kg > qg + off)) p = 0.f;
        }
        const float ds = p * (dpt[a][b] - dvq);
        sPT[kl * C::TS + ql] = p;
        sdST[kl * C::TS + ql] = ds;
        sdS[ql * C::TS + kl] = ds;
      }
    }
    __syncwarp();  // P^T / dS^T rows a thread reads next were written by its half-warp

    // ---- dV += P^T dO, dK += dS^T Q
#pragma unroll 2
    for (int q = 0; q < C::BR; q += 4) {
      float4 p4[4], d4[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        p4[a] = *reinterpret_cast<const float4 *>(sPT + (ty + 16 * a) * C::TS + q);
        d4[a] = *reinterpret_cast<const float4 *>(sdST + (ty + 16 * a) * C::TS + q);
      }
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        VecV ov[C::NV], qv[C::NV];
#pragma unroll
        for (int v = 0; v < C::NV; ++v) {
          ov[v] = *reinterpret_cast<const VecV *>(sdO + (q + qq) * C::RS + C::VW * tx +
                                                  16 * C::VW * v);
          qv[v] = *reinterpret_cast<const VecV *>(sQ + (q + qq) * C::RS + C::VW * tx +
                                                  16 * C::VW * v);
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const float pp = vget(p4[a], qq), dd = vget(d4[a], qq);
#pragma unroll
          for (int v = 0; v < C::NV; ++v)
#pragma unroll
            for (int c = 0; c < C::VW; ++c) {
              dv[a][v * C::VW + c] = fmaf(pp, vget(ov[v], c), dv[a][v * C::VW + c]);
              dk[a][v * C::VW + c] = fmaf(dd, vget(qv[v], c), dk[a][v * C::VW + c]);
            }
        }
      }
    }
    __syncthreads();  // dS complete; everyone is done with sQ, sdO, sLse, sDv

    if (qt + 1 < nqt) {  // prefetch the next query tile behind the dQ product
      const int qn = q0 + C::BR;
      stage_rows<D, 64, C::NT>(sQ, C::RS, Qh, qn, L, tid);
      stage_rows<D, 64, C::NT>(sdO, C::RS, dOh, qn, L, tid);
      stage_vec<64>(sLse, Lh, qn, L, tid);
      stage_vec<64>(sDv, Dh, qn, L, tid);
      cp_async_commit();
    }

    // ---- dQ_tile = scale * dS K, added into global dQ
    float dq[4][C::DPT];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < C::DPT; ++c) dq[a][c] = 0.f;
#pragma unroll 2
    for (int kk = 0; kk < C::BC; kk += 4) {
      float4 s4[4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
        s4[a] = *reinterpret_cast<const float4 *>(sdS + (ty + 16 * a) * C::TS + kk);
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        VecV kv[C::NV];
#pragma unroll
        for (int v = 0; v < C::NV; ++v)
          kv[v] = *reinterpret_cast<const VecV *>(sK + (kk + k4) * C::RS + C::VW * tx +
                                                  16 * C::VW * v);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const float sv = vget(s4[a], k4);
#pragma unroll
          for (int v = 0; v < C::NV; ++v)
#pragma unroll
            for (int c = 0; c < C::VW; ++c)
              dq[a][v * C::VW + c] = fmaf(sv, vget(kv[v], c), dq[a][v * C::VW + c]);
        }
      }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int qg = q0 + ty + 16 * a;
      if (qg < L) {
        float *row = dQh + static_cast<size_t>(qg) * D;
#pragma unroll
        for (int v = 0; v < C::NV; ++v) {
          VecV add;
          float *ap = reinterpret_cast<float *>(&add);
#pragma unroll
          for (int c = 0; c < C::VW; ++c) ap[c] = scale * dq[a][v * C::VW + c];
          atomicAdd(reinterpret_cast<VecV *>(row + C::VW * tx + 16 * C::VW * v), add);
        }
      }
    }
  }

  cp_async_wait<0>();  // no copy may outlive the block (a key block with no queries)

  // ---- store dK (scaled) and dV for this key block
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int kg = k0 + ty + 16 * a;
    if (kg < Lk_rows) {
      float *krow = dK + khead + static_cast<size_t>(kg) * D;
      float *vrow = dV + khead + static_cast<size_t>(kg) * D;
#pragma unroll
      for (int v = 0; v < C::NV; ++v) {
        VecV kk, vv;
        float *kp = reinterpret_cast<float *>(&kk);
        float *vp = reinterpret_cast<float *>(&vv);
#pragma unroll
        for (int c = 0; c < C::VW; ++c) {
          kp[c] = scale * dk[a][v * C::VW + c];
          vp[c] = dv[a][v * C::VW + c];
        }
        *reinterpret_cast<VecV *>(krow + C::VW * tx + 16 * C::VW * v) = kk;
        *reinterpret_cast<VecV *>(vrow + C::VW * tx + 16 * C::VW * v) = vv;
      }
    }
  }
}

// Four consecutive elements widened to f32 (8- or 16-byte loads).
__device__ __forceinline__ void load4(const float *p, float (&g)[4]) {
  const float4 d = *reinterpret_cast<const float4 *>(p);
  g[0] = d.x; g[1] = d.y; g[2] = d.z; g[3] = d.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16 *p, float (&g)[4]) {
  const uint2 raw = *reinterpret_cast<const uint2 *>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
  g[0] = a.x; g[1] = a.y; g[2] = b.x; g[3] = b.y;
}
__device__ __forceinline__ void load4(const __half *p, float (&g)[4]) {
  const uint2 raw = *reinterpret_cast<const uint2 *>(p);
  const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
  g[0] = a.x; g[1] = a.y; g[2] = b.x; g[3] = b.y;
}

// Dvec_i = sum_d dO_id O_id. G = D/4 threads per row, 4 elements per thread.
template <int D, typename TO, typename TdO>
__global__ void __launch_bounds__(256) dvec_kernel(const TO *__restrict__ O,
                                                   const TdO *__restrict__ dO,
                                                   float *__restrict__ Dvec, long long rows) {
  constexpr int G = D / 4;
  const long long row = (static_cast<long long>(blockIdx.x) * 256 + threadIdx.x) / G;
  const int lane = threadIdx.x % G;
  float acc = 0.f;
  if (row < rows) {
    float o[4], g[4];
    load4(O + row * D + lane * 4, o);
    load4(dO + row * D + lane * 4, g);
    acc = o[0] * g[0];
    acc = fmaf(o[1], g[1], acc);
    acc = fmaf(o[2], g[2], acc);
    acc = fmaf(o[3], g[3], acc);
  }
  acc = group_sum<G>(acc);
  if (row < rows && lane == 0) Dvec[row] = acc;
}

// dst = src rounded (RNE) to a 16-bit type, 4 elements per thread.
template <typename T16>
__global__ void __launch_bounds__(256) f32_to_16_kernel(const float *__restrict__ src,
                                                        T16 *__restrict__ dst, size_t n4) {
  const size_t i = static_cast<size_t>(blockIdx.x) * 256 + threadIdx.x;
  if (i >= n4) return;
  const float4 v = reinterpret_cast<const float4 *>(src)[i];
  uint2 out;
  if constexpr (sizeof(T16) == 2 && std::is_same<T16, __half>::value) {
    __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    out = make_uint2(*reinterpret_cast<uint32_t *>(&a), *reinterpret_cast<uint32_t *>(&b));
  } else {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    out = make_uint2(*reinterpret_cast<uint32_t *>(&a), *reinterpret_cast<uint32_t *>(&b));
  }
  reinterpret_cast<uint2 *>(dst)[i] = out;
}

template <int D>
cudaError_t launch_dkdv(const float *Q, const float *K, const float *V, const float *dO,
                        const float *LSE, const float *Dvec, float *dQ, float *dK, float *dV,
                        const MgProblem &p, cudaStream_t st) {
  using C = BwdCfg<D>;
  auto kern = strict_dkdv_kernel<D>;
  cudaError_t e = mg_set_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM_BYTES,
                                   D == 32 ? 3 : (D == 64 ? 4 : 5));
  if (e != cudaSuccess) return e;
  const int BH = p.B * p.H;
  const int nkt = (p.Lk + C::BC - 1) / C::BC;
  const long long grid = static_cast<long long>(nkt) * BH;
  kern<<<static_cast<unsigned>(grid), C::NT, C::SMEM_BYTES, st>>>(
      Q, K, V, dO, LSE, Dvec, dQ, dK, dV, BH, p.L, p.Lk, p.causal, p.off, p.scale,
      p.scale * kLog2e, p.kv_len, p.H, p.br);
  return cudaGetLastError();
}

template <int D, typename TO, typename TdO>
cudaError_t launch_dvec(const TO *O, const TdO *dO, float *Dvec, const MgProblem &p,
                        cudaStream_t st) {
  const long long rows = static_cast<long long>(p.B) * p.H * p.L;
  const long long threads = rows * (D / 4);
  const long long blocks = (threads + 255) / 256;
  dvec_kernel<D, TO, TdO><<<static_cast<unsigned>(blocks), 256, 0, st>>>(O, dO, Dvec, rows);
  return cudaGetLastError();
}

template <typename TO, typename TdO>
cudaError_t dvec_dispatch(const TO *O, const TdO *dO, float *Dvec, const MgProblem &p,
                          cudaStream_t st) {
  switch (p.D) {
    case 32: return launch_dvec<32>(O, dO, Dvec, p, st);
    case 64: return launch_dvec<64>(O, dO, Dvec, p, st);
    case 128: return launch_dvec<128>(O, dO, Dvec, p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t mg_launch_strict_dkdv(const float *Q, const float *K, const float *V,
                                  const float *dO, const float *LSE, const float *Dvec,
                                  float *dQ, float *dK, float *dV, const MgProblem &p,
                                  cudaStream_t st) {
  switch (p.D) {
    case 32: return launch_dkdv<32>(Q, K, V, dO, LSE, Dvec, dQ, dK, dV, p, st);
    case 64: return launch_dkdv<64>(Q, K, V, dO, LSE, Dvec, dQ, dK, dV, p, st);
    case 128: return launch_dkdv<128>(Q, K, V, dO, LSE, Dvec, dQ, dK, dV, p, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t mg_launch_dvec_f32(const float *O, const float *dO, float *Dvec, const MgProblem &p,
                               cudaStream_t st) {
  return dvec_dispatch(O, dO, Dvec, p, st);
}


cudaError_t mg_launch_dvec_16(const void *O, const void *dO, float *Dvec, const MgProblem &p,
                              cudaStream_t st) {
  if (p.f16) {
    const __half *d = static_cast<const __half *>(dO);
    if (p.out16) return dvec_dispatch(static_cast<const __half *>(O), d, Dvec, p, st);
    return dvec_dispatch(static_cast<const float *>(O), d, Dvec, p, st);
  }
  const __nv_bfloat16 *d = static_cast<const __nv_bfloat16 *>(dO);
  if (p.out16) return dvec_dispatch(static_cast<const __nv_bfloat16 *>(O), d, Dvec, p, st);
  return dvec_dispatch(static_cast<const float *>(O), d, Dvec, p, st);
}

cudaError_t mg_launch_f32_to_16(const float *src, void *dst, size_t n, bool f16,
                                cudaStream_t st) {
  if (n % 4) return cudaErrorInvalidValue;
  const size_t n4 = n / 4;
  if (n4 == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((n4 + 255) / 256);
  if (f16)
    f32_to_16_kernel<__half><<<blocks, 256, 0, st>>>(src, static_cast<__half *>(dst), n4);
  else
    f32_to_16_kernel<__nv_bfloat16>
        <<<blocks, 256, 0, st>>>(src, static_cast<__nv_bfloat16 *>(dst), n4);
  return cudaGetLastError();
}
