// strict_fwd.cu -- STRICT_F32 tiled attention forward on FP32 CUDA cores.
//
// The tiled attention forward archetype of "Meganeura: Portable GPU Training
// and Inference through Vulkan and Metal" (Section 3.3) under its strict-f32
// contract (Section 4.2: no reduced-input matrix path; here no tensor cores and
// no TF32 at all). Every product is an f32 FFMA.
//
// One CTA of 256 threads owns BR = 128 query rows of one (b, h) head and walks
// the key axis in tiles of BC = 64 keys with an online softmax (running row max
// m and row sum l, in base 2 with log2(e) folded into the scale). Thread
// (ty, tx) = (tid / 16, tid % 16) owns query rows ty + 16 i (i < 8), score
// columns tx + 16 j (j < 4) and output columns VW*tx + 16*VW*v. The 16 threads
// that share a row sit in one half-warp, so row max / row sum are xor-shuffles
// and the P tile that feeds P*V is exchanged through shared memory with only a
// warp barrier. K and V tiles arrive by cp.async into single buffers that are
// refilled as soon as their last reader is done (K during the softmax and the
// P*V product, V during the next Q*K^T).
#include "internal.h"
#include "strict_common.cuh"

namespace {

using namespace mg_strict;

template <int D>
struct FwdCfg {
  static constexpr int BR = 128, BC = 64, NT = 256;
  static constexpr int QS = D + 4;   // padded row strides (floats)
  static constexpr int KS = D + 4;
  static constexpr int VS = D;
  static constexpr int PS = BC + 16; // rows ty and ty+1 land 16 banks apart
  static constexpr int DPT = D / 16; // output columns per thread
  static constexpr int VW = DPT >= 4 ? 4 : DPT;
  static constexpr int NV = DPT / VW;
  static constexpr int SMEM_FLOATS = BR * QS + BC * KS + BC * VS + BR * PS;
  static constexpr int SMEM_BYTES = SMEM_FLOATS * 4;
};

template <int D>
__global__ void __launch_bounds__(256, 1)
    strict_fwd_kernel(const float *__restrict__ Q, const float *__restrict__ K,
                      const float *__restrict__ V, float *__restrict__ O,
                      float *__restrict__ LSE, int BH, int L, int Lk_rows, int causal, int off0,
                      float scale_log2, const int *__restrict__ kv_len, int H, int br) {
  using C = FwdCfg<D>;
  using VecV = typename VecT<C::VW>::T;
  extern __shared__ float4 smem_f4[];
  float *sQ = reinterpret_cast<float *>(smem_f4);
  float *sK = sQ + C::BR * C::QS;
  float *sV = sK + C::BC * C::KS;
  float *sP = sV + C::BC * C::VS;

  const int nqt = (L + C::BR - 1) / C::BR;
  // Heaviest causal query tiles (largest qt) are scheduled first.
  const int qt = nqt - 1 - static_cast<int>(blockIdx.x / BH);
  const int bh = static_cast<int>(blockIdx.x % BH);
  const int q0 = qt * C::BR;
  // query rows L, key rows Lk (all Lk_rows rows, or the batch element's padded
  // length; rows past it are never staged); causal: query i sees key j iff
  // j <= i + off
  const MgKeys keys = mg_keys(kv_len, bh, H, L, Lk_rows, off0, br);
  const int Lk = keys.len, off = keys.off;
  const size_t head = static_cast<size_t>(bh) * L * D;
  const size_t khead = static_cast<size_t>(bh) * Lk_rows * D;
  const float *Qh = Q + head, *Kh = K + khead, *Vh = V + khead;

  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;

  int nkt = (Lk + C::BC - 1) / C::BC;
  if (causal) {
    const int last = min(q0 + C::BR, L) - 1 + off;  // last key any row of the tile sees
    nkt = last < 0 ? 0 : min(nkt, last / C::BC + 1);
  }

  stage_rows<D, C::BR, C::NT>(sQ, C::QS, Qh, q0, L, tid);
  stage_rows<D, C::BC, C::NT>(sK, C::KS, Kh, 0, Lk, tid);
  cp_async_commit();
  stage_rows<D, C::BC, C::NT>(sV, C::VS, Vh, 0, Lk, tid);
  cp_async_commit();

  float o[8][C::DPT];
  float m[8], l[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    m[i] = -CUDART_INF_F;
    l[i] = 0.f;
#pragma unroll
    for (int c = 0; c < C::DPT; ++c) o[i][c] = 0.f;
  }

  for (int kt = 0; kt < nkt; ++kt) {
    const int k0 = kt * C::BC;
    cp_async_wait<1>();  // Q and K tile kt have landed; V tile kt may be in flight
    __syncthreads();

    // ---- S = Q K^T (f32 FFMA), 8 x 4 scores per thread
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
#pragma unroll 4
    for (int k = 0; k < D; k += 4) {
      float4 kv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        kv[j] = *reinterpret_cast<const float4 *>(sK + (tx + 16 * j) * C::KS + k);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 qv = *reinterpret_cast<const float4 *>(sQ + (ty + 16 * i) * C::QS + k);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          s[i][j] = fmaf(qv.x, kv[j].x, s[i][j]);
          s[i][j] = fmaf(qv.y, kv[j].y, s[i][j]);
          s[i][j] = fmaf(qv.z, kv[j].z, s[i][j]);
          s[i][j] = fmaf(qv.w, kv[j].w, s[i][j]);
        }
      }
    }
    __syncthreads();  // every thread is done reading sK
    if (kt + 1 < nkt) {
      stage_rows<D, C::BC, C::NT>(sK, C::KS, Kh, k0 + C::BC, Lk, tid);
      cp_async_commit();
    }

    // ---- online softmax (base 2), P tile to shared memory
    const bool need_mask = (k0 + C::BC > Lk) || (causal && k0 + C::BC - 1 > q0 + off);
    float alpha[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int qi = q0 + ty + 16 * i;
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float v = s[i][j] * scale_log2;
        if (need_mask) {
          const int kj = k0 + tx + 16 * j;
          if (kj >= Lk || (causal && kj > qi + off)) v = -CUDART_INF_F;
        }
        s[i][j] = v;
        mx = fmaxf(mx, v);
      }
      mx = group_max<16>(mx);
      const float mnew = fmaxf(m[i], mx);
      const float mref = (mnew == -CUDART_INF_F) ? 0.f : mnew;  // fully masked so far
      alpha[i] = exp2f(m[i] - mref);
      m[i] = mnew;
      float rs = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float pv = exp2f(s[i][j] - mref);
        s[i][j] = pv;
        rs += pv;
      }
      l[i] = fmaf(l[i], alpha[i], rs);  // per-thread partial; reduced at the end
#pragma unroll
      for (int j = 0; j < 4; ++j) sP[(ty + 16 * i) * C::PS + tx + 16 * j] = s[i][j];
#pragma unroll
      for (int c = 0; c < C::DPT; ++c) o[i][c] *= alpha[i];
    }
    __syncwarp();  // the P rows a thread reads were written by its own half-warp

    if (kt + 1 < nkt)
      cp_async_wait<1>();
    else
      cp_async_wait<0>();
    __syncthreads();  // V tile kt visible to all

    // ---- O += P V
#pragma unroll 2
    for (int k = 0; k < C::BC; k += 4) {
      float4 pv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        pv[i] = *reinterpret_cast<const float4 *>(sP + (ty + 16 * i) * C::PS + k);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        VecV vv[C::NV];
#pragma unroll
        for (int v = 0; v < C::NV; ++v)
          vv[v] = *reinterpret_cast<const VecV *>(sV + (k + kk) * C::VS + C::VW * tx +
                                                  16 * C::VW * v);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float p = vget(pv[i], kk);
#pragma unroll
          for (int v = 0; v < C::NV; ++v)
#pragma unroll
            for (int c = 0; c < C::VW; ++c)
              o[i][v * C::VW + c] = fmaf(p, vget(vv[v], c), o[i][v * C::VW + c]);
        }
      }
    }
    __syncthreads();  // every thread is done reading sV
    if (kt + 1 < nkt) {
      stage_rows<D, C::BC, C::NT>(sV, C::VS, Vh, k0 + C::BC, Lk, tid);
      cp_async_commit();
    }
  }

  cp_async_wait<0>();  // no copy may outlive the block (a tile with no keys skips the loop)

  // ---- epilogue: O = O_acc / l, LSE = ln 2 * (m + log2 l); a row without any
  // allowed key (l = 0) gets O = 0 and LSE = -inf
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float lt = group_sum<16>(l[i]);
    const int qi = q0 + ty + 16 * i;
    if (qi < L) {
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      float *orow = O + head + static_cast<size_t>(qi) * D;
#pragma unroll
      for (int v = 0; v < C::NV; ++v) {
        float tmp[C::VW];
#pragma unroll
        for (int c = 0; c < C::VW; ++c) tmp[c] = o[i][v * C::VW + c] * inv;
        *reinterpret_cast<VecV *>(orow + C::VW * tx + 16 * C::VW * v) =
            *reinterpret_cast<const VecV *>(tmp);
      }
      if (tx == 0) LSE[static_cast<size_t>(bh) * L + qi] = (m[i] + log2f(lt)) * kLn2;
    }
  }
}

template <int D>
cudaError_t launch(const float *Q, const float *K, const float *V, float *O, float *LSE,
                   const MgProblem &p, cudaStream_t st) {
  using C = FwdCfg<D>;
  auto kern = strict_fwd_kernel<D>;
  cudaError_t e = mg_set_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM_BYTES,
                                   D == 32 ? 0 : (D == 64 ? 1 : 2));
  if (e != cudaSuccess) return e;
  const int BH = p.B * p.H;
  const int nqt = (p.L + C::BR - 1) / C::BR;
  const long long grid = static_cast<long long>(nqt) * BH;
  kern<<<static_cast<unsigned>(grid), C::NT, C::SMEM_BYTES, st>>>(
      Q, K, V, O, LSE, BH, p.L, p.Lk, p.causal, p.off, p.scale * kLog2e, p.kv_len, p.H, p.br);
  return cudaGetLastError();
}

}  // namespace

cudaError_t mg_launch_strict_fwd(const float *Q, const float *K, const float *V, float *O,
                                 float *LSE, const MgProblem &p, cudaStream_t st) {
  switch (p.D) {
    case 32: return launch<32>(Q, K, V, O, LSE, p, st);
    case 64: return launch<64>(Q, K, V, O, LSE, p, st);
    case 128: return launch<128>(Q, K, V, O, LSE, p, st);
    default: return cudaErrorInvalidValue;
  }
}
