// conv_grad.cu -- the two derivatives of a channels-last 2-D convolution on the
// tcgen05 tensor cores: input gradient dX (an implicit GEMM over pixels x input
// channels, reducing over taps x output channels) and weight gradient dW (a GEMM
// per tap over output x input channels, reducing over pixels, split across CTAs).
//
// "Meganeura: Portable GPU Training and Inference through Vulkan and Metal"
// lists convolution input and weight derivatives among the backward nodes
// (Section 3.1) and names the kernels that own its ResNet-50 training gap
// (Section 7.3, "Convolution derivatives own the ResNet gap": an input-gradient
// GEMM and a weight-gradient GEMM with a variant for small outputs). Their
// definition, with X [N][H][W][C], Wt [K][R][S][C] and dY [N][P][Q][K]:
//   dX[n,h,w,c] = sum of dY[n,p,q,k] Wt[k,r,s,c] over p*st - pad + r = h, q*st - pad + s = w
//   dW[k,r,s,c] = sum_{n,p,q} dY[n,p,q,k] X[n, p*st - pad + r, q*st - pad + s, c]
//
// Both kernels: 128 threads; warp 0 lane 0 issues TMA loads into an NST-stage
// ring, warp 1 lane 0 issues the MMAs (f32 accumulator of 128 lanes x BN
// columns in tensor memory), then all four warps read the accumulator back
// (lane = accumulator row). Shared memory is sized for two CTAs per SM, so one
// CTA's read-back overlaps the other's main loop. Every operand tile is a 4-D
// TMA box with 128-byte swizzle; coordinates outside the tensor read as zero,
// which supplies the convolution's zero padding and the tails of C and K.
//
// Input gradient. The output pixels are split by stride phase (h mod st,
// w mod st): within one phase, the taps that reach it are r = r0, r0+st, ... with
// r0 = (ph + pad) mod st, and tap r reads dY row i + (ph + pad - r) / st for
// phase row i -- a unit-stride window of dY. A tile is a box of phase pixels
// (BW x BH x BNi <= 128 rows = the MMA's M); the reduction runs over (tap,
// 64-channel chunk of K): A = the shifted dY box (K-major), B = Wt[k-chunk][r][s]
// [c-tile] (MN-major: c is contiguous). Rows past the box hold stale data and
// produce rows that are never stored.
//
// Weight gradient. A CTA owns one tap (r, s), a 128-wide block of K and a BN
// block of C, and a range of pixel boxes (exactly 64 pixels each, zero-filled
// past the image); A = dY box^T (MN-major, k contiguous), B = the X box the tap
// reads (MN-major, c contiguous). With stride 2 the tap's input pixels
// (p*2 + r - pad) form a unit-stride box of one of four phase views of X (a
// tensor map whose row and column strides are doubled). Partial sums are added
// into dW (zeroed first) with f32 vector atomics.
#include <stdint.h>

#include <algorithm>

#include "internal.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace {

using namespace mg_tc;

template <int BN>
struct ConvCfg {
  static constexpr int BM = 128;                   // accumulator rows (MMA M)
  static constexpr int NST = BN == 128 ? 3 : 4;    // ring stages (two CTAs per SM)
  static constexpr int A_BYTES = BM * 128;         // 128 rows x 64 elements
  static constexpr int B_BYTES = BN * 128;         // BN/64 boxes of 64 rows x 128 bytes
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int OFF_BAR = NST * STAGE;
  static constexpr int B_FULL = 0;
  static constexpr int B_EMPTY = NST;
  static constexpr int B_ACC = 2 * NST;
  static constexpr int NBAR = 2 * NST + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int NTHREADS = 128;
  static constexpr int TMEM_COLS = BN;
  static_assert(2 * SMEM_BYTES <= 228 * 1024, "two CTAs per SM");
};

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return false;
  }
  return true;
}

struct DgradArgs {
  int N, H, W, C, K, R, S, st, pad, P, Q;
  int BW, BH, BNi;     // pixel box of one tile (phase pixels)
  int nphase;          // st * st
  int tile_end[4];     // prefix sums of the tiles of each phase
  float *dX;
  unsigned int *err;
  unsigned long long timeout_ns;
};

struct WgradArgs {
  int N, H, W, C, K, R, S, st, pad, P, Q;
  int BW, BH, BNi;     // pixel box of one reduction step (exactly 64 pixels)
  int KB;              // 128-row blocks of K
  int Z;               // pixel-range splits
  int phase_empty;     // bit (pr * st + pc): that phase view of X has no pixel
  float *dW;
  unsigned int *err;
  unsigned long long timeout_ns;
};

// Shared prologue: barriers, tensor memory, abort state.
template <class C>
__device__ __forceinline__ uint32_t conv_setup(uint8_t *smem, uint32_t sbase, int warp) {
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    for (int i = 0; i < C::NBAR; ++i) mbar_init(sbase + C::OFF_BAR + 8u * i, 1);
    *reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4) = 0;
    fence_barrier_init();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return *tmem_slot;
}

template <class C>
__device__ __forceinline__ void conv_teardown(uint32_t tmem, int warp) {
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ input gradient
template <int BN, bool F16>
__global__ void __launch_bounds__(128, 2)
    conv_dgrad_kernel(const __grid_constant__ CUtensorMap tmdY,
                      const __grid_constant__ CUtensorMap tmW, const DgradArgs a) {
  using C = ConvCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return sbase + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // tile -> phase, then (n block, phase-row block, phase-column block)
  int t = static_cast<int>(blockIdx.x), phase = 0;
  while (phase + 1 < a.nphase && t >= a.tile_end[phase]) ++phase;
  if (phase > 0) t -= a.tile_end[phase - 1];
  const int st = a.st, ph = phase / st, pw = phase % st;
  const int Hph = (a.H - ph + st - 1) / st, Wph = (a.W - pw + st - 1) / st;
  const int TJ = (Wph + a.BW - 1) / a.BW, TI = (Hph + a.BH - 1) / a.BH;
  const int j0 = (t % TJ) * a.BW;
  const int i0 = ((t / TJ) % TI) * a.BH;
  const int n0 = (t / TJ / TI) * a.BNi;
  const int c0 = static_cast<int>(blockIdx.y) * BN;
  // taps that reach this phase
  const int r0 = (ph + a.pad) % st, s0 = (pw + a.pad) % st;
  const int nr = r0 < a.R ? (a.R - r0 + st - 1) / st : 0;
  const int ns = s0 < a.S ? (a.S - s0 + st - 1) / st : 0;
  const int KC = (a.K + 63) / 64;
  const int T = nr * ns * KC;

  // Step s: K chunk kc = s % KC of tap (r, sx); its dY box starts at phase pixel
  // (i0 + dr, j0 + dq). A box wholly outside dY would only add zeros: such a step
  // is left out (no load is ever issued for a box with no element in the tensor).
  struct Step {
    int kc, r, sx, dr, dq;
    bool live;
  };
  auto step = [&](int s) {
    Step x;
    x.kc = s % KC;
    const int rs = s / KC;
    x.r = r0 + (rs / ns) * st;
    x.sx = s0 + (rs % ns) * st;
    x.dr = (ph + a.pad - x.r) / st;  // exact: ph + pad - r is a multiple of st
    x.dq = (pw + a.pad - x.sx) / st;
    x.live = i0 + x.dr < a.P && i0 + x.dr + a.BH > 0 && j0 + x.dq < a.Q && j0 + x.dq + a.BW > 0;
    return x;
  };
  int first_live = 0;
  while (first_live < T && !step(first_live).live) ++first_live;
  const bool any = first_live < T;

  const uint32_t tmem = conv_setup<C>(smem, sbase, warp);
  const Abort ab = make_abort(reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4), a.err,
                              a.timeout_ns);
  const int nbox = min(BN / 64, (a.C - c0 + 63) / 64);  // W boxes with a channel < C
  const uint32_t tx = static_cast<uint32_t>(a.BW * a.BH * a.BNi) * 128u + nbox * 8192u;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int s = first_live, u = 0; s < T; ++s) {
        const Step x = step(s);
        if (!x.live) continue;
        const int stg = u % C::NST;
        if (u >= C::NST && !mbar_wait(bar(C::B_EMPTY + stg), ((u / C::NST) - 1) & 1, ab)) break;
        const uint32_t sa = sbase + stg * C::STAGE;
        mbar_arrive_expect_tx(bar(C::B_FULL + stg), tx);
        tma_load_4d(sa, &tmdY, x.kc * 64, j0 + x.dq, i0 + x.dr, n0, bar(C::B_FULL + stg));
        for (int b = 0; b < nbox; ++b)
          tma_load_4d(sa + C::A_BYTES + b * 8192, &tmW, c0 + 64 * b, x.sx, x.r, x.kc * 64,
                      bar(C::B_FULL + stg));
        issued = ++u;
      }
      for (int u = max(0, issued - C::NST); u < issued; ++u)
        drain_wait(bar(C::B_FULL + u % C::NST), (u / C::NST) & 1, 2000000000ull);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_16_f32(128, BN, false, true, F16);
      for (int s = first_live, u = 0; s < T; ++s) {
        if (!step(s).live) continue;
        const int stg = u % C::NST;
        if (!mbar_wait(bar(C::B_FULL + stg), (u / C::NST) & 1, ab)) break;
        tc_fence_after();
        const uint32_t sa = opaque_u32(sbase + stg * C::STAGE);
        const uint64_t da = sdesc_sw128(sa, 0, 1024);
        const uint64_t db = sdesc_sw128(sa + C::A_BYTES, 8192, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem, sdesc_add(da, kk * 32), sdesc_add(db, kk * 2048), idesc,
                 (u > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(C::B_EMPTY + stg));
        ++u;
      }
      // the accumulator barrier arrives after every MMA (and every earlier commit)
      // has completed; wait for it here as well, so that no arrive is still in
      // flight when the CTA exits (also when no MMA was issued)
      mma_commit(bar(C::B_ACC));
      drain_wait(bar(C::B_ACC), 0, 2000000000ull);
    }
    __syncwarp();
  }

  // ------------------------------------------------------------ read-back (all warps)
  const int m = 32 * warp + lane;
  const int ww = m % a.BW, hh = (m / a.BW) % a.BH, nn = m / (a.BW * a.BH);
  const int i = i0 + hh, j = j0 + ww, n = n0 + nn;
  const bool valid = nn < a.BNi && n < a.N && i < Hph && j < Wph;
  const size_t row =
      valid ? ((static_cast<size_t>(n) * a.H + (i * st + ph)) * a.W + (j * st + pw)) * a.C : 0;
  bool ok = true;
  if (any) ok = mbar_wait_warp(bar(C::B_ACC), 0, ab);
  if (ok) {
    tc_fence_after();
#pragma unroll
    for (int cc = 0; cc < BN / 32; ++cc) {
      uint32_t r[32];
      if (any) {
        tmem_ld32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + 32 * cc, r);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = 0u;  // no tap reaches these pixels
      }
      const int cb = c0 + 32 * cc;
      if (valid) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          if (cb + e < a.C)
            *reinterpret_cast<float4 *>(a.dX + row + cb + e) =
                make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]),
                            __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
      }
    }
  }
  conv_teardown<C>(tmem, warp);
}

// ------------------------------------------------------------------ weight gradient
template <int BN, bool F16>
__global__ void __launch_bounds__(128, 2)
    conv_wgrad_kernel(const __grid_constant__ CUtensorMap tmdY,
                      const __grid_constant__ CUtensorMap tmX0,
                      const __grid_constant__ CUtensorMap tmX1,
                      const __grid_constant__ CUtensorMap tmX2,
                      const __grid_constant__ CUtensorMap tmX3, const WgradArgs a) {
  using C = ConvCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return sbase + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int st = a.st;
  const int tap = static_cast<int>(blockIdx.y), r = tap / a.S, sx = tap % a.S;
  const int k0 = (static_cast<int>(blockIdx.z) % a.KB) * 128;
  const int c0 = (static_cast<int>(blockIdx.z) / a.KB) * BN;
  // input pixel of output (p, q) under this tap: (p*st + ar, q*st + as), in the
  // phase view (pr, pc) at (p + fr, q + fc)
  const int ar = r - a.pad, as = sx - a.pad;
  const int pr = ((ar % st) + st) % st, pc = ((as % st) + st) % st;
  const int fr = (ar - pr) / st, fc = (as - pc) / st;
  const int phase = pr * st + pc;
  if ((a.phase_empty >> phase) & 1) return;  // the tap reads only padding: adds nothing
  const CUtensorMap *tmX = phase == 0 ? &tmX0 : (phase == 1 ? &tmX1 : (phase == 2 ? &tmX2 : &tmX3));
  // this CTA's range of pixel boxes
  const int TQ = (a.Q + a.BW - 1) / a.BW, TP = (a.P + a.BH - 1) / a.BH;
  const int TN = (a.N + a.BNi - 1) / a.BNi;
  const long long tiles = static_cast<long long>(TQ) * TP * TN;
  const int z = static_cast<int>(blockIdx.x);
  const long long tb = tiles * z / a.Z, te = tiles * (z + 1) / a.Z;
  const int T = static_cast<int>(te - tb);
  if (T <= 0) return;

  // Step s: pixel box tb + s of the dY grid; the X box this tap reads starts at
  // phase pixel (p0 + fr, q0 + fc). A step whose X box lies wholly outside the
  // phase view only adds zeros and is left out (no box without an element in
  // its tensor is ever loaded).
  const int Hp = (a.H - pr + st - 1) / st, Wp = (a.W - pc + st - 1) / st;
  struct Step {
    int n0, p0, q0;
    bool live;
  };
  auto step = [&](int s) {
    Step x;
    const long long t = tb + s;
    x.q0 = static_cast<int>(t % TQ) * a.BW;
    x.p0 = static_cast<int>((t / TQ) % TP) * a.BH;
    x.n0 = static_cast<int>(t / TQ / TP) * a.BNi;
    x.live = x.p0 + fr < Hp && x.p0 + fr + a.BH > 0 && x.q0 + fc < Wp && x.q0 + fc + a.BW > 0;
    return x;
  };
  int first_live = 0;
  while (first_live < T && !step(first_live).live) ++first_live;
  if (first_live == T) return;  // nothing to add

  const uint32_t tmem = conv_setup<C>(smem, sbase, warp);
  const Abort ab = make_abort(reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4), a.err,
                              a.timeout_ns);
  // boxes with an element in their tensor: dY's second 64 output channels exist
  // only if K > k0 + 64; X boxes only for channels below C. Rows of A (columns of
  // B) left unloaded hold stale values that reach only accumulator rows
  // (columns) past K (C), which are never stored.
  const int na = a.K > k0 + 64 ? 2 : 1;
  const int nb = min(BN / 64, (a.C - c0 + 63) / 64);
  const uint32_t tx = static_cast<uint32_t>(na + nb) * 8192u;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int s = first_live, u = 0; s < T; ++s) {
        const Step x = step(s);
        if (!x.live) continue;
        const int stg = u % C::NST;
        if (u >= C::NST && !mbar_wait(bar(C::B_EMPTY + stg), ((u / C::NST) - 1) & 1, ab)) break;
        const uint32_t sa = sbase + stg * C::STAGE;
        mbar_arrive_expect_tx(bar(C::B_FULL + stg), tx);
        for (int b = 0; b < na; ++b)
          tma_load_4d(sa + b * 8192, &tmdY, k0 + 64 * b, x.q0, x.p0, x.n0, bar(C::B_FULL + stg));
        for (int b = 0; b < nb; ++b)
          tma_load_4d(sa + C::A_BYTES + b * 8192, tmX, c0 + 64 * b, x.q0 + fc, x.p0 + fr, x.n0,
                      bar(C::B_FULL + stg));
        issued = ++u;
      }
      for (int u = max(0, issued - C::NST); u < issued; ++u)
        drain_wait(bar(C::B_FULL + u % C::NST), (u / C::NST) & 1, 2000000000ull);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_16_f32(128, BN, true, true, F16);
      for (int s = first_live, u = 0; s < T; ++s) {
        if (!step(s).live) continue;
        const int stg = u % C::NST;
        if (!mbar_wait(bar(C::B_FULL + stg), (u / C::NST) & 1, ab)) break;
        tc_fence_after();
        const uint32_t sa = opaque_u32(sbase + stg * C::STAGE);
        const uint64_t da = sdesc_sw128(sa, 8192, 1024);
        const uint64_t db = sdesc_sw128(sa + C::A_BYTES, 8192, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem, sdesc_add(da, kk * 2048), sdesc_add(db, kk * 2048), idesc,
                 (u > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(C::B_EMPTY + stg));
        ++u;
      }
      // the accumulator barrier arrives after every MMA (and every earlier commit)
      // has completed; wait for it here as well, so that no arrive is still in
      // flight when the CTA exits (also when no MMA was issued)
      mma_commit(bar(C::B_ACC));
      drain_wait(bar(C::B_ACC), 0, 2000000000ull);
    }
    __syncwarp();
  }

  // ------------------------------------------------------------ read-back: add into dW
  const int k = k0 + 32 * warp + lane;
  if (mbar_wait_warp(bar(C::B_ACC), 0, ab)) {
    tc_fence_after();
    float *dst = a.dW + ((static_cast<size_t>(k) * a.R + r) * a.S + sx) * a.C;
#pragma unroll
    for (int cc = 0; cc < BN / 32; ++cc) {
      uint32_t v[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + 32 * cc, v);
      tmem_wait_ld();
      const int cb = c0 + 32 * cc;
      if (k < a.K) {
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          if (cb + e < a.C)
            atomicAdd(reinterpret_cast<float4 *>(dst + cb + e),
                      make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                                  __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])));
      }
    }
  }
  conv_teardown<C>(tmem, warp);
}

int pow2_at_least(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// Pixel box of at most (exactly, with exact = true) `rows` pixels over a
// (n, rows-of-H, cols-of-W) grid: as wide as the image (a power of two when
// exact), then as tall, then several images.
void pixel_box(int N, int Hg, int Wg, int rows, bool exact, int &BW, int &BH, int &BNi) {
  if (exact) {
    BW = std::min(pow2_at_least(Wg), rows);
    BH = std::min(pow2_at_least(Hg), rows / BW);
    BNi = rows / (BW * BH);
  } else {
    BW = std::min(Wg, rows);
    BH = std::min(Hg, rows / BW);
    BNi = BH == Hg ? std::max(1, std::min(N, rows / (BW * BH))) : 1;
  }
}

template <int BN, bool F16>
cudaError_t launch_dgrad(const void *dY, const void *Wt, float *dX, const MgConvProblem &p,
                         unsigned int *err, cudaStream_t s) {
  using C = ConvCfg<BN>;
  const int st = p.stride;
  const long long K = p.K, C_ = p.C;
  CUtensorMap tdy, tw;
  DgradArgs a{};
  a.N = p.N; a.H = p.H; a.W = p.W; a.C = p.C; a.K = p.K; a.R = p.R; a.S = p.S;
  a.st = st; a.pad = p.pad; a.P = p.P; a.Q = p.Q;
  pixel_box(p.N, (p.H + st - 1) / st, (p.W + st - 1) / st, 128, false, a.BW, a.BH, a.BNi);
  {
    const long long dims[4] = {K, p.Q, p.P, p.N};
    const long long str[3] = {K * 2, static_cast<long long>(p.Q) * K * 2,
                              static_cast<long long>(p.P) * p.Q * K * 2};
    const int box[4] = {64, a.BW, a.BH, a.BNi};
    cudaError_t e = mg_tmap_16_4d(&tdy, dY, dims, str, box, F16);
    if (e != cudaSuccess) return e;
  }
  {
    const long long dims[4] = {C_, p.S, p.R, K};
    const long long str[3] = {C_ * 2, static_cast<long long>(p.S) * C_ * 2,
                              static_cast<long long>(p.R) * p.S * C_ * 2};
    const int box[4] = {64, 1, 1, 64};
    cudaError_t e = mg_tmap_16_4d(&tw, Wt, dims, str, box, F16);
    if (e != cudaSuccess) return e;
  }
  a.nphase = st * st;
  long long total = 0;
  for (int ph = 0; ph < a.nphase; ++ph) {
    const int hp = (p.H - ph / st + st - 1) / st, wp = (p.W - ph % st + st - 1) / st;
    const long long tiles = hp > 0 && wp > 0
                                ? static_cast<long long>((hp + a.BH - 1) / a.BH) *
                                      ((wp + a.BW - 1) / a.BW) * ((p.N + a.BNi - 1) / a.BNi)
                                : 0;
    total += tiles;
    a.tile_end[ph] = static_cast<int>(total);
  }
  if (total < 1 || total > 0x7fffffffLL) return cudaErrorInvalidValue;
  a.dX = dX;
  a.err = err;
  a.timeout_ns = mg_wait_limit_ns();
  auto kern = conv_dgrad_kernel<BN, F16>;
  cudaError_t e = mg_set_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM_BYTES,
                                   32 + (BN == 128 ? 1 : 0) + (F16 ? 2 : 0));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(total), static_cast<unsigned>((p.C + BN - 1) / BN));
  kern<<<grid, C::NTHREADS, C::SMEM_BYTES, s>>>(tdy, tw, a);
  return cudaGetLastError();
}

template <int BN, bool F16>
cudaError_t launch_wgrad(const void *X, const void *dY, float *dW, const MgConvProblem &p,
                         unsigned int *err, cudaStream_t s) {
  using C = ConvCfg<BN>;
  const int st = p.stride;
  const long long K = p.K, C_ = p.C;
  WgradArgs a{};
  a.N = p.N; a.H = p.H; a.W = p.W; a.C = p.C; a.K = p.K; a.R = p.R; a.S = p.S;
  a.st = st; a.pad = p.pad; a.P = p.P; a.Q = p.Q;
  pixel_box(p.N, p.P, p.Q, 64, true, a.BW, a.BH, a.BNi);
  CUtensorMap tdy, tx[4];
  {
    const long long dims[4] = {K, p.Q, p.P, p.N};
    const long long str[3] = {K * 2, static_cast<long long>(p.Q) * K * 2,
                              static_cast<long long>(p.P) * p.Q * K * 2};
    const int box[4] = {64, a.BW, a.BH, a.BNi};
    cudaError_t e = mg_tmap_16_4d(&tdy, dY, dims, str, box, F16);
    if (e != cudaSuccess) return e;
  }
  // phase views of X: rows pr, pr + st, ...; columns pc, pc + st, ...
  for (int ph = 0; ph < 4; ++ph) {
    const int pr = ph < st * st ? ph / st : 0, pc = ph < st * st ? ph % st : 0;
    const int hp = (p.H - pr + st - 1) / st, wp = (p.W - pc + st - 1) / st;
    if (ph < st * st && (hp < 1 || wp < 1)) a.phase_empty |= 1 << ph;
    const long long dims[4] = {C_, std::max(wp, 1), std::max(hp, 1), p.N};
    const long long str[3] = {C_ * 2 * st, static_cast<long long>(p.W) * C_ * 2 * st,
                              static_cast<long long>(p.H) * p.W * C_ * 2};
    const int box[4] = {64, a.BW, a.BH, a.BNi};
    const void *base = static_cast<const uint16_t *>(X) +
                       (static_cast<size_t>(pr) * p.W + pc) * static_cast<size_t>(p.C);
    cudaError_t e = mg_tmap_16_4d(&tx[ph], base, dims, str, box, F16);
    if (e != cudaSuccess) return e;
  }
  a.KB = (p.K + 127) / 128;
  const int CB = (p.C + BN - 1) / BN;
  const long long tiles = static_cast<long long>((p.Q + a.BW - 1) / a.BW) *
                          ((p.P + a.BH - 1) / a.BH) * ((p.N + a.BNi - 1) / a.BNi);
  // splits: about four CTAs per SM over the whole grid, at least 4 pixel boxes each
  const long long base = static_cast<long long>(a.KB) * CB * p.R * p.S;
  const long long want = (4LL * mg_sm_count() + base - 1) / base;
  a.Z = static_cast<int>(std::max(1LL, std::min(want, tiles / 4)));
  a.dW = dW;
  a.err = err;
  a.timeout_ns = mg_wait_limit_ns();
  auto kern = conv_wgrad_kernel<BN, F16>;
  cudaError_t e = mg_set_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM_BYTES,
                                   36 + (BN == 128 ? 1 : 0) + (F16 ? 2 : 0));
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(a.Z), static_cast<unsigned>(p.R * p.S),
                  static_cast<unsigned>(a.KB * CB));
  kern<<<grid, C::NTHREADS, C::SMEM_BYTES, s>>>(tdy, tx[0], tx[1], tx[2], tx[3], a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t mg_launch_conv_dgrad(const void *dY, const void *Wt, float *dX,
                                 const MgConvProblem &p, unsigned int *err, cudaStream_t s) {
  const bool wide = p.C > 64;
  if (p.f16) return wide ? launch_dgrad<128, true>(dY, Wt, dX, p, err, s)
                         : launch_dgrad<64, true>(dY, Wt, dX, p, err, s);
  return wide ? launch_dgrad<128, false>(dY, Wt, dX, p, err, s)
              : launch_dgrad<64, false>(dY, Wt, dX, p, err, s);
}

cudaError_t mg_launch_conv_wgrad(const void *X, const void *dY, float *dW,
                                 const MgConvProblem &p, unsigned int *err, cudaStream_t s) {
  const bool wide = p.C > 64;
  if (p.f16) return wide ? launch_wgrad<128, true>(X, dY, dW, p, err, s)
                         : launch_wgrad<64, true>(X, dY, dW, p, err, s);
  return wide ? launch_wgrad<128, false>(X, dY, dW, p, err, s)
              : launch_wgrad<64, false>(X, dY, dW, p, err, s);
}
