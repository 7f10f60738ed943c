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
// Both kernels are persistent (one CTA per SM, work items strided over the
// grid) with 192 threads: warp 4 lane 0 issues TMA loads into an NST-stage ring
// that runs on across work items, warp 5 lane 0 issues the MMAs into one of two
// f32 accumulators (128 lanes x BN columns each) in tensor memory, and warps
// 0-3 read the other accumulator back (lane = accumulator row), so that the
// read-back of one item overlaps the main loop of the next. Every operand tile
// is a 4-D TMA box with 128-byte swizzle; coordinates outside the tensor read as
// zero, which supplies the convolution's zero padding and the tails of C and K.
//
// Input gradient. The output pixels are split by stride phase (h mod st,
// w mod st): within one phase, the taps that reach it are r = r0, r0+st, ... with
// r0 = (ph + pad) mod st, and tap r reads dY row i + (ph + pad - r) / st for
// phase row i -- a unit-stride window of dY. A tile is a box of phase pixels
// (BW x BH x BNi <= 128 rows = the MMA's M); the reduction runs over (tap,
// 64-channel chunk of K): A = the shifted dY box (K-major), B = Wt[k-chunk][r][s]
// [c-tile] (MN-major: c is contiguous). Rows past the box hold stale data and
// produce rows that are never stored. When the tiles are too few to fill the
// GPU (small images, the small-output case), each tile's reduction is split
// into groups whose partial sums are added into a zeroed dX with TMA f32
// add-reductions.
//
// Weight gradient. A CTA owns one tap (r, s), a 128-wide block of K and a BN
// block of C, and a range of pixel boxes (exactly 64 pixels each, zero-filled
// past the image); A = dY box^T (MN-major, k contiguous), B = the X box the tap
// reads (MN-major, c contiguous). With stride 2 the tap's input pixels
// (p*2 + r - pad) form a unit-stride box of one of four phase views of X (a
// tensor map whose row and column strides are doubled). Partial sums are added
// into dW (zeroed first) with TMA f32 add-reductions.
#include <stdint.h>
#include <stdlib.h>

#include <algorithm>

#include "internal.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace {

using namespace mg_tc;

template <int BN>
struct ConvCfg {
  static constexpr int BM = 128;                  // accumulator rows (MMA M)
  static constexpr int A_BYTES = BM * 128;        // 128 rows x 64 elements
  static constexpr int B_BYTES = BN * 128;        // BN/64 boxes of 64 rows x 128 bytes
  static constexpr int STAGE = A_BYTES + B_BYTES;
  // ring stages, continuous across work items: as many as fit beside the staging
  // ring (24, 32 or 48 KB a stage)
  static constexpr int NST = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
  // accumulator read-back staging: a ring of two 16 KB buffers, each one 32-column
  // chunk (dX: 128 pixel rows x 32 f32; dW: four warps' 32 rows x 32 f32, 4 KB a
  // warp), 128-byte rows with 128-byte swizzle
  static constexpr int OFF_STG = NST * STAGE;
  static constexpr int STG_CHUNK = BM * 128;
  static constexpr int OFF_BAR = OFF_STG + 2 * STG_CHUNK;
  static constexpr int B_FULL = 0;                // NST: stage loaded
  static constexpr int B_EMPTY = NST;             // NST: stage consumed by its MMAs
  static constexpr int B_AFULL = 2 * NST;         // 2: accumulator buffer complete
  static constexpr int B_AEMPTY = 2 * NST + 2;    // 2: accumulator buffer read out (4 warps)
  static constexpr int B_DRAIN = 2 * NST + 4;
  static constexpr int B_SFULL = 2 * NST + 5;     // 2: staging buffer written (4 warps, dX)
  static constexpr int B_SFREE = 2 * NST + 7;     // 2: staging buffer read by its TMA store
  static constexpr int NBAR = 2 * NST + 9;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int NTHREADS = 192;            // warps 0-3 read-back, 4 TMA, 5 MMA
  static constexpr int TMEM_COLS = 2 * BN;        // two accumulator buffers
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
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
  int tile_end[4];     // prefix sums of the pixel tiles of each phase
  int CB;              // BN-wide blocks of C
  int G;               // groups the reduction steps of a tile are split into
  int items;           // tiles * CB * G
  float *dX;           // G > 1: zeroed by the launcher, partial sums added
  unsigned int *err;
  unsigned long long timeout_ns;
};

struct WgradArgs {
  int N, H, W, C, K, R, S, st, pad, P, Q;
  int BW, BH, BNi;     // pixel box of one reduction step (exactly 64 pixels)
  int KB, CB;          // 128-row blocks of K, BN-wide blocks of C
  int Z;               // pixel-range splits
  int items;           // Z * R * S * KB * CB
  int phase_empty;     // bit (pr * st + pc): that phase view of X has no pixel
  float *dW;           // zeroed by the caller; partial sums added
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
  if (threadIdx.x == 128) {
    for (int i = 0; i < C::NBAR; ++i)
      mbar_init(sbase + C::OFF_BAR + 8u * i,
                (i == C::B_AEMPTY || i == C::B_AEMPTY + 1 || i == C::B_SFULL ||
                 i == C::B_SFULL + 1)
                    ? 4u
                    : 1u);
    *reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4) = 0;
    fence_barrier_init();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return *tmem_slot;
}

// Row m of a staged 128-byte-row chunk: 8 16-byte pieces, piece k stored at
// position k ^ (m mod 8) (the 128-byte swizzle the TMA store reads back).
__device__ __forceinline__ void stage_row(uint32_t row_addr, int m, const uint32_t (&r)[32]) {
#pragma unroll
  for (int k = 0; k < 8; ++k)
    st_shared_v4(row_addr + ((k ^ (m & 7)) << 4), r[4 * k], r[4 * k + 1], r[4 * k + 2],
                 r[4 * k + 3]);
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
// One work item: a pixel tile of one stride phase, a BN block of C, and group g
// of the tile's reduction steps (tap, 64-channel chunk of K).
struct DgradItem {
  int ph, pw, Hph, Wph, i0, j0, n0, c0;
  int r0, s0, ns, KC, sb, se;  // steps [sb, se) of the tile's nr * ns * KC
  int dr0, dq0;                // dY row (column) offset of the first tap r0 (s0)
};

__device__ __forceinline__ DgradItem dgrad_item(const DgradArgs &a, int item, int BN) {
  DgradItem d;
  const int g = item % a.G;
  const int cb = (item / a.G) % a.CB;
  int t = item / a.G / a.CB, phase = 0;
#pragma unroll
  for (int q = 0; q < 3; ++q)
    if (q + 1 < a.nphase && t >= a.tile_end[q]) phase = q + 1;
  if (phase > 0) t -= a.tile_end[phase - 1];
  const int st = a.st;
  d.ph = phase / st;
  d.pw = phase % st;
  d.Hph = (a.H - d.ph + st - 1) / st;
  d.Wph = (a.W - d.pw + st - 1) / st;
  const int TJ = (d.Wph + a.BW - 1) / a.BW, TI = (d.Hph + a.BH - 1) / a.BH;
  d.j0 = (t % TJ) * a.BW;
  d.i0 = ((t / TJ) % TI) * a.BH;
  d.n0 = (t / TJ / TI) * a.BNi;
  d.c0 = cb * BN;
  // taps that reach this phase: r = r0, r0 + st, ... (likewise s)
  d.r0 = (d.ph + a.pad) % st;
  d.s0 = (d.pw + a.pad) % st;
  const int nr = d.r0 < a.R ? (a.R - d.r0 + st - 1) / st : 0;
  d.ns = d.s0 < a.S ? (a.S - d.s0 + st - 1) / st : 0;
  d.KC = (a.K + 63) / 64;
  const int T = nr * d.ns * d.KC;
  d.sb = T * g / a.G;
  d.se = T * (g + 1) / a.G;
  d.dr0 = (d.ph + a.pad - d.r0) / st;  // exact; tap r0 + i st reads row offset dr0 - i
  d.dq0 = (d.pw + a.pad - d.s0) / st;
  return d;
}

// Steps of an item in order, without divisions per step. Step (ri, si, kc): K
// chunk kc of tap (r0 + ri st, s0 + si st), whose dY box starts at phase pixel
// (i0 + dr0 - ri, j0 + dq0 - si). A box wholly outside dY would only add zeros:
// such a step is not live and is left out, so that no load is ever issued for a
// box without an element in its tensor.
struct DgradSteps {
  int s, kc, si, ri;
  __device__ __forceinline__ DgradSteps(const DgradItem &d) : s(d.sb), kc(0), si(0), ri(0) {
    if (d.sb < d.se) {
      kc = d.sb % d.KC;
      const int rs = d.sb / d.KC;
      si = rs % d.ns;
      ri = rs / d.ns;
    }
  }
  __device__ __forceinline__ bool live(const DgradArgs &a, const DgradItem &d) const {
    const int i = d.i0 + d.dr0 - ri, j = d.j0 + d.dq0 - si;
    return i < a.P && i + a.BH > 0 && j < a.Q && j + a.BW > 0;
  }
  __device__ __forceinline__ void next(const DgradItem &d) {
    ++s;
    if (++kc == d.KC) {
      kc = 0;
      if (++si == d.ns) {
        si = 0;
        ++ri;
      }
    }
  }
};

template <int BN, bool F16>
__global__ void __launch_bounds__(192, 1)
    conv_dgrad_kernel(const __grid_constant__ CUtensorMap tmdY,
                      const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmO0,
                      const __grid_constant__ CUtensorMap tmO1,
                      const __grid_constant__ CUtensorMap tmO2,
                      const __grid_constant__ CUtensorMap tmO3, const __grid_constant__ DgradArgs a) {
  using C = ConvCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return sbase + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t tmem = conv_setup<C>(smem, sbase, warp);
  const Abort ab = make_abort(reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4), a.err,
                              a.timeout_ns);
  const uint32_t a_tx = static_cast<uint32_t>(a.BW * a.BH * a.BNi) * 128u;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int u = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < a.items; item += gridDim.x) {
        const DgradItem d = dgrad_item(a, item, BN);
        const int nbox = min(BN / 64, (a.C - d.c0 + 63) / 64);  // W boxes with a channel < C
        for (DgradSteps x(d); x.s < d.se; x.next(d)) {
          if (!x.live(a, d)) continue;
          const int stg = u % C::NST;
          if (u >= C::NST && !(ok = mbar_wait(bar(C::B_EMPTY + stg), ((u / C::NST) - 1) & 1, ab)))
            break;
          const uint32_t sa = sbase + stg * C::STAGE;
          const int r = d.r0 + x.ri * a.st, sx = d.s0 + x.si * a.st;
          mbar_arrive_expect_tx(bar(C::B_FULL + stg), a_tx + nbox * 8192u);
          tma_load_4d(sa, &tmdY, x.kc * 64, d.j0 + d.dq0 - x.si, d.i0 + d.dr0 - x.ri, d.n0,
                      bar(C::B_FULL + stg));
          for (int b = 0; b < nbox; ++b)
            tma_load_4d(sa + C::A_BYTES + b * 8192, &tmW, d.c0 + 64 * b, sx, r, x.kc * 64,
                        bar(C::B_FULL + stg));
          ++u;
        }
      }
      for (int v = max(0, u - C::NST); v < u; ++v)
        drain_wait(bar(C::B_FULL + v % C::NST), (v / C::NST) & 1, 2000000000ull);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_16_f32(128, BN, false, true, F16);
      int u = 0, it = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < a.items; item += gridDim.x, ++it) {
        const DgradItem d = dgrad_item(a, item, BN);
        const int buf = it & 1;
        if (it >= 2 && !(ok = mbar_wait(bar(C::B_AEMPTY + buf), ((it >> 1) - 1) & 1, ab))) break;
        tc_fence_after();
        const uint32_t acc = tmem + buf * BN;
        bool first = true;
        for (DgradSteps x(d); x.s < d.se; x.next(d)) {
          if (!x.live(a, d)) continue;
          const int stg = u % C::NST;
          if (!(ok = mbar_wait(bar(C::B_FULL + stg), (u / C::NST) & 1, ab))) break;
          tc_fence_after();
          const uint32_t sa = opaque_u32(sbase + stg * C::STAGE);
          const uint64_t da = sdesc_sw128(sa, 0, 1024);
          const uint64_t db = sdesc_sw128(sa + C::A_BYTES, 8192, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(acc, sdesc_add(da, kk * 32), sdesc_add(db, kk * 2048), idesc,
                   (!first || kk > 0) ? 1u : 0u);
          mma_commit(bar(C::B_EMPTY + stg));
          first = false;
          ++u;
        }
        mma_commit(bar(C::B_AFULL + buf));  // also when no step was live
      }
      // every arrive of the commits above lands before the CTA exits
      mma_commit(bar(C::B_DRAIN));
      drain_wait(bar(C::B_DRAIN), 0, 2000000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ read-back (warps 0-3)
    // Accumulator rows are the tile's pixels in box order. Per 32-channel chunk,
    // each thread stages its row in one of two shared-memory buffers and one
    // thread stores the pixel box with TMA (a phase view of dX: elements past the
    // image are not written), or adds it into the zeroed dX when the steps are
    // split. A buffer is refilled once the store two chunks back has read it; gc
    // counts the chunks staged so far (the same sequence in every thread).
    const int m = 32 * warp + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
    int it = 0, gc = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < a.items; item += gridDim.x, ++it) {
      const DgradItem d = dgrad_item(a, item, BN);
      bool any = false;
      for (DgradSteps x(d); x.s < d.se && !any; x.next(d)) any = x.live(a, d);
      const bool store = any || a.G == 1;  // no live step: zeros, or nothing to add
      const int buf = it & 1;
      if (!(ok = mbar_wait_warp(bar(C::B_AFULL + buf), (it >> 1) & 1, ab))) break;
      tc_fence_after();
      const int ph = d.ph * a.st + d.pw;
      const CUtensorMap *mo = ph == 0 ? &tmO0 : (ph == 1 ? &tmO1 : (ph == 2 ? &tmO2 : &tmO3));
      const int nch = store ? min(BN / 32, (a.C - d.c0 + 31) / 32) : 0;
      for (int cc = 0; cc < nch; ++cc, ++gc) {
        uint32_t r[32];
        if (any) {
          tmem_ld32(tmem + lane_off + buf * BN + 32 * cc, r);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = 0u;  // no tap reaches these pixels
        }
        if (cc == nch - 1) {  // the accumulator buffer is read out
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C::B_AEMPTY + buf));
        }
        const int sb = gc & 1;
        const uint32_t sa = sbase + C::OFF_STG + sb * C::STG_CHUNK;
        if (gc >= 2 && !(ok = mbar_wait_warp(bar(C::B_SFREE + sb), ((gc >> 1) - 1) & 1, ab)))
          break;
        stage_row(sa + m * 128, m, r);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_SFULL + sb));
        if (warp == 0) {
          if (!(ok = mbar_wait_warp(bar(C::B_SFULL + sb), (gc >> 1) & 1, ab))) break;
          if (lane == 0) {
            if (a.G == 1)
              tma_store_4d(mo, sa, d.c0 + 32 * cc, d.j0, d.i0, d.n0);
            else
              tma_reduce_add_4d(mo, sa, d.c0 + 32 * cc, d.j0, d.i0, d.n0);
            bulk_commit_group();
            // the previous chunk's store has read the other buffer
            bulk_wait_group_read1();
            if (gc >= 1) mbar_arrive(bar(C::B_SFREE + (sb ^ 1)));
          }
          __syncwarp();
        }
      }
      if (ok && nch == 0) {  // nothing to store: the accumulator is free at once
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_AEMPTY + buf));
      }
    }
    if (threadIdx.x == 0) bulk_wait_group0();
  }
  conv_teardown<C>(tmem, warp);
}

// ------------------------------------------------------------------ weight gradient
// One work item: pixel range z, tap (r, s), a 128-row block of K and a BN block
// of C. Step s: pixel box tb + s of the dY grid; the X box the tap reads starts
// at phase pixel (p0 + fr, q0 + fc) of phase view (pr, pc). A step whose X box
// lies wholly outside the view only adds zeros and is left out.
struct WgradItem {
  int r, sx, k0, c0, fr, fc, phase, Hp, Wp;
  int TQ, TP;
  int tb, te;  // pixel boxes [tb, te) of the dY grid
};

__device__ __forceinline__ WgradItem wgrad_item(const WgradArgs &a, int item, int BN) {
  WgradItem w;
  const int cb = item % a.CB;
  const int kb = (item / a.CB) % a.KB;
  const int tap = (item / a.CB / a.KB) % (a.R * a.S);
  const int z = item / a.CB / a.KB / (a.R * a.S);
  const int st = a.st;
  w.r = tap / a.S;
  w.sx = tap % a.S;
  w.k0 = kb * 128;
  w.c0 = cb * BN;
  const int ar = w.r - a.pad, as = w.sx - a.pad;
  const int pr = ((ar % st) + st) % st, pc = ((as % st) + st) % st;
  w.fr = (ar - pr) / st;
  w.fc = (as - pc) / st;
  w.phase = pr * st + pc;
  w.Hp = (a.H - pr + st - 1) / st;
  w.Wp = (a.W - pc + st - 1) / st;
  w.TQ = (a.Q + a.BW - 1) / a.BW;
  w.TP = (a.P + a.BH - 1) / a.BH;
  const long long tiles = static_cast<long long>(w.TQ) * w.TP * ((a.N + a.BNi - 1) / a.BNi);
  w.tb = static_cast<int>(tiles * z / a.Z);
  w.te = (a.phase_empty >> w.phase) & 1 ? w.tb : static_cast<int>(tiles * (z + 1) / a.Z);
  return w;
}

// Pixel boxes of an item in order, without divisions per step: box (qi, pi, ni)
// starts at dY pixel (n0, p0, q0) = (ni BNi, pi BH, qi BW).
struct WgradSteps {
  int t, q0, p0, n0;
  __device__ __forceinline__ WgradSteps(const WgradArgs &a, const WgradItem &w) : t(w.tb) {
    q0 = (t % w.TQ) * a.BW;
    p0 = ((t / w.TQ) % w.TP) * a.BH;
    n0 = (t / w.TQ / w.TP) * a.BNi;
  }
  __device__ __forceinline__ bool live(const WgradArgs &a, const WgradItem &w) const {
    return p0 + w.fr < w.Hp && p0 + w.fr + a.BH > 0 && q0 + w.fc < w.Wp && q0 + w.fc + a.BW > 0;
  }
  __device__ __forceinline__ void next(const WgradArgs &a, const WgradItem &w) {
    ++t;
    if ((q0 += a.BW) >= w.TQ * a.BW) {
      q0 = 0;
      if ((p0 += a.BH) >= w.TP * a.BH) {
        p0 = 0;
        n0 += a.BNi;
      }
    }
  }
};

template <int BN, bool F16>
__global__ void __launch_bounds__(192, 1)
    conv_wgrad_kernel(const __grid_constant__ CUtensorMap tmdY,
                      const __grid_constant__ CUtensorMap tmX0,
                      const __grid_constant__ CUtensorMap tmX1,
                      const __grid_constant__ CUtensorMap tmX2,
                      const __grid_constant__ CUtensorMap tmX3,
                      const __grid_constant__ CUtensorMap tmdW,
                      const __grid_constant__ WgradArgs a) {
  using C = ConvCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return sbase + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t tmem = conv_setup<C>(smem, sbase, warp);
  const Abort ab = make_abort(reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4), a.err,
                              a.timeout_ns);

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int u = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < a.items; item += gridDim.x) {
        const WgradItem w = wgrad_item(a, item, BN);
        const CUtensorMap *tmX =
            w.phase == 0 ? &tmX0 : (w.phase == 1 ? &tmX1 : (w.phase == 2 ? &tmX2 : &tmX3));
        // boxes with an element in their tensor: dY's second 64 output channels
        // exist only if K > k0 + 64; X boxes only for channels below C. Rows of
        // A (columns of B) left unloaded hold stale values that reach only
        // accumulator rows (columns) past K (C), which are never stored.
        const int na = a.K > w.k0 + 64 ? 2 : 1;
        const int nb = min(BN / 64, (a.C - w.c0 + 63) / 64);
        const uint32_t tx = static_cast<uint32_t>(na + nb) * 8192u;
        for (WgradSteps x(a, w); x.t < w.te; x.next(a, w)) {
          if (!x.live(a, w)) continue;
          const int stg = u % C::NST;
          if (u >= C::NST && !(ok = mbar_wait(bar(C::B_EMPTY + stg), ((u / C::NST) - 1) & 1, ab)))
            break;
          const uint32_t sa = sbase + stg * C::STAGE;
          mbar_arrive_expect_tx(bar(C::B_FULL + stg), tx);
          for (int b = 0; b < na; ++b)
            tma_load_4d(sa + b * 8192, &tmdY, w.k0 + 64 * b, x.q0, x.p0, x.n0,
                        bar(C::B_FULL + stg));
          for (int b = 0; b < nb; ++b)
            tma_load_4d(sa + C::A_BYTES + b * 8192, tmX, w.c0 + 64 * b, x.q0 + w.fc,
                        x.p0 + w.fr, x.n0, bar(C::B_FULL + stg));
          ++u;
        }
      }
      for (int v = max(0, u - C::NST); v < u; ++v)
        drain_wait(bar(C::B_FULL + v % C::NST), (v / C::NST) & 1, 2000000000ull);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_16_f32(128, BN, true, true, F16);
      int u = 0, it = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < a.items; item += gridDim.x, ++it) {
        const WgradItem w = wgrad_item(a, item, BN);
        const int buf = it & 1;
        if (it >= 2 && !(ok = mbar_wait(bar(C::B_AEMPTY + buf), ((it >> 1) - 1) & 1, ab))) break;
        tc_fence_after();
        const uint32_t acc = tmem + buf * BN;
        bool first = true;
        for (WgradSteps x(a, w); x.t < w.te; x.next(a, w)) {
          if (!x.live(a, w)) continue;
          const int stg = u % C::NST;
          if (!(ok = mbar_wait(bar(C::B_FULL + stg), (u / C::NST) & 1, ab))) break;
          tc_fence_after();
          const uint32_t sa = opaque_u32(sbase + stg * C::STAGE);
          const uint64_t da = sdesc_sw128(sa, 8192, 1024);
          const uint64_t db = sdesc_sw128(sa + C::A_BYTES, 8192, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(acc, sdesc_add(da, kk * 2048), sdesc_add(db, kk * 2048), idesc,
                   (!first || kk > 0) ? 1u : 0u);
          mma_commit(bar(C::B_EMPTY + stg));
          first = false;
          ++u;
        }
        mma_commit(bar(C::B_AFULL + buf));  // also when no step was live
      }
      mma_commit(bar(C::B_DRAIN));
      drain_wait(bar(C::B_DRAIN), 0, 2000000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ read-back: add into dW
    // Warp w owns accumulator rows k0 + 32w .. k0 + 32w + 31: per 32-channel chunk
    // it stages them in one of its two 4 KB buffers and adds them into dW with a
    // TMA reduction (a [K][R*S][C] view: rows past K and channels past C are not
    // written); a buffer is refilled once the reduction two chunks back has read
    // it (the warp's own bulk groups).
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
    const uint32_t stg = sbase + C::OFF_STG + warp * 2 * 32 * 128;
    int it = 0, gc = 0;
    for (int item = blockIdx.x; item < a.items; item += gridDim.x, ++it) {
      const WgradItem w = wgrad_item(a, item, BN);
      bool any = false;
      for (WgradSteps x(a, w); x.t < w.te && !any; x.next(a, w)) any = x.live(a, w);
      const int buf = it & 1;
      if (!mbar_wait_warp(bar(C::B_AFULL + buf), (it >> 1) & 1, ab)) break;
      tc_fence_after();
      const int nch =
          any && w.k0 + 32 * warp < a.K ? min(BN / 32, (a.C - w.c0 + 31) / 32) : 0;
      for (int cc = 0; cc < nch; ++cc, ++gc) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + buf * BN + 32 * cc, v);
        tmem_wait_ld();
        const uint32_t sa = stg + (gc & 1) * 32 * 128;
        if (lane == 0) bulk_wait_group_read1();
        __syncwarp();
        stage_row(sa + lane * 128, lane, v);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(&tmdW, sa, w.c0 + 32 * cc, w.r * a.S + w.sx, w.k0 + 32 * warp);
          bulk_commit_group();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_AEMPTY + buf));
    }
    if (lane == 0) bulk_wait_group0();
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

// Input-gradient tiling: the pixel box, the prefix sums of the tiles of each
// stride phase, their total, and the fewest reduction steps of a phase with pixels.
struct DgradGeom {
  int BW, BH, BNi;
  int tile_end[4];
  long long tiles;
  int tmin;
};

DgradGeom dgrad_geom(const MgConvProblem &p) {
  DgradGeom g{};
  const int st = p.stride;
  pixel_box(p.N, (p.H + st - 1) / st, (p.W + st - 1) / st, 128, false, g.BW, g.BH, g.BNi);
  g.tmin = 1 << 30;
  for (int ph = 0; ph < st * st; ++ph) {
    const int hp = (p.H - ph / st + st - 1) / st, wp = (p.W - ph % st + st - 1) / st;
    const long long n = hp > 0 && wp > 0
                            ? static_cast<long long>((hp + g.BH - 1) / g.BH) *
                                  ((wp + g.BW - 1) / g.BW) * ((p.N + g.BNi - 1) / g.BNi)
                            : 0;
    if (n > 0) {
      const int r0 = (ph / st + p.pad) % st, s0 = (ph % st + p.pad) % st;
      const int nr = r0 < p.R ? (p.R - r0 + st - 1) / st : 0;
      const int ns = s0 < p.S ? (p.S - s0 + st - 1) / st : 0;
      g.tmin = std::min(g.tmin, nr * ns * ((p.K + 63) / 64));
    }
    g.tiles += n;
    g.tile_end[ph] = static_cast<int>(std::min<long long>(g.tiles, 0x7fffffffLL));
  }
  return g;
}

// The reduction steps of each tile are split into groups (partial sums added into
// a zeroed dX) when there are at most half as many work items as SMs and at least
// 8 steps a tile.
bool dgrad_split(const DgradGeom &g, int C, int BN, int sms) {
  return 2 * g.tiles * ((C + BN - 1) / BN) <= sms && g.tmin >= 8;
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
  const DgradGeom geo = dgrad_geom(p);
  a.BW = geo.BW;
  a.BH = geo.BH;
  a.BNi = geo.BNi;
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
  for (int ph = 0; ph < 4; ++ph) a.tile_end[ph] = geo.tile_end[ph];
  a.CB = (p.C + BN - 1) / BN;
  // Split each tile's reduction steps into G groups (at least 4 steps each;
  // G * work <= SMs, one wave) whose partial sums are added into a zeroed dX.
  const long long work = geo.tiles * a.CB;
  const int sms = mg_sm_count();
  a.G = 1;
  if (dgrad_split(geo, p.C, BN, sms))
    a.G = static_cast<int>(std::min<long long>({sms / work, geo.tmin / 4, 8}));
  if (work * a.G > 0x7fffffffLL || work < 1) return cudaErrorInvalidValue;
  a.items = static_cast<int>(work * a.G);
  a.dX = dX;
  a.err = err;
  a.timeout_ns = mg_wait_limit_ns();
  if (a.G > 1) {
    cudaError_t e = cudaMemsetAsync(dX, 0, static_cast<size_t>(p.N) * p.H * p.W * p.C * 4, s);
    if (e != cudaSuccess) return e;
  }
  // phase views of dX (f32): rows ph, ph + st, ...; columns pw, pw + st, ...
  CUtensorMap to[4];
  for (int ph = 0; ph < 4; ++ph) {
    const int pr = ph < st * st ? ph / st : 0, pc = ph < st * st ? ph % st : 0;
    const int hp = (p.H - pr + st - 1) / st, wp = (p.W - pc + st - 1) / st;
    const long long dims[4] = {C_, std::max(wp, 1), std::max(hp, 1), p.N};
    const long long str[3] = {C_ * 4 * st, static_cast<long long>(p.W) * C_ * 4 * st,
                              static_cast<long long>(p.H) * p.W * C_ * 4};
    const int box[4] = {32, a.BW, a.BH, a.BNi};
    cudaError_t e = mg_tmap_f32_nd(&to[ph], dX + (static_cast<size_t>(pr) * p.W + pc) * p.C, 4,
                                   dims, str, box);
    if (e != cudaSuccess) return e;
  }
  auto kern = conv_dgrad_kernel<BN, F16>;
  cudaError_t e = mg_set_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM_BYTES,
                                   32 + 2 * (BN / 128) + (F16 ? 1 : 0));
  if (e != cudaSuccess) return e;
  const int grid = std::min(a.items, sms);
  kern<<<grid, C::NTHREADS, C::SMEM_BYTES, s>>>(tdy, tw, to[0], to[1], to[2], to[3], a);
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
  a.CB = (p.C + BN - 1) / BN;
  const long long tiles = static_cast<long long>((p.Q + a.BW - 1) / a.BW) *
                          ((p.P + a.BH - 1) / a.BH) * ((p.N + a.BNi - 1) / a.BNi);
  // pixel-range splits: about two work items per SM, at least 4 pixel boxes each
  const long long base = static_cast<long long>(a.KB) * a.CB * p.R * p.S;
  const int sms = mg_sm_count();
  const long long want = (2LL * sms + base - 1) / base;
  a.Z = static_cast<int>(std::max(1LL, std::min(want, tiles / 4)));
  if (base * a.Z > 0x7fffffffLL) return cudaErrorInvalidValue;
  a.items = static_cast<int>(base * a.Z);
  a.dW = dW;
  a.err = err;
  a.timeout_ns = mg_wait_limit_ns();
  // dW as [K][R*S][C] f32, boxes of 32 channels x 1 tap x 32 output channels
  CUtensorMap tdw;
  {
    const long long dims[3] = {C_, static_cast<long long>(p.R) * p.S, K};
    const long long str[2] = {C_ * 4, static_cast<long long>(p.R) * p.S * C_ * 4};
    const int box[3] = {32, 1, 32};
    cudaError_t e = mg_tmap_f32_nd(&tdw, dW, 3, dims, str, box);
    if (e != cudaSuccess) return e;
  }
  auto kern = conv_wgrad_kernel<BN, F16>;
  cudaError_t e = mg_set_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM_BYTES,
                                   40 + 2 * (BN / 128) + (F16 ? 1 : 0));
  if (e != cudaSuccess) return e;
  const int grid = std::min(a.items, sms);
  kern<<<grid, C::NTHREADS, C::SMEM_BYTES, s>>>(tdy, tx[0], tx[1], tx[2], tx[3], tdw, a);
  return cudaGetLastError();
}

}  // namespace

// Accumulator width N (columns of C per work item): 64 for C <= 64, 256 for
// C >= 256 (a quarter fewer operand bytes per FLOP through shared memory than
// N = 128, which an M = 128 product with both operands there would saturate at
// the full tensor rate), else 128. MG_CONV_MAX_N=128 or 64 caps it.
int conv_bn(int C) {
  static const int cap = [] {
    const char *v = getenv("MG_CONV_MAX_N");
    const int c = v ? atoi(v) : 256;
    return c >= 256 ? 256 : (c >= 128 ? 128 : 64);
  }();
  const int bn = C >= 256 ? 256 : (C > 64 ? 128 : 64);
  return std::min(bn, cap);
}

cudaError_t mg_launch_conv_dgrad(const void *dY, const void *Wt, float *dX,
                                 const MgConvProblem &p, unsigned int *err, cudaStream_t s) {
  int bn = conv_bn(p.C);
  if (bn == 256) {
    // 128-wide tiles where 256-wide ones would need the split reduction (a zeroed
    // dX and added partial sums) that 128-wide ones do without
    const DgradGeom g = dgrad_geom(p);
    const int sms = mg_sm_count();
    if (dgrad_split(g, p.C, 256, sms) && !dgrad_split(g, p.C, 128, sms)) bn = 128;
  }
  switch (bn * 2 + (p.f16 ? 1 : 0)) {
    case 513: return launch_dgrad<256, true>(dY, Wt, dX, p, err, s);
    case 512: return launch_dgrad<256, false>(dY, Wt, dX, p, err, s);
    case 257: return launch_dgrad<128, true>(dY, Wt, dX, p, err, s);
    case 256: return launch_dgrad<128, false>(dY, Wt, dX, p, err, s);
    case 129: return launch_dgrad<64, true>(dY, Wt, dX, p, err, s);
    default: return launch_dgrad<64, false>(dY, Wt, dX, p, err, s);
  }
}

cudaError_t mg_launch_conv_wgrad(const void *X, const void *dY, float *dW,
                                 const MgConvProblem &p, unsigned int *err, cudaStream_t s) {
  switch (conv_bn(p.C) * 2 + (p.f16 ? 1 : 0)) {
    case 513: return launch_wgrad<256, true>(X, dY, dW, p, err, s);
    case 512: return launch_wgrad<256, false>(X, dY, dW, p, err, s);
    case 257: return launch_wgrad<128, true>(X, dY, dW, p, err, s);
    case 256: return launch_wgrad<128, false>(X, dY, dW, p, err, s);
    case 129: return launch_wgrad<64, true>(X, dY, dW, p, err, s);
    default: return launch_wgrad<64, false>(X, dY, dW, p, err, s);
  }
}
