// accel_dkdv_pp.cu -- ACCEL_BF16 dK/dV kernel of the two-pass backward with two
// query blocks in flight ("ping-pong"), on tcgen05 tensor cores.
//
// "Meganeura: Portable GPU Training and Inference through Vulkan and Metal"
// splits the attention derivative into a dQ kernel and a fused dK+dV kernel
// (Section 3.3; Section 8 makes fused dK+dV an invariant). This file is the
// fused dK+dV kernel; the dQ pass is accel_dq.cu. Derivative operands keep f32
// accumulation (Sections 3.1 and 4.2); P and dS are rounded to bf16 only where
// they enter an MMA.
//
// Per CTA: keys k0 .. k0+127 of one (b, h) head (TMEM lanes = keys). K and V are
// loaded once; the query axis is walked in blocks of 64 rows, Q and dO (plus
// LSE and Dvec) through a 4-stage ring. Per query block i:
//   S^T  = K Q_i^T            dP^T = V dO_i^T            (TMEM, f32)
//   P^T  = exp2(S^T scale log2e - LSE_i log2e), masked   dS^T = P^T (dP^T - Dvec_i)
//   dV  += P^T dO_i           dK  += dS^T Q_i            (A operands from TMEM, bf16)
// Two softmax warpgroups take alternate blocks, each with its own S^T / dP^T
// columns in TMEM, so the tensor core computes S and dP of block i+1 while one
// warpgroup turns block i into P and dS, and the other warpgroup's block keeps
// the MMA queue fed in turn. MMA issue order: S(i+1), dP(i+1), dV(i), dK(i).
// TMEM columns: dV [0, DP), dK [DP, 2 DP), then per warpgroup w: S^T at
// 2 DP + 128 w (64 columns), dP^T at 2 DP + 128 w + 64 (64 columns). P^T and
// dS^T (bf16, two per column) overwrite the first 32 columns of their S^T and
// dP^T after those were read.
// Warp roles: 0-3 softmax warpgroup 0 (even blocks), 4-7 warpgroup 1 (odd
// blocks), 8 TMA producer (plus LSE/Dvec staging), 9 MMA issuer. Every wait is
// bounded; on a give-up the CTA sets the device error word and leaves through the
// normal teardown (own copies and MMAs drained first).
#include <climits>

#include "internal.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace {

using namespace mg_tc;

template <int DP>
struct PPCfg {
  static constexpr int BN = 128;   // keys per CTA
  static constexpr int BQ = 64;    // queries per block
  static constexpr int NQS = 4;    // Q/dO/LSE/Dvec ring stages
  static constexpr int NCHUNK = DP / 64;
  static constexpr int KV_TILE = BN * DP * 2;
  static constexpr int BOX_KV = BN * 128;
  static constexpr int Q_TILE = BQ * DP * 2;
  static constexpr int BOX_Q = BQ * 128;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_TILE;
  static constexpr int OFF_Q = OFF_V + KV_TILE;           // NQS stages
  static constexpr int OFF_DO = OFF_Q + NQS * Q_TILE;     // NQS stages
  static constexpr int OFF_LSE = OFF_DO + NQS * Q_TILE;   // NQS x BQ f32
  static constexpr int OFF_DV = OFF_LSE + NQS * BQ * 4;   // NQS x BQ f32
  static constexpr int OFF_BAR = OFF_DV + NQS * BQ * 4;
  static constexpr int B_KVFULL = 0;
  static constexpr int B_QFULL = 1;                  // NQS
  static constexpr int B_QEMPTY = B_QFULL + NQS;     // NQS
  static constexpr int B_SFULL = B_QEMPTY + NQS;     // 2 (warpgroup)
  static constexpr int B_DPFULL = B_SFULL + 2;       // 2
  static constexpr int B_PREADY = B_DPFULL + 2;      // 2
  static constexpr int B_DSREADY = B_PREADY + 2;     // 2
  static constexpr int B_ACCDONE = B_DSREADY + 2;
  static constexpr int B_DRAIN = B_ACCDONE + 1;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int NTHREADS = 320;
  static constexpr int TMEM_COLS = 512;
  static constexpr int T_DV = 0;
  static constexpr int T_DK = DP;
  static constexpr int T_W = 2 * DP;   // + 128 w: S^T, + 64: dP^T
  static_assert(T_W + 256 <= TMEM_COLS, "TMEM column budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return false;
  }
  return true;
}

template <int DP, bool F16>
__global__ void __launch_bounds__(320, 1)
    accel_dkdv_pp_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmdO, const float *__restrict__ LSE,
                         const float *__restrict__ Dvec, void *__restrict__ dK,
                         void *__restrict__ dV, int out16, int BH, int L, int Lk_rows, int D, int causal,
                         int off0, float scale, float scale_log2, unsigned int *err,
                         unsigned long long timeout_ns, const int *__restrict__ kv_len, int H,
                         int br, int hilo) {
  using C = PPCfg<DP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  float *sLse = reinterpret_cast<float *>(smem + C::OFF_LSE);
  float *sDv = reinterpret_cast<float *>(smem + C::OFF_DV);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Head-major order: CTAs that run together share a few heads' Q/dO in L2;
  // within a head the heaviest causal key block (kb = 0) goes first.
  // L query rows, Lk_rows key rows of which this head attends to Lk (all, or
  // the batch element's padded length); causal: query i sees key j iff
  // j <= i + off
  const int nkb = (Lk_rows + C::BN - 1) / C::BN;
  const int bh = static_cast<int>(blockIdx.x / nkb);
  const int kb = static_cast<int>(blockIdx.x % nkb);
  const int k0 = kb * C::BN;
  const MgKeys keys = mg_keys(kv_len, bh, H, L, Lk_rows, off0, br);
  const int Lk = keys.len, off = keys.off;
  const int nqb = (L + C::BQ - 1) / C::BQ;
  const int qb0 = causal ? max(0, k0 - off) / C::BQ : 0;  // first block with a query seeing k0
  const int n = k0 >= Lk ? 0 : max(0, nqb - qb0);

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 256) {
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i >= C::B_QEMPTY && i < C::B_QEMPTY + C::NQS) cnt = 1 + 4;
      if (i >= C::B_PREADY && i < C::B_DSREADY + 2) cnt = 4;
      mbar_init(bar(i), cnt);
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab = make_abort(abort_flag, err, timeout_ns);

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::B_KVFULL), 2 * C::KV_TILE);
      for (int c = 0; c < C::NCHUNK; ++c) {
        tma_load_3d(sbase + C::OFF_K + c * C::BOX_KV, &tmK, c * 64, k0, bh, bar(C::B_KVFULL));
        tma_load_3d(sbase + C::OFF_V + c * C::BOX_KV, &tmV, c * 64, k0, bh, bar(C::B_KVFULL));
      }
    }
    int issued = 0;
    for (int i = 0; i < n; ++i) {
      const int st = i % C::NQS;
      if (i >= C::NQS && !mbar_wait_warp(bar(C::B_QEMPTY + st), ((i / C::NQS) - 1) & 1, ab))
        break;
      const int q0 = (qb0 + i) * C::BQ;
      // LSE (pre-scaled to base 2; +inf past L so that P = 0 there) and Dvec.
      for (int r = lane; r < C::BQ; r += 32) {
        const int qg = q0 + r;
        const bool v = qg < L;
        // +inf also for a row with an empty softmax (LSE = -inf): its P is 0
        const float lse = v ? LSE[static_cast<size_t>(bh) * L + qg] : -INFINITY;
        sLse[st * C::BQ + r] = lse == -INFINITY ? INFINITY : lse * kLog2e;
        sDv[st * C::BQ + r] = v ? Dvec[static_cast<size_t>(bh) * L + qg] : 0.f;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::B_QFULL + st), 2 * C::Q_TILE);
        for (int c = 0; c < C::NCHUNK; ++c) {
          tma_load_3d(sbase + C::OFF_Q + st * C::Q_TILE + c * C::BOX_Q, &tmQ, c * 64, q0, bh,
                      bar(C::B_QFULL + st));
          tma_load_3d(sbase + C::OFF_DO + st * C::Q_TILE + c * C::BOX_Q, &tmdO, c * 64, q0, bh,
                      bar(C::B_QFULL + st));
        }
      }
      issued = i + 1;
    }
    if (lane == 0) {
      drain_wait(bar(C::B_KVFULL), 0, 2000000000ull);
      for (int i = max(0, issued - C::NQS); i < issued; ++i)
        drain_wait(bar(C::B_QFULL + i % C::NQS), (i / C::NQS) & 1, 2000000000ull);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idSP = idesc_16_f32(128, C::BQ, false, false, F16);
      constexpr uint32_t idKV = idesc_16_f32(128, DP, false, true, F16);
      bool ok = mbar_wait(bar(C::B_KVFULL), 0, ab);
      // base descriptors; each MMA adds a compile-time byte offset
      const uint32_t sb = opaque_u32(sbase);
      const uint64_t dK0 = sdesc_sw128(sb + C::OFF_K, 0, 1024);
      const uint64_t dV0 = sdesc_sw128(sb + C::OFF_V, 0, 1024);
      const uint64_t dQ0 = sdesc_sw128(sb + C::OFF_Q, 0, 1024);
      const uint64_t dO0 = sdesc_sw128(sb + C::OFF_DO, 0, 1024);
      const uint64_t dQmn = sdesc_sw128(sb + C::OFF_Q, C::BOX_Q, 1024);
      const uint64_t dOmn = sdesc_sw128(sb + C::OFF_DO, C::BOX_Q, 1024);
      // X^T = A * B_i^T with A in {K, V}, B_i in {Q_i, dO_i}; both K-major.
      auto issue_T = [&](uint64_t dA_, uint64_t dB_, uint32_t d) {
        // opaque copies: the per-step descriptors are formed here, not hoisted
        const uint64_t dA = opaque_u64(dA_), dB = opaque_u64(dB_);
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk) {
          const uint32_t oa = (kk >> 2) * C::BOX_KV + (kk & 3) * 32;
          const uint32_t ob = (kk >> 2) * C::BOX_Q + (kk & 3) * 32;
          mma_ss(d, sdesc_add(dA, oa), sdesc_add(dB, ob), idSP, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_SdP = [&](int i) -> bool {
        const int st = i % C::NQS, w = i & 1;
        if (!mbar_wait(bar(C::B_QFULL + st), (i / C::NQS) & 1, ab)) return false;
        tc_fence_after();
        const uint32_t tw = tmem + C::T_W + 128 * w;
        issue_T(dK0, sdesc_add(dQ0, st * C::Q_TILE), tw);
        mma_commit(bar(C::B_SFULL + w));
        issue_T(dV0, sdesc_add(dO0, st * C::Q_TILE), tw + 64);
        mma_commit(bar(C::B_DPFULL + w));
        return true;
      };
      // acc (+)= X^T (TMEM, bf16, 64 queries in 32 columns) * Y_i (MN-major smem)
      auto issue_acc = [&](uint32_t tA, uint64_t dY_, uint32_t d, bool first) {
        const uint64_t dY = opaque_u64(dY_);
        const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk)
          mma_ts(d, tA + 8 * kk, sdesc_add(dY, kk * 2048), idKV, kk > 0 ? 1u : acc0);
      };
      if (ok && n > 0) ok = issue_SdP(0);
      for (int i = 0; ok && i < n; ++i) {
        const int st = i % C::NQS, w = i & 1;
        const uint32_t tw = tmem + C::T_W + 128 * w;
        if (i + 1 < n && !(ok = issue_SdP(i + 1))) break;
        if (!(ok = mbar_wait(bar(C::B_PREADY + w), (i >> 1) & 1, ab))) break;
        tc_fence_after();
        issue_acc(tw, sdesc_add(dOmn, st * C::Q_TILE), tmem + C::T_DV, i == 0);
        if (!(ok = mbar_wait(bar(C::B_DSREADY + w), (i >> 1) & 1, ab))) break;
        tc_fence_after();
        issue_acc(tw + 64, sdesc_add(dQmn, st * C::Q_TILE), tmem + C::T_DK, i == 0);
        // hi/lo policy: dK also accumulates the lo part of dS^T (dP^T columns 32..63)
        if (hilo) issue_acc(tw + 96, sdesc_add(dQmn, st * C::Q_TILE), tmem + C::T_DK, false);
        mma_commit(bar(C::B_QEMPTY + st));
      }
      mma_commit(bar(C::B_ACCDONE));
      mma_commit(bar(C::B_DRAIN));
      drain_wait(bar(C::B_DRAIN), 0, 2000000000ull);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax warpgroups
    const int w = warp >> 2;
    const int quarter = warp & 3;
    const int kr = 32 * quarter + lane;  // key row within the block = TMEM lane
    const int kg = k0 + kr;
    const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
    const uint32_t tS = tmem + lane_off + C::T_W + 128 * w;
    const uint32_t tDP = tS + 64;
    // smallest query index that may see this thread's key (past Lk: none may)
    const int qmin = kg >= Lk ? INT_MAX : (causal ? kg - off : INT_MIN);
    bool ok = true;
    for (int i = w; i < n; i += 2) {
      const int st = i % C::NQS;
      const int q0 = (qb0 + i) * C::BQ;
      const uint32_t ph = (i >> 1) & 1;
      if (!(ok = mbar_wait_warp(bar(C::B_QFULL + st), (i / C::NQS) & 1, ab))) break;
      if (!(ok = mbar_wait_warp(bar(C::B_SFULL + w), ph, ab))) break;
      tc_fence_after();
      // query column e of the block is masked iff e < lim0 (e is q - q0)
      const int lim0 =
          qmin == INT_MIN ? INT_MIN : (qmin == INT_MAX ? INT_MAX : qmin - q0);
      const bool need_mask = lim0 > 0;
      const float *lse = sLse + st * C::BQ;
      const float *dvq = sDv + st * C::BQ;
      float p[C::BQ];
      {
        uint32_t r[64];
        tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(r));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 64; e += 4) {
          const float4 l4 = *reinterpret_cast<const float4 *>(lse + e);
          p[e] = ex2(fmaf(__uint_as_float(r[e]), scale_log2, -l4.x));
          p[e + 1] = ex2(fmaf(__uint_as_float(r[e + 1]), scale_log2, -l4.y));
          p[e + 2] = ex2(fmaf(__uint_as_float(r[e + 2]), scale_log2, -l4.z));
          p[e + 3] = ex2(fmaf(__uint_as_float(r[e + 3]), scale_log2, -l4.w));
        }
        if (need_mask) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (e < lim0) p[e] = 0.f;
        }
      }
      // P^T over the first 32 columns of S^T (already read)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack16<F16>(p[32 * c + 2 * e], p[32 * c + 2 * e + 1]);
        tmem_st16(tS + 16 * c, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_PREADY + w));

      if (!(ok = mbar_wait_warp(bar(C::B_DPFULL + w), ph, ab))) break;
      tc_fence_after();
      {
        uint32_t r[64];
        tmem_ld32(tDP, *reinterpret_cast<uint32_t(*)[32]>(r));
        tmem_ld32(tDP + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
        tmem_wait_ld();
        // dS^T over the first 32 columns of dP^T, 16 columns (32 queries) at a time;
        // under the hi/lo policy its lo part over columns 32..63
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const int q = 32 * c + e;
            const float4 d4 = *reinterpret_cast<const float4 *>(dvq + q);
            const float s0 = p[q] * (__uint_as_float(r[q]) - d4.x);
            const float s1 = p[q + 1] * (__uint_as_float(r[q + 1]) - d4.y);
            const float s2 = p[q + 2] * (__uint_as_float(r[q + 2]) - d4.z);
            const float s3 = p[q + 3] * (__uint_as_float(r[q + 3]) - d4.w);
            pk[e / 2] = pack16<F16>(s0, s1);
            pk[e / 2 + 1] = pack16<F16>(s2, s3);
          }
          tmem_st16(tDP + 16 * c, pk);
          if (hilo) {
            // the same dS values again (same arithmetic, same result), split
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const int q = 32 * c + e;
              const float4 d4 = *reinterpret_cast<const float4 *>(dvq + q);
              uint32_t h;
              pack16_hilo<F16>(p[q] * (__uint_as_float(r[q]) - d4.x),
                               p[q + 1] * (__uint_as_float(r[q + 1]) - d4.y), h, pk[e / 2]);
              pack16_hilo<F16>(p[q + 2] * (__uint_as_float(r[q + 2]) - d4.z),
                               p[q + 3] * (__uint_as_float(r[q + 3]) - d4.w), h, pk[e / 2 + 1]);
            }
            tmem_st16(tDP + 32 + 16 * c, pk);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(C::B_DSREADY + w));
        mbar_arrive(bar(C::B_QEMPTY + st));
      }
    }
    // dK (scaled) and dV of this key block: warpgroup w stores half the columns
    if (ok && n > 0) ok = mbar_wait_warp(bar(C::B_ACCDONE), 0, ab);
    if (ok && n == 0 && kg < Lk_rows) {
      // no query sees this key block: dK = dV = 0 (warpgroup w writes its half)
      const size_t row = (static_cast<size_t>(bh) * Lk_rows + kg) * D;
      for (int c = 0; c < DP / 2 && w * (DP / 2) + c < D; c += 4) {
        store4<F16>(dV, out16, row + w * (DP / 2) + c, 0.f, 0.f, 0.f, 0.f);
        store4<F16>(dK, out16, row + w * (DP / 2) + c, 0.f, 0.f, 0.f, 0.f);
      }
    }
    if (ok && n > 0) {
      tc_fence_after();
      const bool valid = kg < Lk_rows;
      const size_t row = (static_cast<size_t>(bh) * Lk_rows + (valid ? kg : 0)) * D;
#pragma unroll
      for (int c = 0; c < DP / 64; ++c) {
        const int col = w * (DP / 2) + 32 * c;
        uint32_t rv[32], rk[32];
        tmem_ld32(tmem + lane_off + C::T_DV + col, rv);
        tmem_ld32(tmem + lane_off + C::T_DK + col, rk);
        tmem_wait_ld();
        if (valid && col < D) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            store4<F16>(dV, out16, row + col + e, __uint_as_float(rv[e]),
                        __uint_as_float(rv[e + 1]), __uint_as_float(rv[e + 2]),
                        __uint_as_float(rv[e + 3]));
            store4<F16>(dK, out16, row + col + e, __uint_as_float(rk[e]) * scale,
                        __uint_as_float(rk[e + 1]) * scale, __uint_as_float(rk[e + 2]) * scale,
                        __uint_as_float(rk[e + 3]) * scale);
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  // Reconverge single-lane roles first: __syncthreads is an aligned barrier.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int DP, bool F16>
cudaError_t launch(const void *Q, const void *K, const void *V, const void *dO, const float *LSE,
                   const float *Dvec, void *dK, void *dV, const MgProblem &p, unsigned int *err,
                   cudaStream_t st) {
  using C = PPCfg<DP>;
  const int BH = p.B * p.H;
  CUtensorMap tq, tk, tv, tdo;
  cudaError_t e;
  if ((e = mg_tmap_16(&tq, Q, p.D, p.L, BH, C::BQ, F16)) != cudaSuccess) return e;
  if ((e = mg_tmap_16(&tdo, dO, p.D, p.L, BH, C::BQ, F16)) != cudaSuccess) return e;
  if ((e = mg_tmap_16(&tk, K, p.D, p.Lk, BH, C::BN, F16)) != cudaSuccess) return e;
  if ((e = mg_tmap_16(&tv, V, p.D, p.Lk, BH, C::BN, F16)) != cudaSuccess) return e;
  auto kern = accel_dkdv_pp_kernel<DP, F16>;
  if ((e = mg_set_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM_BYTES,
                            (DP == 64 ? 16 : 17) + (F16 ? 12 : 0))) != cudaSuccess)
    return e;
  const int nkb = (p.Lk + C::BN - 1) / C::BN;
  const long long grid = static_cast<long long>(nkb) * BH;
  kern<<<static_cast<unsigned>(grid), C::NTHREADS, C::SMEM_BYTES, st>>>(
      tq, tk, tv, tdo, LSE, Dvec, dK, dV, p.out16, BH, p.L, p.Lk, p.D, p.causal, p.off,
      p.scale, p.scale * kLog2e, err, mg_wait_limit_ns(), p.kv_len, p.H, p.br, p.hilo);
  return cudaGetLastError();
}

}  // namespace

cudaError_t mg_launch_accel_dkdv_pp(const void *Q, const void *K, const void *V, const void *dO,
                                    const float *LSE, const float *Dvec, void *dK, void *dV,
                                    const MgProblem &p, unsigned int *err, cudaStream_t st) {
  if (p.f16) {
    if (p.D <= 64) return launch<64, true>(Q, K, V, dO, LSE, Dvec, dK, dV, p, err, st);
    return launch<128, true>(Q, K, V, dO, LSE, Dvec, dK, dV, p, err, st);
  }
  if (p.D <= 64) return launch<64, false>(Q, K, V, dO, LSE, Dvec, dK, dV, p, err, st);
  return launch<128, false>(Q, K, V, dO, LSE, Dvec, dK, dV, p, err, st);
}
