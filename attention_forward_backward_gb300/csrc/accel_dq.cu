// accel_dq.cu -- ACCEL_BF16 dQ pass of the attention backward on tcgen05.
//
// The dQ archetype of "Meganeura: Portable GPU Training and Inference through
// Vulkan and Metal" (Section 3.3: the derivative is split into a dQ kernel and a
// fused dK+dV kernel; Section 7.3 profiles the pair). Here it is its own pass
// over 128-row query blocks, so that dQ is accumulated in tensor memory and
// stored once, without atomics or reductions:
//
//   for every key tile j (128 keys) the query block attends to:
//     S   = Q K_j^T                  (TMEM, f32; Q resident in smem)
//     dP  = dO V_j^T                 (TMEM, f32; dO resident in smem)
//     P   = exp2(S scale log2e - LSE log2e), masked    (one thread per row)
//     dS  = P (dP - Dvec), rounded to bf16 into the S columns
//     dQ += dS K_j                   (A = dS from TMEM, B = K_j from smem)
//   dQ = scale * dQ                  (TMEM -> global, f32)
//
// S is double-buffered in TMEM so that S(j+2) is computed while the softmax
// warps work on tile j+1; the issue order per tile is dQ(j), dP(j+1), S(j+2).
// Warps 0-3 and 4-7 are two warpgroups splitting the 128 key columns of a tile
// (64 each; thread = query row = TMEM lane); warp 8 is the TMA producer
// (separate K and V rings, since K_j is needed until dQ(j) and V_j only until
// dP(j)), warp 9 issues the MMAs. Every wait is bounded.
#include "internal.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace {

using namespace mg_tc;

template <int DP>
struct DqCfg {
  static constexpr int BM = 128;  // query rows per CTA (TMEM lanes)
  static constexpr int BN = 128;  // keys per tile
  static constexpr int NKS = 3;   // K ring: K_j lives from S(j) to dQ(j)
  static constexpr int NVS = 2;   // V ring: V_j lives from dP(j) issue to completion
  static constexpr int NCHUNK = DP / 64;
  static constexpr int Q_TILE = BM * DP * 2;
  static constexpr int KV_TILE = BN * DP * 2;
  static constexpr int BOX_Q = BM * 128;
  static constexpr int BOX_KV = BN * 128;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + Q_TILE;
  static constexpr int OFF_K = OFF_DO + Q_TILE;
  static constexpr int OFF_V = OFF_K + NKS * KV_TILE;
  static constexpr int OFF_BAR = OFF_V + NVS * KV_TILE;
  static constexpr int B_QFULL = 0;
  static constexpr int B_KFULL = 1;                  // NKS
  static constexpr int B_KEMPTY = B_KFULL + NKS;     // NKS
  static constexpr int B_VFULL = B_KEMPTY + NKS;     // NVS
  static constexpr int B_VEMPTY = B_VFULL + NVS;     // NVS
  static constexpr int B_SFULL = B_VEMPTY + NVS;     // 2 (S buffer)
  static constexpr int B_DPFULL = B_SFULL + 2;
  static constexpr int B_DSREADY = B_DPFULL + 1;     // 2 (tile parity)
  static constexpr int B_DQDONE = B_DSREADY + 2;
  static constexpr int B_DRAIN = B_DQDONE + 1;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int NTHREADS = 320;
  static constexpr int TMEM_COLS = 512;
  static constexpr int T_S = 0;        // 2 x 128
  static constexpr int T_DP = 256;     // 128
  static constexpr int T_DQ = 384;     // DP
  static_assert(T_DQ + DP <= TMEM_COLS, "TMEM column budget");
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
    accel_dq_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const float *__restrict__ LSE,
                    const float *__restrict__ Dvec, void *__restrict__ dQ, int out16, int BH, int L,
                    int Lk_rows, int D, int causal, int off0, float scale, float scale_log2,
                    const int *__restrict__ kv_len, int H, int br, unsigned int *err,
                    unsigned long long timeout_ns, int hilo) {
  using C = DqCfg<DP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Heaviest causal query blocks (largest qb) of every head go first.
  const int nqb = (L + C::BM - 1) / C::BM;
  const int qb = nqb - 1 - static_cast<int>(blockIdx.x / BH);
  const int bh = static_cast<int>(blockIdx.x % BH);
  const int q0 = qb * C::BM;
  // Lk key rows (all Lk_rows rows, or the batch element's padded length);
  // causal: query i sees key j iff j <= i + off
  const MgKeys keys = mg_keys(kv_len, bh, H, L, Lk_rows, off0, br);
  const int Lk = keys.len, off = keys.off;
  const int nkt_all = (Lk + C::BN - 1) / C::BN;
  const int last = min(q0 + C::BM, L) - 1 + off;  // last key any row of the block sees
  const int n = !causal ? nkt_all : (last < 0 ? 0 : min(nkt_all, last / C::BN + 1));

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 256) {
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == C::B_DSREADY || i == C::B_DSREADY + 1) cnt = 8;
      mbar_init(bar(i), cnt);
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmdO);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab = make_abort(abort_flag, err, timeout_ns);

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      mbar_arrive_expect_tx(bar(C::B_QFULL), 2 * C::Q_TILE);
      for (int c = 0; c < C::NCHUNK; ++c) {
        tma_load_3d(sbase + C::OFF_Q + c * C::BOX_Q, &tmQ, c * 64, q0, bh, bar(C::B_QFULL));
        tma_load_3d(sbase + C::OFF_DO + c * C::BOX_Q, &tmdO, c * 64, q0, bh, bar(C::B_QFULL));
      }
      int issued_v = 0;
      for (int j = 0; j < n; ++j) {
        const int sk = j % C::NKS, sv = j % C::NVS;
        if (j >= C::NKS && !mbar_wait(bar(C::B_KEMPTY + sk), ((j / C::NKS) - 1) & 1, ab)) break;
        mbar_arrive_expect_tx(bar(C::B_KFULL + sk), C::KV_TILE);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(sbase + C::OFF_K + sk * C::KV_TILE + c * C::BOX_KV, &tmK, c * 64,
                      j * C::BN, bh, bar(C::B_KFULL + sk));
        issued = j + 1;
        if (j >= C::NVS && !mbar_wait(bar(C::B_VEMPTY + sv), ((j / C::NVS) - 1) & 1, ab)) break;
        mbar_arrive_expect_tx(bar(C::B_VFULL + sv), C::KV_TILE);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(sbase + C::OFF_V + sv * C::KV_TILE + c * C::BOX_KV, &tmV, c * 64,
                      j * C::BN, bh, bar(C::B_VFULL + sv));
        issued_v = j + 1;
      }
      drain_wait(bar(C::B_QFULL), 0, 2000000000ull);
      for (int j = max(0, issued - C::NKS); j < issued; ++j)
        drain_wait(bar(C::B_KFULL + j % C::NKS), (j / C::NKS) & 1, 2000000000ull);
      for (int j = max(0, issued_v - C::NVS); j < issued_v; ++j)
        drain_wait(bar(C::B_VFULL + j % C::NVS), (j / C::NVS) & 1, 2000000000ull);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idSD = idesc_16_f32(128, C::BN, false, false, F16);
      constexpr uint32_t idQ = idesc_16_f32(128, DP, false, true, F16);
      // base descriptors; each MMA adds a compile-time byte offset
      const uint32_t sb = opaque_u32(sbase);
      const uint64_t dQ0 = sdesc_sw128(sb + C::OFF_Q, 0, 1024);
      const uint64_t dO0 = sdesc_sw128(sb + C::OFF_DO, 0, 1024);
      const uint64_t dK0 = sdesc_sw128(sb + C::OFF_K, 0, 1024);
      const uint64_t dV0 = sdesc_sw128(sb + C::OFF_V, 0, 1024);
      const uint64_t dKmn = sdesc_sw128(sb + C::OFF_K, C::BOX_KV, 1024);
      bool ok = mbar_wait(bar(C::B_QFULL), 0, ab);
      // X = A_res B_j^T with A_res in {Q, dO} resident and B_j in {K_j, V_j}; K-major.
      auto issue_T = [&](uint64_t dA_, uint64_t dB_, uint32_t d) {
        // opaque copies: the per-step descriptors are formed here, not hoisted
        const uint64_t dA = opaque_u64(dA_), dB = opaque_u64(dB_);
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk) {
          const uint32_t oa = (kk >> 2) * C::BOX_Q + (kk & 3) * 32;
          const uint32_t ob = (kk >> 2) * C::BOX_KV + (kk & 3) * 32;
          mma_ss(d, sdesc_add(dA, oa), sdesc_add(dB, ob), idSD, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_S = [&](int j) -> bool {
        const int s = j % C::NKS;
        if (!mbar_wait(bar(C::B_KFULL + s), (j / C::NKS) & 1, ab)) return false;
        issue_T(dQ0, sdesc_add(dK0, s * C::KV_TILE), tmem + C::T_S + (j & 1) * 128);
        mma_commit(bar(C::B_SFULL + (j & 1)));
        return true;
      };
      auto issue_dP = [&](int j) -> bool {
        const int s = j % C::NVS;
        if (!mbar_wait(bar(C::B_VFULL + s), (j / C::NVS) & 1, ab)) return false;
        issue_T(dO0, sdesc_add(dV0, s * C::KV_TILE), tmem + C::T_DP);
        mma_commit(bar(C::B_DPFULL));
        mma_commit(bar(C::B_VEMPTY + s));  // V_j is free once dP(j) completes
        return true;
      };
      if (ok && n > 0) ok = issue_S(0);
      if (ok && n > 0) ok = issue_dP(0);
      if (ok && n > 1) ok = issue_S(1);
      for (int j = 0; ok && j < n; ++j) {
        const int s = j % C::NKS;
        if (!(ok = mbar_wait(bar(C::B_DSREADY + (j & 1)), (j >> 1) & 1, ab))) break;
        tc_fence_after();
        // dQ += dS K_j: A = dS (bf16 packed in the S buffer; warpgroup g holds keys
        // 64g .. 64g+63 in columns 64g .. 64g+31), B = K_j MN-major.
        const uint64_t dk = opaque_u64(sdesc_add(dKmn, s * C::KV_TILE));
        const uint32_t aS = tmem + C::T_S + (j & 1) * 128, acc0 = j > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          const uint32_t acol = (kk >> 2) * 64 + (kk & 3) * 8;
          mma_ts(tmem + C::T_DQ, aS + acol, sdesc_add(dk, kk * 2048), idQ, kk > 0 ? 1u : acc0);
        }
        // hi/lo policy: dQ also accumulates dS's lo part (columns 64g+32 .. 64g+63)
        if (hilo) {
#pragma unroll
          for (int kk = 0; kk < C::BN / 16; ++kk) {
            const uint32_t acol = (kk >> 2) * 64 + 32 + (kk & 3) * 8;
            mma_ts(tmem + C::T_DQ, aS + acol, sdesc_add(dk, kk * 2048), idQ, 1u);
          }
        }
        mma_commit(bar(C::B_KEMPTY + s));
        if (j + 1 < n && !(ok = issue_dP(j + 1))) break;
        if (j + 2 < n && !(ok = issue_S(j + 2))) break;
      }
      mma_commit(bar(C::B_DQDONE));
      mma_commit(bar(C::B_DRAIN));
      drain_wait(bar(C::B_DRAIN), 0, 2000000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int g = warp >> 2;                 // key columns 64g .. 64g+63 of each tile
    const int rl = 32 * (warp & 3) + lane;   // query row within the block = TMEM lane
    const int qrow = q0 + rl;
    const bool vrow = qrow < L;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const float lse2 = vrow ? LSE[static_cast<size_t>(bh) * L + qrow] * kLog2e : INFINITY;
    const float dvr = vrow ? Dvec[static_cast<size_t>(bh) * L + qrow] : 0.f;
    // last allowed key of this row (negative: none, the row's softmax is empty and
    // every P is masked to 0 after the exponential)
    const int lim = causal ? min(Lk - 1, qrow + off) : (Lk - 1);
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int k0 = j * C::BN + 64 * g;
      if (!(ok = mbar_wait_warp(bar(C::B_SFULL + (j & 1)), (j >> 1) & 1, ab))) break;
      tc_fence_after();
      const bool need_mask = k0 + 63 > lim || !vrow;
      const uint32_t tS = tmem + lane_off + C::T_S + (j & 1) * 128 + 64 * g;
      float p[64];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        tmem_ld32(tS + 32 * c, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float x = ex2(fmaf(__uint_as_float(r[e]), scale_log2, -lse2));
          if (need_mask && k0 + 32 * c + e > lim) x = 0.f;
          p[32 * c + e] = x;
        }
      }
      if (!(ok = mbar_wait_warp(bar(C::B_DPFULL), j & 1, ab))) break;
      tc_fence_after();
      const uint32_t tDP = tmem + lane_off + C::T_DP + 64 * g;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        tmem_ld32(tDP + 32 * c, r);
        tmem_wait_ld();
        uint32_t pk[16], pl[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float d0 = p[32 * c + 2 * e] * (__uint_as_float(r[2 * e]) - dvr);
          const float d1 = p[32 * c + 2 * e + 1] * (__uint_as_float(r[2 * e + 1]) - dvr);
          if (hilo)
            pack16_hilo<F16>(d0, d1, pk[e], pl[e]);
          else
            pk[e] = pack16<F16>(d0, d1);
        }
        // dS over the S columns this warpgroup has already read (its lo part, under
        // the hi/lo policy, 32 columns further on)
        tmem_st16(tS + 16 * c, pk);
        if (hilo) tmem_st16(tS + 32 + 16 * c, pl);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_DSREADY + (j & 1)));
    }
    if (ok && n > 0) ok = mbar_wait_warp(bar(C::B_DQDONE), 0, ab);
    if (ok && n == 0 && vrow) {
      // no key tile for this query block: dQ = 0 (warpgroup g writes its half)
      const size_t row = (static_cast<size_t>(bh) * L + qrow) * D;
      for (int c = 0; c < DP / 2 && g * (DP / 2) + c < D; c += 4)
        store4<F16>(dQ, out16, row + g * (DP / 2) + c, 0.f, 0.f, 0.f, 0.f);
    }
    if (ok && n > 0) {
      tc_fence_after();
      const size_t row = (static_cast<size_t>(bh) * L + (vrow ? qrow : 0)) * D;
#pragma unroll
      for (int c = 0; c < DP / 64; ++c) {
        const int col = g * (DP / 2) + 32 * c;
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + C::T_DQ + col, r);
        tmem_wait_ld();
        if (vrow && col < D) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            store4<F16>(dQ, out16, row + col + e, __uint_as_float(r[e]) * scale,
                        __uint_as_float(r[e + 1]) * scale, __uint_as_float(r[e + 2]) * scale,
                        __uint_as_float(r[e + 3]) * scale);
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
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
                   const float *Dvec, void *dQ, const MgProblem &p, unsigned int *err,
                   cudaStream_t st) {
  using C = DqCfg<DP>;
  const int BH = p.B * p.H;
  CUtensorMap tq, tdo, tk, tv;
  cudaError_t e;
  if ((e = mg_tmap_16(&tq, Q, p.D, p.L, BH, C::BM, F16)) != cudaSuccess) return e;
  if ((e = mg_tmap_16(&tdo, dO, p.D, p.L, BH, C::BM, F16)) != cudaSuccess) return e;
  if ((e = mg_tmap_16(&tk, K, p.D, p.Lk, BH, C::BN, F16)) != cudaSuccess) return e;
  if ((e = mg_tmap_16(&tv, V, p.D, p.Lk, BH, C::BN, F16)) != cudaSuccess) return e;
  auto kern = accel_dq_kernel<DP, F16>;
  if ((e = mg_set_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM_BYTES,
                            (DP == 64 ? 10 : 11) + (F16 ? 12 : 0))) != cudaSuccess)
    return e;
  const int nqb = (p.L + C::BM - 1) / C::BM;
  const long long grid = static_cast<long long>(nqb) * BH;
  kern<<<static_cast<unsigned>(grid), C::NTHREADS, C::SMEM_BYTES, st>>>(
      tq, tdo, tk, tv, LSE, Dvec, dQ, p.out16, BH, p.L, p.Lk, p.D, p.causal, p.off, p.scale,
      p.scale * kLog2e, p.kv_len, p.H, p.br, err, mg_wait_limit_ns(), p.hilo);
  return cudaGetLastError();
}

}  // namespace

cudaError_t mg_launch_accel_dq(const void *Q, const void *K, const void *V, const void *dO,
                               const float *LSE, const float *Dvec, void *dQ, const MgProblem &p,
                               unsigned int *err, cudaStream_t st) {
  if (p.f16) {
    if (p.D <= 64) return launch<64, true>(Q, K, V, dO, LSE, Dvec, dQ, p, err, st);
    return launch<128, true>(Q, K, V, dO, LSE, Dvec, dQ, p, err, st);
  }
  if (p.D <= 64) return launch<64, false>(Q, K, V, dO, LSE, Dvec, dQ, p, err, st);
  return launch<128, false>(Q, K, V, dO, LSE, Dvec, dQ, p, err, st);
}
