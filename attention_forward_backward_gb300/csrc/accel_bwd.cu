// accel_bwd.cu -- ACCEL_BF16 attention backward on tcgen05 tensor cores: one
// fused kernel per 128-key block that accumulates dK and dV in tensor memory
// and adds its dQ contribution into global f32 dQ with TMA bulk reductions.
//
// "Meganeura: Portable GPU Training and Inference through Vulkan and Metal"
// splits the attention derivative into a dQ kernel and a fused dK+dV kernel
// (Section 3.3; Section 8 makes fused dK+dV an invariant) and profiles the pair
// as the dominant backward cost (Section 7.3). Derivative operands keep f32
// accumulation (Sections 3.1 and 4.2); P and dS are rounded to bf16 only where
// they enter an MMA, exactly like the forward's P.
//
// Per CTA: keys k0 .. k0+127 of one (b, h) head (TMEM lanes = keys). K and V
// are loaded once; the query axis is walked in blocks of BQ rows (64 for
// D = 128, 128 for D = 64), Q and dO by TMA through a 2-stage ring.
// Per query block i:
//   S^T  = K Q_i^T            (TMEM, f32)     dP^T = V dO_i^T   (TMEM, f32)
//   P^T  = exp2(S^T scale log2e - LSE_i log2e), masked        (softmax warps)
//   dV  += P^T dO_i           (A = P^T from TMEM, bf16)
//   dS^T = P^T (dP^T - Dvec_i)                                (softmax warps)
//   dK  += dS^T Q_i           (A = dS^T from TMEM, bf16)
//   dQ_i = dS K               (dS^T also staged in smem; for D = 128 the MMA
//                              computes dQ_i^T = K^T dS^T so that M = 128)
// dQ_i leaves TMEM through a swizzled f32 staging tile and a TMA tensor
// add-reduction into dQ (zeroed by the host call beforehand); bulk reductions
// sustain far more L2 throughput than per-element f32 reductions would.
// MMA issue order per block: dV(i), S(i+1), dP(i+1), dK(i), dQ(i), so that the
// tensor core computes the next block's scores while the softmax warps turn
// dP(i) into dS(i), and dK/dQ run while they turn S(i+1) into P(i+1). dP^T is
// double-buffered in TMEM for D = 128 (for D = 64 it goes after dQ(i)); Q and
// dO stream through a 3-stage ring so that a tile's load has two blocks of
// lead time.
// Warp roles: 0-3 dQ epilogue, 4 TMA producer (plus LSE/Dvec staging), 5 MMA
// issuer, 8-15 two softmax warpgroups splitting the query columns.
// Every wait is bounded; on a give-up the CTA sets the device error word and
// leaves through the normal teardown (own copies and MMAs drained first).
#include <climits>

#include "internal.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace {

using namespace mg_tc;

template <int DP>
struct BwdCfg {
  static constexpr int BN = 128;                    // keys per CTA
  static constexpr int BQ = DP == 128 ? 64 : 128;   // queries per block
  static constexpr int QPW = BQ / 2;                // query columns per softmax warpgroup
  static constexpr int ND = DP == 128 ? 2 : 1;      // dP^T buffers in TMEM
  static constexpr int NCHUNK = DP / 64;
  static constexpr int KV_TILE = BN * DP * 2;
  static constexpr int BOX_KV = BN * 128;
  static constexpr int Q_TILE = BQ * DP * 2;
  static constexpr int BOX_Q = BQ * 128;
  static constexpr int DS_CHUNK = BN * 128;         // [128 keys][64 q] bf16
  static constexpr int NQC = BQ / 64;               // dS^T chunks
  static constexpr int DS_BUF = NQC * DS_CHUNK;
  static constexpr int NQS = 3;                     // Q/dO ring stages
  static constexpr int NDS = DP == 128 ? 2 : 1;     // dS^T smem buffers
  static constexpr int DQ_BOX = BQ * 128;           // [BQ][32] f32
  static constexpr int DQ_STAGE = (DP / 32) * DQ_BOX;
  // shared memory
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_TILE;
  static constexpr int OFF_Q = OFF_V + KV_TILE;             // NQS stages
  static constexpr int OFF_DO = OFF_Q + NQS * Q_TILE;       // NQS stages
  static constexpr int OFF_DS = OFF_DO + NQS * Q_TILE;      // NDS dS^T tiles
  static constexpr int OFF_DQ = OFF_DS + NDS * DS_BUF;      // dQ staging
  static constexpr int OFF_LSE = OFF_DQ + DQ_STAGE;          // NQS stages x BQ f32
  static constexpr int OFF_DV = OFF_LSE + NQS * BQ * 4;        // NQS stages x BQ f32
  static constexpr int OFF_BAR = OFF_DV + NQS * BQ * 4;
  static constexpr int B_KVFULL = 0;
  static constexpr int B_QFULL = 1;                  // NQS (Q/dO stage)
  static constexpr int B_QEMPTY = B_QFULL + 4;       // NQS
  static constexpr int B_SFULL = B_QEMPTY + 4;
  static constexpr int B_PREADY = B_SFULL + 1;
  static constexpr int B_DPFULL = B_PREADY + 1;      // 2 (dP buffer)
  static constexpr int B_DSREADY = B_DPFULL + 2;     // 2 (block parity)
  static constexpr int B_DSMFREE = B_DSREADY + 2;    // 2 (dS smem buffer)
  static constexpr int B_DQFULL = B_DSMFREE + 2;
  static constexpr int B_DQEMPTY = B_DQFULL + 1;
  static constexpr int B_ACCDONE = B_DQEMPTY + 1;
  static constexpr int B_DRAIN = B_ACCDONE + 1;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int NTHREADS = 512;
  static constexpr int TMEM_COLS = 512;
  static constexpr int T_DV = 0;
  static constexpr int T_DK = DP;
  static constexpr int T_S = 2 * DP;                  // BQ
  static constexpr int T_DP = T_S + BQ;               // ND x BQ
  static constexpr int T_DQ = T_DP + ND * BQ;         // 64
  static_assert(T_DQ + 64 <= TMEM_COLS, "TMEM column budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return false;
  }
  return true;
}

__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Byte offset of f32 element (row, col) in a [rows][32]-box, 128-byte swizzled
// staging tile (boxes of 32 columns stacked along col / 32).
__device__ __forceinline__ uint32_t dq_stage_off(int row, int col, int box_bytes) {
  const int box = col >> 5, unit = (col & 31) >> 2;
  return static_cast<uint32_t>(box * box_bytes + row * 128 + ((unit ^ (row & 7)) << 4) +
                               ((col & 3) << 2));
}

template <int DP>
__global__ void __launch_bounds__(512, 1)
    accel_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmdO,
                      const __grid_constant__ CUtensorMap tmdQ, const float *__restrict__ LSE,
                      const float *__restrict__ Dvec, float *__restrict__ dQ,
                      float *__restrict__ dK,
                      float *__restrict__ dV, int BH, int L, int Lk, int D, int causal, int off,
                      float scale,
                      float scale_log2, unsigned int *err, unsigned long long timeout_ns) {
  using C = BwdCfg<DP>;
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
  // L query rows, Lk key rows; causal: query i sees key j iff j <= i + off
  const int nkb = (Lk + C::BN - 1) / C::BN;
  const int bh = static_cast<int>(blockIdx.x / nkb);
  const int kb = static_cast<int>(blockIdx.x % nkb);
  const int k0 = kb * C::BN;
  const int nqb = (L + C::BQ - 1) / C::BQ;
  const int qb0 = causal ? max(0, k0 - off) / C::BQ : 0;  // first block with a query seeing k0
  const int n = max(0, nqb - qb0);

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 128) {
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i >= C::B_QEMPTY && i < C::B_QEMPTY + 4) cnt = 1 + 8;
      if (i == C::B_PREADY || i == C::B_DSREADY || i == C::B_DSREADY + 1) cnt = 8;
      if (i == C::B_DQEMPTY) cnt = 4;
      mbar_init(bar(i), cnt);
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
    tma_prefetch_desc(&tmdQ);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab = make_abort(abort_flag, err, timeout_ns);

  if (warp == 4) {
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
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idSP = idesc_bf16_f32(128, C::BQ, false, false);
      constexpr uint32_t idKV = idesc_bf16_f32(128, DP, false, true);
      constexpr uint32_t idDQ =
          DP == 128 ? idesc_bf16_f32(128, C::BQ, true, true) : idesc_bf16_f32(128, DP, true, true);
      bool ok = mbar_wait(bar(C::B_KVFULL), 0, ab);
      // base descriptors; each MMA adds a compile-time byte offset
      const uint32_t sb = opaque_u32(sbase);
      const uint64_t dK0 = sdesc_sw128(sb + C::OFF_K, 0, 1024);
      const uint64_t dV0 = sdesc_sw128(sb + C::OFF_V, 0, 1024);
      const uint64_t dQ0 = sdesc_sw128(sb + C::OFF_Q, 0, 1024);
      const uint64_t dO0 = sdesc_sw128(sb + C::OFF_DO, 0, 1024);
      const uint64_t dQmn = sdesc_sw128(sb + C::OFF_Q, C::BOX_Q, 1024);
      const uint64_t dOmn = sdesc_sw128(sb + C::OFF_DO, C::BOX_Q, 1024);
      const uint64_t dKmn = sdesc_sw128(sb + C::OFF_K, C::BOX_KV, 1024);
      const uint64_t dDSmn = sdesc_sw128(sb + C::OFF_DS, C::DS_CHUNK, 1024);
      int qwaited = -1;
      auto wait_q = [&](int i) -> bool {
        if (qwaited >= i) return true;
        qwaited = i;
        return mbar_wait(bar(C::B_QFULL + i % C::NQS), (i / C::NQS) & 1, ab);
      };
      // X^T = A_tile * B_i^T with A in {K, V}, B_i in {Q_i, dO_i}; both K-major.
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
      auto issue_S = [&](int i) -> bool {
        if (!wait_q(i)) return false;
        tc_fence_after();
        issue_T(dK0, sdesc_add(dQ0, (i % C::NQS) * C::Q_TILE), tmem + C::T_S);
        mma_commit(bar(C::B_SFULL));
        return true;
      };
      auto issue_dP = [&](int i) -> bool {
        if (!wait_q(i)) return false;
        tc_fence_after();
        const int db = C::ND == 2 ? (i & 1) : 0;
        issue_T(dV0, sdesc_add(dO0, (i % C::NQS) * C::Q_TILE), tmem + C::T_DP + db * C::BQ);
        mma_commit(bar(C::B_DPFULL + db));
        return true;
      };
      // acc (+)= X^T(tmem, bf16) * Y_i (MN-major smem), K = BQ queries.
      auto issue_acc = [&](uint32_t tA, uint64_t dY_, uint32_t d, bool first) {
        const uint64_t dY = opaque_u64(dY_);
        const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk) {
          const int qq = 16 * kk;
          const uint32_t acol = (qq / C::QPW) * C::QPW + (qq % C::QPW) / 2;
          mma_ts(d, tA + acol, sdesc_add(dY, kk * 2048), idKV, kk > 0 ? 1u : acc0);
        }
      };
      if (ok && n > 0) ok = issue_S(0);
      if (ok && n > 0) ok = issue_dP(0);
      for (int i = 0; ok && i < n; ++i) {
        const int st = i % C::NQS;
        const int db = C::ND == 2 ? (i & 1) : 0;
        if (!(ok = mbar_wait(bar(C::B_PREADY), i & 1, ab))) break;
        tc_fence_after();
        issue_acc(tmem + C::T_S, sdesc_add(dOmn, st * C::Q_TILE), tmem + C::T_DV, i == 0);
        if (i + 1 < n && !(ok = issue_S(i + 1))) break;
        if (C::ND == 2 && i + 1 < n && !(ok = issue_dP(i + 1))) break;
        if (!(ok = mbar_wait(bar(C::B_DSREADY + (i & 1)), (i >> 1) & 1, ab))) break;
        tc_fence_after();
        issue_acc(tmem + C::T_DP + db * C::BQ, sdesc_add(dQmn, st * C::Q_TILE), tmem + C::T_DK,
                  i == 0);
        mma_commit(bar(C::B_QEMPTY + st));
        if (i > 0 && !(ok = mbar_wait(bar(C::B_DQEMPTY), (i - 1) & 1, ab))) break;
        tc_fence_after();
        const uint64_t dDSi = opaque_u64(sdesc_add(dDSmn, (i % C::NDS) * C::DS_BUF));
        const uint64_t dKq = opaque_u64(dKmn);
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          if (DP == 128) {
            // dQ^T [d][q] = K^T [d][key] * dS^T [key][q]
            mma_ss(tmem + C::T_DQ, sdesc_add(dKq, kk * 2048), sdesc_add(dDSi, kk * 2048), idDQ,
                   kk > 0 ? 1u : 0u);
          } else {
            // dQ [q][d] = dS [q][key] * K [key][d]
            mma_ss(tmem + C::T_DQ, sdesc_add(dDSi, kk * 2048), sdesc_add(dKq, kk * 2048), idDQ,
                   kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(bar(C::B_DQFULL));
        mma_commit(bar(C::B_DSMFREE + i % C::NDS));
        if (C::ND == 1 && i + 1 < n && !(ok = issue_dP(i + 1))) break;
      }
      mma_commit(bar(C::B_ACCDONE));
      mma_commit(bar(C::B_DRAIN));
      drain_wait(bar(C::B_DRAIN), 0, 2000000000ull);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ dQ epilogue
    const int t = threadIdx.x;  // TMEM lane: d (D = 128) or query row (D = 64)
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
    const uint32_t stage = sbase + C::OFF_DQ;
    for (int i = 0; i < n; ++i) {
      if (!mbar_wait_warp(bar(C::B_DQFULL), i & 1, ab)) break;
      tc_fence_after();
      uint32_t r[64];
      {
        uint32_t a[32], b2[32];
        tmem_ld32(tmem + lane_off + C::T_DQ, a);
        tmem_ld32(tmem + lane_off + C::T_DQ + 32, b2);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          r[e] = a[e];
          r[32 + e] = b2[e];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_DQEMPTY));
      // The previous reduction must have finished reading the staging tile.
      if (t == 0) bulk_wait_group_read0();
      __syncwarp();  // bar.sync is aligned: the whole warp arrives together
      named_bar_sync(1, 128);
      if (DP == 128) {
        // thread = d; r[q] = dQ^T[d][q]
#pragma unroll
        for (int q = 0; q < 64; ++q)
          st_shared_f32(stage + dq_stage_off(q, t, C::DQ_BOX), __uint_as_float(r[q]) * scale);
      } else {
        // thread = query row; r[d] = dQ[q][d]
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const uint32_t off = dq_stage_off(t, 4 * u, C::DQ_BOX);
          st_shared_v4(stage + off, __float_as_uint(__uint_as_float(r[4 * u]) * scale),
                       __float_as_uint(__uint_as_float(r[4 * u + 1]) * scale),
                       __float_as_uint(__uint_as_float(r[4 * u + 2]) * scale),
                       __float_as_uint(__uint_as_float(r[4 * u + 3]) * scale));
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (t == 0) {
        const int q0 = (qb0 + i) * C::BQ;
        for (int bx = 0; bx < (D + 31) / 32; ++bx)
          tma_reduce_add_3d(&tmdQ, stage + bx * C::DQ_BOX, bx * 32, q0, bh);
        bulk_commit_group();
      }
    }
    if (t == 0) bulk_wait_group0();
  } else if (warp >= 8) {
    // ------------------------------------------------------------ softmax warpgroups
    const int g = (warp - 8) >> 2;
    const int quarter = warp & 3;
    const int kr = 32 * quarter + lane;  // key row within the block = TMEM lane
    const int kg = k0 + kr;
    const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
    const uint32_t sDS = sbase + C::OFF_DS;
    // smallest query index that may see this thread's key (past Lk: none may)
    const int qmin = kg >= Lk ? INT_MAX : (causal ? kg - off : INT_MIN);
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      const int st = i % C::NQS;
      const int db = C::ND == 2 ? (i & 1) : 0;
      const int q0 = (qb0 + i) * C::BQ;
      if (!(ok = mbar_wait_warp(bar(C::B_QFULL + st), (i / C::NQS) & 1, ab))) break;
      if (!(ok = mbar_wait_warp(bar(C::B_SFULL), i & 1, ab))) break;
      tc_fence_after();
      // query column e of this warpgroup's slice is masked iff e < lim0 (e is q - q0 - g QPW)
      const int lim0 = qmin == INT_MIN ? INT_MIN
                                       : (qmin == INT_MAX ? INT_MAX : qmin - (q0 + g * C::QPW));
      const bool need_mask = lim0 > 0;
      const float *lse = sLse + st * C::BQ + g * C::QPW;
      const float *dvq = sDv + st * C::BQ + g * C::QPW;
      const uint32_t tS = tmem + lane_off + C::T_S + g * C::QPW;
      const uint32_t tDP = tmem + lane_off + C::T_DP + db * C::BQ + g * C::QPW;
      float p[C::QPW];
#pragma unroll
      for (int c = 0; c < C::QPW / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tS + 32 * c, r);
        tmem_wait_ld();
        float lv[32];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 v4 = *reinterpret_cast<const float4 *>(lse + 32 * c + e);
          lv[e] = v4.x; lv[e + 1] = v4.y; lv[e + 2] = v4.z; lv[e + 3] = v4.w;
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float x = ex2(fmaf(__uint_as_float(r[e]), scale_log2, -lv[e]));
          if (need_mask && 32 * c + e < lim0) x = 0.f;
          p[32 * c + e] = x;
        }
      }
#pragma unroll
      for (int c = 0; c < C::QPW / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack_bf16(p[32 * c + 2 * e], p[32 * c + 2 * e + 1]);
        tmem_st16(tS + 16 * c, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_PREADY));

      if (!(ok = mbar_wait_warp(bar(C::B_DPFULL + db), (C::ND == 2 ? (i >> 1) : i) & 1, ab)))
        break;
      // this dS staging tile is free once dQ(i - NDS) has completed
      if (i >= C::NDS &&
          !(ok = mbar_wait_warp(bar(C::B_DSMFREE + i % C::NDS), ((i / C::NDS) - 1) & 1, ab)))
        break;
      tc_fence_after();
      const uint32_t sDSi = sDS + (i % C::NDS) * C::DS_BUF;
#pragma unroll
      for (int c = 0; c < C::QPW / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tDP + 32 * c, r);
        tmem_wait_ld();
        float dv[32];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 v4 = *reinterpret_cast<const float4 *>(dvq + 32 * c + e);
          dv[e] = v4.x; dv[e + 1] = v4.y; dv[e + 2] = v4.z; dv[e + 3] = v4.w;
        }
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float d0 = p[32 * c + 2 * e] * (__uint_as_float(r[2 * e]) - dv[2 * e]);
          const float d1 = p[32 * c + 2 * e + 1] * (__uint_as_float(r[2 * e + 1]) - dv[2 * e + 1]);
          pk[e] = pack_bf16(d0, d1);
        }
        tmem_st16(tDP + 16 * c, pk);
        // dS^T row kr, queries ql .. ql+31 into the swizzled smem tile
        const int ql = g * C::QPW + 32 * c;
        const uint32_t chunk = sDSi + (ql >> 6) * C::DS_CHUNK + kr * 128;
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          const int unit = ((ql & 63) >> 3) + u4;
          st_shared_v4(chunk + ((unit ^ (kr & 7)) << 4), pk[4 * u4], pk[4 * u4 + 1],
                       pk[4 * u4 + 2], pk[4 * u4 + 3]);
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(C::B_DSREADY + (i & 1)));
        mbar_arrive(bar(C::B_QEMPTY + st));
      }
    }
    // dK (scaled) and dV of this key block
    if (ok && n > 0) ok = mbar_wait_warp(bar(C::B_ACCDONE), 0, ab);
    if (ok && n == 0 && kg < Lk) {
      // no query sees this key block: dK = dV = 0 (warpgroup w writes its half)
      const size_t row = (static_cast<size_t>(bh) * Lk + kg) * D;
      for (int c = 0; c < DP / 2 && g * (DP / 2) + c < D; c += 4) {
        *reinterpret_cast<float4 *>(dV + row + g * (DP / 2) + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(dK + row + g * (DP / 2) + c) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (ok && n > 0) {
      tc_fence_after();
      const bool valid = kg < Lk;
      const size_t row = (static_cast<size_t>(bh) * Lk + (valid ? kg : 0)) * D;
#pragma unroll
      for (int c = 0; c < DP / 64; ++c) {
        const int col = g * (DP / 2) + 32 * c;
        uint32_t rv[32], rk[32];
        tmem_ld32(tmem + lane_off + C::T_DV + col, rv);
        tmem_ld32(tmem + lane_off + C::T_DK + col, rk);
        tmem_wait_ld();
        if (valid && col < D) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            *reinterpret_cast<float4 *>(dV + row + col + e) =
                make_float4(__uint_as_float(rv[e]), __uint_as_float(rv[e + 1]),
                            __uint_as_float(rv[e + 2]), __uint_as_float(rv[e + 3]));
            *reinterpret_cast<float4 *>(dK + row + col + e) = make_float4(
                __uint_as_float(rk[e]) * scale, __uint_as_float(rk[e + 1]) * scale,
                __uint_as_float(rk[e + 2]) * scale, __uint_as_float(rk[e + 3]) * scale);
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

template <int DP>
cudaError_t launch(const __nv_bfloat16 *Q, const __nv_bfloat16 *K, const __nv_bfloat16 *V,
                   const __nv_bfloat16 *dO, const float *LSE, const float *Dvec, float *dQ,
                   float *dK, float *dV, const MgProblem &p, unsigned int *err,
                   cudaStream_t st) {
  using C = BwdCfg<DP>;
  const int BH = p.B * p.H;
  CUtensorMap tq, tk, tv, tdo, tdq;
  cudaError_t e;
  if ((e = mg_tmap_bf16(&tq, Q, p.D, p.L, BH, C::BQ)) != cudaSuccess) return e;
  if ((e = mg_tmap_bf16(&tdo, dO, p.D, p.L, BH, C::BQ)) != cudaSuccess) return e;
  if ((e = mg_tmap_bf16(&tk, K, p.D, p.Lk, BH, C::BN)) != cudaSuccess) return e;
  if ((e = mg_tmap_bf16(&tv, V, p.D, p.Lk, BH, C::BN)) != cudaSuccess) return e;
  if ((e = mg_tmap_f32(&tdq, dQ, p.D, p.L, BH, C::BQ)) != cudaSuccess) return e;
  auto kern = accel_dkdv_kernel<DP>;
  if ((e = mg_set_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM_BYTES,
                            DP == 64 ? 8 : 9)) != cudaSuccess)
    return e;
  const int nkb = (p.Lk + C::BN - 1) / C::BN;
  const long long grid = static_cast<long long>(nkb) * BH;
  kern<<<static_cast<unsigned>(grid), C::NTHREADS, C::SMEM_BYTES, st>>>(
      tq, tk, tv, tdo, tdq, LSE, Dvec, dQ, dK, dV, BH, p.L, p.Lk, p.D, p.causal, p.off, p.scale,
      p.scale * kLog2e, err, mg_wait_limit_ns());
  return cudaGetLastError();
}

}  // namespace

cudaError_t mg_launch_accel_dkdv(const __nv_bfloat16 *Q, const __nv_bfloat16 *K,
                                 const __nv_bfloat16 *V, const __nv_bfloat16 *dO,
                                 const float *LSE, const float *Dvec, float *dQ, float *dK,
                                 float *dV, const MgProblem &p, unsigned int *err,
                                 cudaStream_t st) {
  if (!dQ) return cudaErrorInvalidValue;  // dK/dV alone: mg_launch_accel_dkdv_pp
  if (p.D <= 64) return launch<64>(Q, K, V, dO, LSE, Dvec, dQ, dK, dV, p, err, st);
  return launch<128>(Q, K, V, dO, LSE, Dvec, dQ, dK, dV, p, err, st);
}
