// accel_bwd.cu -- ACCEL_BF16 attention backward on tcgen05 tensor cores: one
// fused kernel per 128-key block that accumulates dK and dV in tensor memory
// and adds its dQ contribution into global f32 dQ.
//
// "Meganeura: Portable GPU Training and Inference through Vulkan and Metal"
// splits the attention derivative into a dQ kernel and a fused dK+dV kernel
// (Section 3.3; Section 8 makes fused dK+dV an invariant) and profiles the pair
// as the dominant backward cost (Section 7.3). Derivative operands keep f32
// accumulation (Sections 3.1 and 4.2); P and dS are rounded to bf16 only where
// they enter an MMA, exactly like the forward's P.
//
// Per CTA: keys k0 .. k0+127 of one (b, h) head (TMEM lanes = keys). K and V
// are loaded once; the query axis is walked in blocks of 128 rows, Q and dO by
// TMA through two rings of NQS stages each. Per query block j:
//   S^T  = K Q_j^T            (TMEM, f32)     dP^T = V dO_j^T   (TMEM, f32)
//   P^T  = exp2(S^T scale log2e - LSE_j log2e), masked        (softmax warps)
//   dV  += P^T dO_j           (A = P^T from TMEM, bf16)
//   dS^T = P^T (dP^T - Dvec_j)                                (softmax warps)
//   dK  += dS^T Q_j           (A = dS^T: from TMEM at D = 64, from the
//                              shared-memory staging tile at D = 128; bf16)
//   dQ_j = dS K               (dS^T staged in shared memory)
// Every product is a 128 x 128 (D = 128) or 128 x 64 (D = 64) MMA group, so one
// issuing thread keeps up with the tensor core and each byte an operand moves
// through shared memory feeds twice the flops of 64-row query blocks.
//
// Tensor memory (512 columns) holds dV, dK, S^T and dP^T. At D = 128 that is
// all of it, so dQ_j^T = K^T dS_j^T is accumulated over the dP^T columns once
// the softmax has read dP_j from them, and dP_{j+1} waits until the dQ warps
// have read dQ_j^T out. Those warps stage it
// in dO_j's ring stage (dead once dP_j and dV_j, which precede dQ_j, are done),
// 64 query rows at a time, each warp one 32-column box of d, and add it into
// global dQ with TMA tensor add-reductions; the stage returns to the dO
// producer only after those reductions have read it. (Per-element red.global
// reductions from registers were measured about ten times slower to drain.)
// At D = 64 dQ_j = dS K has columns and a staging tile of its own.
//
// MMA issue order (steady state, block j):
//   D = 128: dQ(j), dK(j), dP(j+1), dV(j+1), S(j+2)
//   D = 64:  dK(j), dP(j+1), dQ(j), dV(j+1), S(j+2)
// The softmax turns S(j+1) into P(j+1) while the products of block j run, and
// dP(j+1) into dS(j+1) while dV(j+1) and S(j+2) run. S(j+2) overwrites P(j+1)
// only after dV(j+1) has read it (issue order). At D = 128 dK(j) reads dS^T(j)
// from the shared-memory staging tile (dQ's operand too), so dQ(j) goes first
// into dP^T's columns, dK(j) runs while the dQ warps read dQ(j) out, and dP(j+1)
// waits for that read-out; at D = 64 dK(j) reads dS^T(j) from dP^T's columns and
// dP(j+1) follows it at once, ahead of dQ(j), so that it is done before the
// softmax warps need it.
//
// Warp roles: 0-3 dQ read-out, 4 TMA producer of K, V, Q (plus LSE and Dvec
// staging), 5 MMA issuer, 6 TMA producer of dO, 8-15 two softmax warpgroups
// splitting the 128 query columns. Every wait is bounded; on a give-up the CTA
// sets the device error word and leaves through the normal teardown (own copies
// and MMAs drained first).
#include <climits>

#include "internal.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace {

using namespace mg_tc;

template <int DP>
struct BwdCfg {
  static constexpr int BN = 128;                   // keys per CTA (TMEM lanes)
  static constexpr int BQ = 128;                   // queries per block
  static constexpr int QPW = BQ / 2;               // query columns per softmax warpgroup
  static constexpr int NCHUNK = DP / 64;           // 64-column boxes per row
  static constexpr bool kDqInDp = DP == 128;       // dQ^T accumulated over dP^T's columns
  static constexpr int NQS = DP == 128 ? 2 : 3;    // Q and dO ring stages
  static constexpr int KV_TILE = BN * DP * 2;
  static constexpr int BOX_KV = BN * 128;
  static constexpr int Q_TILE = BQ * DP * 2;
  static constexpr int BOX_Q = BQ * 128;
  static constexpr int DS_CHUNK = BN * 128;        // [128 keys][64 q] bf16
  static constexpr int DS_BUF = (BQ / 64) * DS_CHUNK;
  // dQ staging: D = 64, its own [BQ][64] f32 tile in boxes of [BQ][32] (each
  // read-out warp reduces its 32-row slab); D = 128, half the query rows at a
  // time ([64][128] f32 = one dO stage, boxes of [64][32]) over dO_j's stage
  static constexpr int DQ_ROWS = kDqInDp ? 64 : BQ;
  static constexpr int DQ_BOX = DQ_ROWS * 128;
  static constexpr int DQ_STAGE = kDqInDp ? 0 : (DP / 32) * DQ_BOX;
  static constexpr int DQ_TMA_ROWS = kDqInDp ? 64 : 32;  // rows per reduction box
  // shared memory: 1024-aligned tiles first, then the small items
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_TILE;
  static constexpr int OFF_Q = OFF_V + KV_TILE;             // NQS stages
  static constexpr int OFF_DO = OFF_Q + NQS * Q_TILE;       // NQS stages
  static constexpr int OFF_DS = OFF_DO + NQS * Q_TILE;      // dS^T tile
  static constexpr int OFF_DQ = OFF_DS + DS_BUF;            // dQ staging (D = 64)
  static constexpr int OFF_LSE = OFF_DQ + DQ_STAGE;         // NQS x BQ f32
  static constexpr int OFF_DV = OFF_LSE + NQS * BQ * 4;     // NQS x BQ f32
  static constexpr int OFF_BAR = OFF_DV + NQS * BQ * 4;
  static constexpr int B_KVFULL = 0;
  static constexpr int B_QFULL = 1;                 // NQS (Q stage; also LSE, Dvec)
  static constexpr int B_QFREE = B_QFULL + 4;       // NQS
  static constexpr int B_DOFULL = B_QFREE + 4;      // NQS
  static constexpr int B_DOFREE = B_DOFULL + 4;     // NQS
  static constexpr int B_SFULL = B_DOFREE + 4;
  static constexpr int B_PREADY = B_SFULL + 1;
  static constexpr int B_DPFULL = B_PREADY + 1;
  static constexpr int B_DSREADY = B_DPFULL + 1;
  static constexpr int B_DSMFREE = B_DSREADY + 1;
  static constexpr int B_DQFULL = B_DSMFREE + 1;
  static constexpr int B_DQEMPTY = B_DQFULL + 1;
  static constexpr int B_ACCDONE = B_DQEMPTY + 1;
  static constexpr int B_DRAIN = B_ACCDONE + 1;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  // request up to 1 KB of slack to align the base; the kernel checks the slack
  static constexpr int SMEM_LIMIT = 227 * 1024;
  static constexpr int SMEM_BYTES =
      SMEM_USED + 1024 <= SMEM_LIMIT ? SMEM_USED + 1024 : SMEM_LIMIT;
  static constexpr int NTHREADS = 512;
  static constexpr int TMEM_COLS = 512;
  static constexpr int T_DV = 0;
  static constexpr int T_DK = DP;
  static constexpr int T_S = 2 * DP;                  // BQ columns
  static constexpr int T_DP = T_S + BQ;               // BQ columns
  static constexpr int T_DQ = kDqInDp ? T_DP : T_DP + BQ;
  static_assert(NQS <= 4, "barrier slots");
  static_assert(kDqInDp ? T_DP + BQ <= TMEM_COLS : T_DQ + DP <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_USED <= SMEM_LIMIT, "shared memory budget");
};

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return false;
  }
  return true;
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

// The kernel's bounded waits: at D = 128 the variant that polls the abort flag and
// the clock less often (measured 1.3% faster there, slower at D = 64).
template <int DP>
__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, const Abort &ab) {
  if constexpr (DP == 128) return mbar_wait_poll(bar, parity, ab);
  else return mbar_wait(bar, parity, ab);
}
template <int DP>
__device__ __forceinline__ bool bwait_warp(uint32_t bar, uint32_t parity, const Abort &ab) {
  return __all_sync(0xffffffffu, bwait<DP>(bar, parity, ab));
}

template <int DP, bool F16>
__global__ void __launch_bounds__(512, 1)
    accel_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmdO,
                      const __grid_constant__ CUtensorMap tmdQ, const float *__restrict__ LSE,
                      const float *__restrict__ Dvec, float *__restrict__ dQ,
                      void *__restrict__ dK, void *__restrict__ dV, int out16, int BH, int L,
                      int Lk_rows, int D, int causal, int off0, float scale, float scale_log2,
                      unsigned int *err, unsigned long long timeout_ns,
                      const int *__restrict__ kv_len, int H, int br) {
  using C = BwdCfg<DP>;
  extern __shared__ uint8_t smem_raw[];
  const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_raw);
  uint8_t *smem = reinterpret_cast<uint8_t *>((raw + 1023) & ~static_cast<uintptr_t>(1023));
  // The tiles need a 1024-byte aligned base (128-byte swizzle atoms). If the
  // alignment pad does not fit in the slack requested at launch, report and
  // leave before any barrier or TMEM allocation (uniform over the CTA).
  if (reinterpret_cast<uintptr_t>(smem) - raw + C::SMEM_USED > C::SMEM_BYTES) {
    if (threadIdx.x == 0) atomicOr(err, 1u);
    return;
  }
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
  if (threadIdx.x == 128) {
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i >= C::B_QFREE && i < C::B_QFREE + 4) cnt = 1 + 8;
      if (i == C::B_PREADY || i == C::B_DSREADY) cnt = 8;
      if (i == C::B_DQEMPTY) cnt = 4;
      // D = 128: a dO stage is released by the four dQ warps (it stages dQ)
      if (C::kDqInDp && i >= C::B_DOFREE && i < C::B_DOFREE + 4) cnt = 4;
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
    // ------------------------------------------------------------ producer: K, V, Q, LSE, Dvec
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::B_KVFULL), 2 * C::KV_TILE);
      for (int c = 0; c < C::NCHUNK; ++c) {
        tma_load_3d(sbase + C::OFF_K + c * C::BOX_KV, &tmK, c * 64, k0, bh, bar(C::B_KVFULL));
        tma_load_3d(sbase + C::OFF_V + c * C::BOX_KV, &tmV, c * 64, k0, bh, bar(C::B_KVFULL));
      }
    }
    int issued = 0;
    for (int j = 0; j < n; ++j) {
      const int st = j % C::NQS;
      const int q0 = (qb0 + j) * C::BQ;
      // LSE (pre-scaled to base 2; +inf past L so that P = 0 there) and Dvec,
      // loaded before the wait for the stage so that their latency overlaps it.
      float lse_r[C::BQ / 32], dv_r[C::BQ / 32];
#pragma unroll
      for (int u = 0; u < C::BQ / 32; ++u) {
        const int qg = q0 + 32 * u + lane;
        const bool v = qg < L;
        lse_r[u] = v ? LSE[static_cast<size_t>(bh) * L + qg] : -INFINITY;
        dv_r[u] = v ? Dvec[static_cast<size_t>(bh) * L + qg] : 0.f;
      }
      if (j >= C::NQS && !bwait_warp<DP>(bar(C::B_QFREE + st), ((j / C::NQS) - 1) & 1, ab))
        break;
#pragma unroll
      for (int u = 0; u < C::BQ / 32; ++u) {
        // staged negated (-LSE log2 e), -inf for a row with an empty softmax (LSE =
        // -inf): its P is 0
        sLse[st * C::BQ + 32 * u + lane] = lse_r[u] == -INFINITY ? -INFINITY : -lse_r[u] * kLog2e;
        sDv[st * C::BQ + 32 * u + lane] = dv_r[u];
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::B_QFULL + st), C::Q_TILE);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(sbase + C::OFF_Q + st * C::Q_TILE + c * C::BOX_Q, &tmQ, c * 64, q0, bh,
                      bar(C::B_QFULL + st));
      }
      issued = j + 1;
    }
    if (lane == 0) {
      drain_wait(bar(C::B_KVFULL), 0, 2000000000ull);
      for (int j = max(0, issued - C::NQS); j < issued; ++j)
        drain_wait(bar(C::B_QFULL + j % C::NQS), (j / C::NQS) & 1, 2000000000ull);
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ producer: dO
    if (lane == 0) {
      int issued = 0;
      for (int j = 0; j < n; ++j) {
        const int st = j % C::NQS;
        if (j >= C::NQS && !bwait<DP>(bar(C::B_DOFREE + st), ((j / C::NQS) - 1) & 1, ab)) break;
        const int q0 = (qb0 + j) * C::BQ;
        mbar_arrive_expect_tx(bar(C::B_DOFULL + st), C::Q_TILE);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(sbase + C::OFF_DO + st * C::Q_TILE + c * C::BOX_Q, &tmdO, c * 64, q0, bh,
                      bar(C::B_DOFULL + st));
        issued = j + 1;
      }
      for (int j = max(0, issued - C::NQS); j < issued; ++j)
        drain_wait(bar(C::B_DOFULL + j % C::NQS), (j / C::NQS) & 1, 2000000000ull);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idSP = idesc_16_f32(128, C::BQ, false, false, F16);
      constexpr uint32_t idKV = idesc_16_f32(128, DP, false, true, F16);
      constexpr uint32_t idDQ =
          C::kDqInDp ? idesc_16_f32(128, C::BQ, true, true, F16) : idesc_16_f32(128, DP, true, true, F16);
      bool ok = bwait<DP>(bar(C::B_KVFULL), 0, ab);
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
      // X^T = A_tile * B_j^T with A in {K, V}, B_j in {Q_j, dO_j}; both K-major.
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
      // acc (+)= X^T(tmem, bf16) * Y_j (MN-major smem), K = BQ queries.
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
      auto issue_S = [&](int j) -> bool {
        if (!bwait<DP>(bar(C::B_QFULL + j % C::NQS), (j / C::NQS) & 1, ab)) return false;
        tc_fence_after();
        issue_T(dK0, sdesc_add(dQ0, (j % C::NQS) * C::Q_TILE), tmem + C::T_S);
        mma_commit(bar(C::B_SFULL));
        return true;
      };
      auto issue_dP = [&](int j) -> bool {
        if (!bwait<DP>(bar(C::B_DOFULL + j % C::NQS), (j / C::NQS) & 1, ab)) return false;
        tc_fence_after();
        issue_T(dV0, sdesc_add(dO0, (j % C::NQS) * C::Q_TILE), tmem + C::T_DP);
        mma_commit(bar(C::B_DPFULL));
        return true;
      };
      auto issue_dV = [&](int j) -> bool {
        if (!bwait<DP>(bar(C::B_PREADY), j & 1, ab)) return false;
        // dO_j has landed (dP(j) waited for it; the wait is kept for clarity)
        if (!bwait<DP>(bar(C::B_DOFULL + j % C::NQS), (j / C::NQS) & 1, ab)) return false;
        tc_fence_after();
        issue_acc(tmem + C::T_S, sdesc_add(dOmn, (j % C::NQS) * C::Q_TILE), tmem + C::T_DV,
                  j == 0);
        // D = 64: dO_j's last reader is dV(j) (D = 128: the dQ warps release the
        // stage, which then holds dQ(j))
        if (!C::kDqInDp) mma_commit(bar(C::B_DOFREE + j % C::NQS));
        return true;
      };
      // dK += dS^T Q_j. D = 64: A = dS^T from dP^T's columns (bf16, TMEM). D = 128:
      // A = dS^T from the shared-memory staging tile (K-major: key rows, 64-query
      // chunks), so that dQ(j) may go first and overwrite dP^T's columns at once.
      const uint64_t dDSk = sdesc_sw128(sb + C::OFF_DS, 0, 1024);
      auto issue_dK = [&](int j) -> bool {
        if (!C::kDqInDp && !bwait<DP>(bar(C::B_DSREADY), j & 1, ab)) return false;
        tc_fence_after();
        if constexpr (C::kDqInDp) {
          const uint64_t dA = opaque_u64(dDSk);
          const uint64_t dY = opaque_u64(sdesc_add(dQmn, (j % C::NQS) * C::Q_TILE));
#pragma unroll
          for (int kk = 0; kk < C::BQ / 16; ++kk)
            mma_ss(tmem + C::T_DK, sdesc_add(dA, (kk >> 2) * C::DS_CHUNK + (kk & 3) * 32),
                   sdesc_add(dY, kk * 2048), idKV, (j > 0 || kk > 0) ? 1u : 0u);
          // dQ(j) and dK(j) have read the staging tile
          mma_commit(bar(C::B_DSMFREE));
        } else {
          issue_acc(tmem + C::T_DP, sdesc_add(dQmn, (j % C::NQS) * C::Q_TILE), tmem + C::T_DK,
                    j == 0);
        }
        mma_commit(bar(C::B_QFREE + j % C::NQS));
        return true;
      };
      auto issue_dQ = [&](int j) -> bool {
        // D = 128: dQ(j) is the first product after dS(j)
        if (C::kDqInDp && !bwait<DP>(bar(C::B_DSREADY), j & 1, ab)) return false;
        // D = 64: dQ has columns of its own; wait until dQ(j-1) has been read out
        if (!C::kDqInDp && j > 0 && !bwait<DP>(bar(C::B_DQEMPTY), (j - 1) & 1, ab)) return false;
        tc_fence_after();
        const uint64_t dDS = opaque_u64(dDSmn);
        const uint64_t dKq = opaque_u64(dKmn);
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          if (C::kDqInDp) {
            // dQ^T [d][q] = K^T [d][key] * dS^T [key][q]
            mma_ss(tmem + C::T_DQ, sdesc_add(dKq, kk * 2048), sdesc_add(dDS, kk * 2048), idDQ,
                   kk > 0 ? 1u : 0u);
          } else {
            // dQ [q][d] = dS [q][key] * K [key][d]
            mma_ss(tmem + C::T_DQ, sdesc_add(dDS, kk * 2048), sdesc_add(dKq, kk * 2048), idDQ,
                   kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(bar(C::B_DQFULL));
        if (!C::kDqInDp) mma_commit(bar(C::B_DSMFREE));  // D = 128: after dK(j)
        return true;
      };
      if (ok && n > 0) {
        ok = issue_S(0) && issue_dP(0) && issue_dV(0);
        if (ok && n > 1) ok = issue_S(1);
      }
      for (int i = 0; ok && i < n; ++i) {
        if constexpr (C::kDqInDp) {
          // D = 128: dQ(i) into dP^T's columns as soon as dS(i) is staged, dK(i) (from
          // the staging tile) while the dQ warps read dQ(i) out, then dP(i+1) into
          // the freed columns
          if (!(ok = issue_dQ(i))) break;
          if (!(ok = issue_dK(i))) break;
          if (i + 1 < n) {
            if (!(ok = bwait<DP>(bar(C::B_DQEMPTY), i & 1, ab))) break;
            if (!(ok = issue_dP(i + 1))) break;
          }
        } else {
          // D = 64: dQ has columns of its own, so dP(i+1) follows dK(i) (the last
          // reader of dS^T(i) in dP^T's columns) at once and the softmax warps find it
          // done when they reach dS(i+1)
          if (!(ok = issue_dK(i))) break;
          if (i + 1 < n && !(ok = issue_dP(i + 1))) break;
          if (!(ok = issue_dQ(i))) break;
        }
        if (i + 1 < n) {
          if (!(ok = issue_dV(i + 1))) break;
          if (i + 2 < n && !(ok = issue_S(i + 2))) break;
        }
      }
      mma_commit(bar(C::B_ACCDONE));
      mma_commit(bar(C::B_DRAIN));
      drain_wait(bar(C::B_DRAIN), 0, 2000000000ull);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ dQ read-out
    const int t = threadIdx.x;  // TMEM lane: d (D = 128) or query row (D = 64)
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
    if (C::kDqInDp) {
      // thread t = d: dQ^T[d][q] for the block's 128 query rows, in two halves
      // of 64 rows; warp w stages and reduces box w (d = 32w .. 32w+31)
      for (int j = 0; j < n; ++j) {
        if (!bwait_warp<DP>(bar(C::B_DQFULL), j & 1, ab)) break;
        tc_fence_after();
        const int q0 = (qb0 + j) * C::BQ;
        const uint32_t stage = sbase + C::OFF_DO + (j % C::NQS) * C::Q_TILE;
        // this thread's element of query row q of the staged half sits at
        // rowa[q mod 8] + 1024 (q / 8): the eight swizzled offsets once per block,
        // so that each element costs one multiply and one store
        uint32_t rowa[8];
        {
          const uint32_t sg = stage + (t >> 5) * C::DQ_BOX + ((t & 3) << 2);
          const int unit = (t & 31) >> 2;
#pragma unroll
          for (int b = 0; b < 8; ++b) rowa[b] = sg + b * 128 + ((unit ^ b) << 4);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t r[64];
          tmem_ld32(tmem + lane_off + C::T_DQ + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(r));
          tmem_ld32(tmem + lane_off + C::T_DQ + 64 * h + 32,
                    *reinterpret_cast<uint32_t(*)[32]>(r + 32));
          tmem_wait_ld();
          if (h == 1) {
            // dQ^T's columns are read out: dP of the next block may overwrite them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_DQEMPTY));
            // the first half's reduction must have read the tile before it is reused
            if (lane == 0) bulk_wait_group_read0();
            __syncwarp();
          }
#pragma unroll
          for (int q = 0; q < 64; ++q)
            st_shared_f32(rowa[q & 7] + (q >> 3) * 1024, __uint_as_float(r[q]) * scale);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_3d(&tmdQ, stage + warp * C::DQ_BOX, 32 * warp, q0 + 64 * h, bh);
            bulk_commit_group();
          }
        }
        // the stage is the dO producer's again once both reductions have read it
        if (lane == 0) {
          bulk_wait_group_read0();
          mbar_arrive(bar(C::B_DOFREE + j % C::NQS));
        }
        __syncwarp();
      }
      if (lane == 0) bulk_wait_group0();
    } else {
      // thread t = query row: dQ[q][d], staged in smem and added by TMA. Each
      // warp stages and reduces its own 32 rows (a 32-row slab of the tile), so
      // the four warps never wait on one another.
      const uint32_t stage = sbase + C::OFF_DQ;
      for (int j = 0; j < n; ++j) {
        if (!bwait_warp<DP>(bar(C::B_DQFULL), j & 1, ab)) break;
        tc_fence_after();
        uint32_t r[DP];
#pragma unroll
        for (int c = 0; c < DP / 32; ++c)
          tmem_ld32(tmem + lane_off + C::T_DQ + 32 * c,
                    *reinterpret_cast<uint32_t(*)[32]>(r + 32 * c));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_DQEMPTY));
        // This warp's previous reduction must have finished reading its slab.
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
#pragma unroll
        for (int u = 0; u < DP / 4; ++u) {
          const uint32_t off = dq_stage_off(t, 4 * u, C::DQ_BOX);
          st_shared_v4(stage + off, __float_as_uint(__uint_as_float(r[4 * u]) * scale),
                       __float_as_uint(__uint_as_float(r[4 * u + 1]) * scale),
                       __float_as_uint(__uint_as_float(r[4 * u + 2]) * scale),
                       __float_as_uint(__uint_as_float(r[4 * u + 3]) * scale));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int q0 = (qb0 + j) * C::BQ + 32 * warp;
          for (int bx = 0; bx < (D + 31) / 32; ++bx)
            tma_reduce_add_3d(&tmdQ, stage + bx * C::DQ_BOX + 32 * warp * 128, bx * 32, q0, bh);
          bulk_commit_group();
        }
      }
      if (lane == 0) bulk_wait_group0();
    }
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
    for (int j = 0; j < n; ++j) {
      const int st = j % C::NQS;
      const int q0 = (qb0 + j) * C::BQ;
      if (!(ok = bwait_warp<DP>(bar(C::B_QFULL + st), (j / C::NQS) & 1, ab))) break;
      if (!(ok = bwait_warp<DP>(bar(C::B_SFULL), j & 1, ab))) break;
      tc_fence_after();
      // query column e of this warpgroup's slice is masked iff e < lim0 (e is q - q0 - g QPW)
      const int lim0 = qmin == INT_MIN ? INT_MIN
                                       : (qmin == INT_MAX ? INT_MAX : qmin - (q0 + g * C::QPW));
      const bool need_mask = lim0 > 0;
      const float *lse = sLse + st * C::BQ + g * C::QPW;
      const float *dvq = sDv + st * C::BQ + g * C::QPW;
      const uint32_t tS = tmem + lane_off + C::T_S + g * C::QPW;
      const uint32_t tDP = tmem + lane_off + C::T_DP + g * C::QPW;
      // P^T: all 64 scores of this thread's slice in flight, one wait
      float p[C::QPW];
      {
        uint32_t r[C::QPW];
        tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(r));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
        tmem_wait_ld();
        // P = exp2(s * scale * log2e - LSE log2e): the arguments of two exponents per
        // packed FMA (sm_100+ f32x2) against the negated staged LSE
        const uint64_t sc2 = f2pack(scale_log2, scale_log2);
#pragma unroll
        for (int e = 0; e < C::QPW; e += 4) {
          const float4 l4 = *reinterpret_cast<const float4 *>(lse + e);
          const float2 t01 = f2unpack(f2fma(
              f2pack(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), sc2, f2pack(l4.x, l4.y)));
          const float2 t23 = f2unpack(f2fma(
              f2pack(__uint_as_float(r[e + 2]), __uint_as_float(r[e + 3])), sc2,
              f2pack(l4.z, l4.w)));
          const float tv[4] = {t01.x, t01.y, t23.x, t23.y};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float x = ex2(tv[u]);
            if (need_mask && e + u < lim0) x = 0.f;
            p[e + u] = x;
          }
        }
      }
      {
        uint32_t pk[C::QPW / 2];
#pragma unroll
        for (int e = 0; e < C::QPW / 2; ++e) pk[e] = pack16<F16>(p[2 * e], p[2 * e + 1]);
        tmem_st32(tS, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_PREADY));

      if (!(ok = bwait_warp<DP>(bar(C::B_DPFULL), j & 1, ab))) break;
      // the dS^T staging tile is free once its readers of block j - 1 have completed
      // (dQ(j - 1), and at D = 128 dK(j - 1))
      if (j > 0 && !(ok = bwait_warp<DP>(bar(C::B_DSMFREE), (j - 1) & 1, ab))) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < C::QPW / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tDP + 32 * c, r);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const float4 d4 = *reinterpret_cast<const float4 *>(dvq + 32 * c + 2 * e);
          const int q = 32 * c + 2 * e;
          // dS = P (dP - Dvec) in pairs: one packed subtract and one packed multiply
          // per two elements (sm_100+ f32x2)
          const float2 a01 = f2unpack(f2mul(
              f2pack(p[q], p[q + 1]),
              f2sub(f2pack(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1])),
                    f2pack(d4.x, d4.y))));
          const float2 a23 = f2unpack(f2mul(
              f2pack(p[q + 2], p[q + 3]),
              f2sub(f2pack(__uint_as_float(r[2 * e + 2]), __uint_as_float(r[2 * e + 3])),
                    f2pack(d4.z, d4.w))));
          pk[e] = pack16<F16>(a01.x, a01.y);
          pk[e + 1] = pack16<F16>(a23.x, a23.y);
        }
        // D = 64: dK reads dS^T from dP^T's columns; D = 128: from the staging tile only
        if constexpr (!C::kDqInDp) tmem_st16(tDP + 16 * c, pk);
        // dS^T row kr, queries ql .. ql+31 into the swizzled smem tile
        const int ql = g * C::QPW + 32 * c;
        const uint32_t chunk = sDS + (ql >> 6) * C::DS_CHUNK + kr * 128;
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
        mbar_arrive(bar(C::B_DSREADY));
        mbar_arrive(bar(C::B_QFREE + st));
      }
    }
    // dK (scaled) and dV of this key block
    if (ok && n > 0) ok = bwait_warp<DP>(bar(C::B_ACCDONE), 0, ab);
    if (ok && n == 0 && kg < Lk_rows) {
      // no query sees this key block: dK = dV = 0 (warpgroup g writes its half)
      const size_t row = (static_cast<size_t>(bh) * Lk_rows + kg) * D;
      for (int c = 0; c < DP / 2 && g * (DP / 2) + c < D; c += 4) {
        store4<F16>(dV, out16, row + g * (DP / 2) + c, 0.f, 0.f, 0.f, 0.f);
        store4<F16>(dK, out16, row + g * (DP / 2) + c, 0.f, 0.f, 0.f, 0.f);
      }
    }
    if (ok && n > 0) {
      tc_fence_after();
      const bool valid = kg < Lk_rows;
      const size_t row = (static_cast<size_t>(bh) * Lk_rows + (valid ? kg : 0)) * D;
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
                   const float *Dvec, float *dQ, void *dK, void *dV, const MgProblem &p,
                   unsigned int *err, cudaStream_t st) {
  using C = BwdCfg<DP>;
  const int BH = p.B * p.H;
  CUtensorMap tq, tk, tv, tdo, tdq;
  cudaError_t e;
  if ((e = mg_tmap_16(&tq, Q, p.D, p.L, BH, C::BQ, F16)) != cudaSuccess) return e;
  if ((e = mg_tmap_16(&tdo, dO, p.D, p.L, BH, C::BQ, F16)) != cudaSuccess) return e;
  if ((e = mg_tmap_16(&tk, K, p.D, p.Lk, BH, C::BN, F16)) != cudaSuccess) return e;
  if ((e = mg_tmap_16(&tv, V, p.D, p.Lk, BH, C::BN, F16)) != cudaSuccess) return e;
  // dQ add-reductions: D = 64 in 32-row slabs (one per read-out warp), D = 128
  // in [64 rows][32 columns] boxes (one per warp and half block)
  if ((e = mg_tmap_f32(&tdq, dQ, p.D, p.L, BH, C::DQ_TMA_ROWS)) != cudaSuccess) return e;
  auto kern = accel_dkdv_kernel<DP, F16>;
  if ((e = mg_set_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM_BYTES,
                            (DP == 64 ? 8 : 9) + (F16 ? 12 : 0))) != cudaSuccess)
    return e;
  const int nkb = (p.Lk + C::BN - 1) / C::BN;
  const long long grid = static_cast<long long>(nkb) * BH;
  kern<<<static_cast<unsigned>(grid), C::NTHREADS, C::SMEM_BYTES, st>>>(
      tq, tk, tv, tdo, tdq, LSE, Dvec, dQ, dK, dV, p.out16, BH, p.L, p.Lk, p.D, p.causal, p.off,
      p.scale, p.scale * kLog2e, err, mg_wait_limit_ns(), p.kv_len, p.H, p.br);
  return cudaGetLastError();
}

}  // namespace

cudaError_t mg_launch_accel_dkdv(const void *Q, const void *K, const void *V, const void *dO,
                                 const float *LSE, const float *Dvec, float *dQ, void *dK,
                                 void *dV, const MgProblem &p, unsigned int *err,
                                 cudaStream_t st) {
  if (!dQ) return cudaErrorInvalidValue;  // dK/dV alone: mg_launch_accel_dkdv_pp
  if (p.f16) {
    if (p.D <= 64) return launch<64, true>(Q, K, V, dO, LSE, Dvec, dQ, dK, dV, p, err, st);
    return launch<128, true>(Q, K, V, dO, LSE, Dvec, dQ, dK, dV, p, err, st);
  }
  if (p.D <= 64) return launch<64, false>(Q, K, V, dO, LSE, Dvec, dQ, dK, dV, p, err, st);
  return launch<128, false>(Q, K, V, dO, LSE, Dvec, dQ, dK, dV, p, err, st);
}
