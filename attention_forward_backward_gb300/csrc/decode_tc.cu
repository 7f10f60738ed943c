// decode_tc.cu -- split-key attention forward for a few query rows (decoding)
// on the tcgen05 tensor cores, for the accelerated contracts.
//
// The forward of the attention node ("Meganeura: Portable GPU Training and
// Inference through Vulkan and Metal", Section 3.1) for Lq <= 8 query rows of
// one head against a long key axis, split over CTAs exactly as the CUDA-core
// decode kernel splits it (decode_fwd.cu): every CTA writes the online-softmax
// state of its keys as one partial record per query row, [O (unnormalised,
// relative to m), m (base 2), l], which the merge kernel there combines.
//
// With eight query rows every K and V element feeds eight FFMAs, which keeps
// an FP32 kernel from streaming K and V at HBM speed. Here both products run on
// the tensor cores with the keys on the MMA's M axis and the query rows padded
// to N = 16:
//   S^T [128 keys x 16] = K_tile [128 x D] . Q^T        (A = K, K-major; B = Q)
//   O^T [D x 16]       += V_tile^T [D x 128] . P^T      (A = V, MN-major; B = P)
// S^T lands in tensor memory with one key per lane; the four softmax warps own
// one key each, exchange per-row maxima through shared memory once per tile,
// and write P^T (16-bit, RNE, the contract's operand rounding) into shared memory
// as the second product's B operand. The running reference maximum of a row
// only moves when a tile's maximum exceeds it by more than 8 (a factor 256 in
// P); O^T in tensor memory is then rescaled after the previous product
// finished. Each thread keeps the row sums of its own keys, added once at the
// end. Roles: warps 0-3 softmax and read-out (lane = key, later lane = output
// column d), warp 4 TMA producer (Q once, K and V through a ring), warp 5 MMA
// issuer. Every wait is bounded.
#include <math.h>

#include "internal.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace {

using namespace mg_tc;

constexpr int kRows = 8;  // query rows handled (Lq <= 8); the MMA's N is 16

template <int DP>
struct DecCfg {
  static constexpr int BN = 128;                // keys per tile (TMEM lanes of S^T)
  static constexpr int NQ = 16;                 // MMA N: query rows, zero padded
  static constexpr int NST = DP == 128 ? 3 : 4; // K/V ring stages
  static constexpr int NCHUNK = DP / 64;        // 64-column boxes per row
  static constexpr int KV_TILE = BN * DP * 2;
  static constexpr int BOX_KV = BN * 128;
  static constexpr int Q_BOX = NQ * 128;        // [16 rows][64 cols]
  static constexpr int P_BYTES = NQ * BN * 2;   // P^T [16 rows][128 keys]: 2 boxes of [16][64]
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = 4096;
  static constexpr int OFF_V = OFF_K + NST * KV_TILE;
  // the O^T product reads a 128-wide M operand: at DP = 64 its second half falls
  // in the next 16 KB (garbage rows of O^T that are never read), kept inside
  static constexpr int OFF_P = OFF_V + NST * KV_TILE + (DP == 64 ? BOX_KV : 0);
  static constexpr int OFF_RED = OFF_P + 2 * P_BYTES;  // [2][4 warps][8 rows] f32: tile maxima
  static constexpr int OFF_LSUM = OFF_RED + 2 * 4 * kRows * 4;  // [4 warps][8 rows]: row sums
  static constexpr int OFF_BAR = OFF_LSUM + 4 * kRows * 4;
  static constexpr int B_QFULL = 0;
  static constexpr int B_KFULL = 1;                  // NST
  static constexpr int B_VFULL = B_KFULL + NST;      // NST
  static constexpr int B_KVEMPTY = B_VFULL + NST;    // NST
  static constexpr int B_SFULL = B_KVEMPTY + NST;    // 2: S^T buffer ready
  static constexpr int B_PREADY = B_SFULL + 2;       // 2: P^T written (128 threads)
  static constexpr int B_PVDONE = B_PREADY + 2;      // 2: O^T product of that P done
  static constexpr int B_RED = B_PVDONE + 2;         // 2: row maxima exchanged (4 warps)
  static constexpr int B_ODONE = B_RED + 2;
  static constexpr int B_LSUM = B_ODONE + 1;         // row sums written (4 warps)
  static constexpr int NBAR = B_LSUM + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int NTHREADS = 192;
  static constexpr int TMEM_COLS = 64;
  static constexpr int T_S = 0;    // S^T buffers at 0 and 16
  static constexpr int T_O = 32;   // O^T (lane = d, column = query row)
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return false;
  }
  return true;
}

// 16-bit element (row q, key k) of P^T in its K-major, 128-byte-swizzled layout:
// box k / 64 of [16 rows][64 keys], 16-byte piece ((k mod 64) / 8) ^ (q mod 8).
__device__ __forceinline__ uint32_t p_offset(int q, int k) {
  return static_cast<uint32_t>((k >> 6) * 2048 + q * 128 + ((((k & 63) >> 3) ^ (q & 7)) << 4) +
                               (k & 7) * 2);
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

template <bool F16>
__device__ __forceinline__ uint16_t to16(float x) {
  if (F16) return __half_as_ushort(__float2half_rn(x));
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

template <int DP, bool F16, int LQ>
__global__ void __launch_bounds__(192, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, float *__restrict__ part, int Lq,
                     int Lk, int D, int causal, int off, int S, int chunk, float scale_log2,
                     unsigned int *err, unsigned long long timeout_ns) {
  using C = DecCfg<DP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return sbase + C::OFF_BAR + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  float *red = reinterpret_cast<float *>(smem + C::OFF_RED);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = static_cast<int>(blockIdx.x) / S, sp = static_cast<int>(blockIdx.x) % S;
  const int k_begin = sp * chunk;
  const int k_end = min(Lk, k_begin + chunk);
  const int n = (k_end - k_begin + C::BN - 1) / C::BN;  // >= 1: k_begin < Lk

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 128) {
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == C::B_PREADY || i == C::B_PREADY + 1) cnt = 128;
      if (i == C::B_RED || i == C::B_RED + 1 || i == C::B_LSUM) cnt = 4;
      mbar_init(bar(i), cnt);
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (threadIdx.x < 128) {
    // rows 8..15 of both P^T buffers stay zero (padding of the MMA's N)
    for (int b = 0; b < 2; ++b)
      for (int q = kRows; q < C::NQ; ++q)
        st_shared_u16(sbase + C::OFF_P + b * C::P_BYTES + p_offset(q, threadIdx.x), 0);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab = make_abort(abort_flag, err, timeout_ns);
  // the merge may be scheduled now; it waits for this grid's records itself
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::B_QFULL), C::NCHUNK * C::Q_BOX);
      for (int c = 0; c < C::NCHUNK; ++c)
        tma_load_3d(sbase + C::OFF_Q + c * C::Q_BOX, &tmQ, c * 64, 0, bh, bar(C::B_QFULL));
      int issued = 0;
      for (int j = 0; j < n; ++j) {
        const int st = j % C::NST;
        if (j >= C::NST && !mbar_wait(bar(C::B_KVEMPTY + st), ((j / C::NST) - 1) & 1, ab)) break;
        const int row = k_begin + j * C::BN;
        mbar_arrive_expect_tx(bar(C::B_KFULL + st), C::KV_TILE);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(sbase + C::OFF_K + st * C::KV_TILE + c * C::BOX_KV, &tmK, c * 64, row, bh,
                      bar(C::B_KFULL + st));
        mbar_arrive_expect_tx(bar(C::B_VFULL + st), C::KV_TILE);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(sbase + C::OFF_V + st * C::KV_TILE + c * C::BOX_KV, &tmV, c * 64, row, bh,
                      bar(C::B_VFULL + st));
        issued = j + 1;
      }
      // no copy may still be in flight when the CTA leaves
      drain_wait(bar(C::B_QFULL), 0, 2000000000ull);
      for (int j = max(0, issued - C::NST); j < issued; ++j) {
        drain_wait(bar(C::B_KFULL + j % C::NST), (j / C::NST) & 1, 2000000000ull);
        drain_wait(bar(C::B_VFULL + j % C::NST), (j / C::NST) & 1, 2000000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_16_f32(128, C::NQ, false, false, F16);
      constexpr uint32_t idO = idesc_16_f32(128, C::NQ, true, false, F16);
      const uint32_t sb = opaque_u32(sbase);
      const uint64_t dQ0 = sdesc_sw128(sb + C::OFF_Q, 0, 1024);
      const uint64_t dK0 = sdesc_sw128(sb + C::OFF_K, 0, 1024);
      const uint64_t dVmn = sdesc_sw128(sb + C::OFF_V, C::BOX_KV, 1024);
      const uint64_t dP0 = sdesc_sw128(sb + C::OFF_P, 0, 1024);
      bool ok = mbar_wait(bar(C::B_QFULL), 0, ab);
      // S^T(j) = K_j Q^T into S buffer j & 1
      auto issue_S = [&](int j) -> bool {
        const int st = j % C::NST;
        if (!mbar_wait(bar(C::B_KFULL + st), (j / C::NST) & 1, ab)) return false;
        tc_fence_after();
        const uint64_t dK = opaque_u64(sdesc_add(dK0, st * C::KV_TILE));
        const uint32_t d = tmem + C::T_S + 16 * (j & 1);
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk)
          mma_ss(d, sdesc_add(dK, (kk >> 2) * C::BOX_KV + (kk & 3) * 32),
                 sdesc_add(dQ0, (kk >> 2) * C::Q_BOX + (kk & 3) * 32), idS, kk > 0 ? 1u : 0u);
        mma_commit(bar(C::B_SFULL + (j & 1)));
        return true;
      };
      if (ok) ok = issue_S(0);
      if (ok && n > 1) ok = issue_S(1);
      for (int j = 0; ok && j < n; ++j) {
        const int st = j % C::NST, b = j & 1;
        if (!(ok = mbar_wait(bar(C::B_PREADY + b), (j >> 1) & 1, ab))) break;
        if (!(ok = mbar_wait(bar(C::B_VFULL + st), (j / C::NST) & 1, ab))) break;
        tc_fence_after();
        // O^T += V_j^T P_j^T
        const uint64_t dV = opaque_u64(sdesc_add(dVmn, st * C::KV_TILE));
        const uint64_t dP = opaque_u64(sdesc_add(dP0, b * C::P_BYTES));
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          mma_ss(tmem + C::T_O, sdesc_add(dV, kk * 2048),
                 sdesc_add(dP, (kk >> 2) * 2048 + (kk & 3) * 32), idO,
                 (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(C::B_PVDONE + b));
        mma_commit(bar(C::B_KVEMPTY + st));
        if (j + 2 < n && !(ok = issue_S(j + 2))) break;
      }
      mma_commit(bar(C::B_ODONE));
      drain_wait(bar(C::B_ODONE), 0, 2000000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (warps 0-3)
    const int kl = 32 * warp + lane;  // key within a tile = lane of S^T
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
    float m[kRows], lp[kRows];
#pragma unroll
    for (int q = 0; q < LQ; ++q) {
      m[q] = -INFINITY;  // reference maximum (base 2), the same in every thread
      lp[q] = 0.f;       // sum of this thread's P against that reference
    }
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int b = j & 1;
      if (!(ok = mbar_wait_warp(bar(C::B_SFULL + b), (j >> 1) & 1, ab))) break;
      tc_fence_after();
      uint32_t r[16];
      tmem_ld16(tmem + lane_off + C::T_S + 16 * b, r);
      tmem_wait_ld();
      const int kg = k_begin + j * C::BN + kl;
      float sc[kRows], tm[kRows];
#pragma unroll
      for (int q = 0; q < LQ; ++q) {
        const bool allowed = kg < k_end && q < Lq && (!causal || kg <= q + off);
        sc[q] = allowed ? __uint_as_float(r[q]) * scale_log2 : -INFINITY;
        tm[q] = sc[q];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int q = 0; q < LQ; ++q) tm[q] = fmaxf(tm[q], __shfl_xor_sync(0xffffffffu, tm[q], o));
      }
      float *rb = red + b * 4 * kRows;
      if (lane == 0) {
#pragma unroll
        for (int q = 0; q < LQ; ++q) rb[warp * kRows + q] = tm[q];
        mbar_arrive(bar(C::B_RED + b));
      }
      if (!(ok = mbar_wait_warp(bar(C::B_RED + b), (j >> 1) & 1, ab))) break;
      // tile maximum of every row; the reference moves only when it grows by > 8
      bool resc = false;
      float alpha[kRows];
#pragma unroll
      for (int q = 0; q < LQ; ++q) {
        const float t = fmaxf(fmaxf(rb[q], rb[kRows + q]), fmaxf(rb[2 * kRows + q], rb[3 * kRows + q]));
        alpha[q] = 1.f;
        if (t > m[q] + 8.f) {
          alpha[q] = exp2f(m[q] - t);  // m = -inf: 0
          m[q] = t;
          resc = true;
        }
      }
      // P^T buffer b was last read by the O^T product of tile j - 2
      if (j >= 2 && !(ok = mbar_wait_warp(bar(C::B_PVDONE + b), ((j - 2) >> 1) & 1, ab))) break;
      if (resc) {
#pragma unroll
        for (int q = 0; q < LQ; ++q) lp[q] *= alpha[q];
        if (j > 0) {
          // O^T holds the products of tiles < j: rescale it once tile j - 1's is done
          if (!(ok = mbar_wait_warp(bar(C::B_PVDONE + (b ^ 1)), ((j - 1) >> 1) & 1, ab))) break;
          tc_fence_after();
          uint32_t o[16];
          tmem_ld16(tmem + lane_off + C::T_O, o);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < LQ; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha[q]);
          tmem_st16(tmem + lane_off + C::T_O, o);
          tmem_wait_st();
        }
      }
      const uint32_t pb = sbase + C::OFF_P + b * C::P_BYTES;
#pragma unroll
      for (int q = 0; q < LQ; ++q) {
        const float mu = m[q] == -INFINITY ? 0.f : m[q];  // no allowed key yet: P = 0
        const float pv = exp2f(sc[q] - mu);
        lp[q] += pv;
        st_shared_u16(pb + p_offset(q, kl), to16<F16>(pv));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::B_PREADY + b));
    }
    // ------------------------------------------------------------ partial record
    // row sums over the CTA's keys, then O^T (lane = output column d)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int q = 0; q < LQ; ++q) lp[q] += __shfl_xor_sync(0xffffffffu, lp[q], o);
    }
    float *ls = reinterpret_cast<float *>(smem + C::OFF_LSUM);
    if (lane == 0) {
#pragma unroll
      for (int q = 0; q < LQ; ++q) ls[warp * kRows + q] = lp[q];
      mbar_arrive(bar(C::B_LSUM));
    }
    if (ok) ok = mbar_wait_warp(bar(C::B_LSUM), 0, ab);
    if (ok) ok = mbar_wait_warp(bar(C::B_ODONE), 0, ab);
    if (ok) {
      tc_fence_after();
      uint32_t o[16];
      tmem_ld16(tmem + lane_off + C::T_O, o);
      tmem_wait_ld();
      float *rec = part + (static_cast<size_t>(bh) * S + sp) * Lq * (D + 4);
#pragma unroll
      for (int q = 0; q < LQ; ++q) {
        if (q >= Lq) break;
        if (kl < D) rec[q * (D + 4) + kl] = __uint_as_float(o[q]);
        if (kl == 0) {
          rec[q * (D + 4) + D] = m[q];
          rec[q * (D + 4) + D + 1] = ls[q] + ls[kRows + q] + ls[2 * kRows + q] + ls[3 * kRows + q];
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

template <int DP, bool F16, int LQ>
cudaError_t launch(const void *Q, const void *K, const void *V, float *part, const MgProblem &p,
                   int S, int chunk, unsigned int *err, cudaStream_t st) {
  using C = DecCfg<DP>;
  const int BH = p.B * p.H;
  CUtensorMap tq, tk, tv;
  cudaError_t e;
  if ((e = mg_tmap_16(&tq, Q, p.D, p.L, BH, C::NQ, F16)) != cudaSuccess) return e;
  if ((e = mg_tmap_16(&tk, K, p.D, p.Lk, BH, C::BN, F16)) != cudaSuccess) return e;
  if ((e = mg_tmap_16(&tv, V, p.D, p.Lk, BH, C::BN, F16)) != cudaSuccess) return e;
  auto kern = decode_tc_kernel<DP, F16, LQ>;
  constexpr int lq_slot = LQ == 1 ? 0 : (LQ == 2 ? 1 : (LQ == 4 ? 2 : 3));
  if ((e = mg_set_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM_BYTES,
                            48 + lq_slot * 4 + (DP == 64 ? 0 : 1) + (F16 ? 2 : 0))) !=
      cudaSuccess)
    return e;
  kern<<<static_cast<unsigned>(static_cast<long long>(BH) * S), C::NTHREADS, C::SMEM_BYTES, st>>>(
      tq, tk, tv, part, p.L, p.Lk, p.D, p.causal, p.off, S, chunk, p.scale * kLog2e, err,
      mg_wait_limit_ns());
  return cudaGetLastError();
}

// Row count rounded up to 1, 2, 4 or 8 (the softmax handles that many rows).
template <bool F16>
cudaError_t dispatch_rows(const void *Q, const void *K, const void *V, float *part,
                          const MgProblem &p, int S, int chunk, unsigned int *err,
                          cudaStream_t st) {
  const bool d64 = p.D <= 64;
  if (p.L <= 1) return d64 ? launch<64, F16, 1>(Q, K, V, part, p, S, chunk, err, st)
                           : launch<128, F16, 1>(Q, K, V, part, p, S, chunk, err, st);
  if (p.L <= 2) return d64 ? launch<64, F16, 2>(Q, K, V, part, p, S, chunk, err, st)
                           : launch<128, F16, 2>(Q, K, V, part, p, S, chunk, err, st);
  if (p.L <= 4) return d64 ? launch<64, F16, 4>(Q, K, V, part, p, S, chunk, err, st)
                           : launch<128, F16, 4>(Q, K, V, part, p, S, chunk, err, st);
  return d64 ? launch<64, F16, 8>(Q, K, V, part, p, S, chunk, err, st)
             : launch<128, F16, 8>(Q, K, V, part, p, S, chunk, err, st);
}

}  // namespace

cudaError_t mg_launch_decode_tc_partial(const void *Q, const void *K, const void *V, float *part,
                                        const MgProblem &p, int S, int chunk, unsigned int *err,
                                        cudaStream_t st) {
  return p.f16 ? dispatch_rows<true>(Q, K, V, part, p, S, chunk, err, st)
               : dispatch_rows<false>(Q, K, V, part, p, S, chunk, err, st);
}
