// accel_fwd.cu -- ACCEL_BF16 tiled attention forward on tcgen05 tensor cores.
//
// The tiled attention forward archetype of "Meganeura: Portable GPU Training
// and Inference through Vulkan and Metal" (Section 3.3) under its accelerated
// contract (Section 4.2: matrix inputs rounded to a 16-bit format, f32
// accumulation, f32 stores). The pages' kernel is a WGSL cooperative-matrix
// shader; this one is written for sm_103a:
//
// * One CTA owns two 128-row query tiles (A, B) of one (b, h) head and walks
//   the key axis in 128-key tiles. Q, K, V arrive by TMA (128-byte swizzle) into
//   shared memory: Q once, K and V through an NSTAGE ring.
// * Warp 9 issues every MMA from one thread: S_q = Q_q K^T (f32 in TMEM,
//   128 x 128) and O_q += P_q V with P taken straight from TMEM (bf16, written
//   over the first 64 columns of S_q). Issue order S_A S_B PV_A S_A' PV_B S_B'
//   ... lets one softmax warpgroup work while the tensor core serves the other.
// * Warps 0-3 and 4-7 are the softmax warpgroups of tiles A and B: one thread
//   per query row (its TMEM lane), all 128 scores of a tile loaded with a
//   single TMEM wait. Online softmax in base 2 with log2(e) folded into the
//   scale. The running reference max only moves when a row max grows
//   by more than 8 (a factor 256 in P); O in TMEM is then rescaled after the
//   previous P V finished. Any reference max gives the same exact result once
//   O is divided by the row sum taken against that same max.
// * Warp 8 is the TMA producer.
// Every wait is bounded (a few seconds); a wait that gives up sets the device
// error word and the CTA leaves through the same teardown as a normal exit.
#include <string.h>

#include <algorithm>

#include "internal.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace {

using namespace mg_tc;

template <int DP>
struct FwdCfg {
  static constexpr int BM = 128;  // query rows per tile (TMEM lanes)
  static constexpr int NQ = 2;    // query tiles per CTA
  static constexpr int BN = 128;  // keys per tile
  static constexpr int NSTAGE = DP == 128 ? 2 : 3;
  static constexpr int NCHUNK = DP / 64;  // 64-column boxes per row
  static constexpr int Q_TILE = BM * DP * 2;
  static constexpr int KV_TILE = BN * DP * 2;
  static constexpr int BOX_Q = BM * 128;
  static constexpr int BOX_KV = BN * 128;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQ * Q_TILE;
  static constexpr int OFF_V = OFF_K + NSTAGE * KV_TILE;
  static constexpr int OFF_BAR = OFF_V + NSTAGE * KV_TILE;
  // barriers
  static constexpr int B_QFULL = 0;
  static constexpr int B_KFULL = 1;
  static constexpr int B_VFULL = B_KFULL + NSTAGE;
  static constexpr int B_KVEMPTY = B_VFULL + NSTAGE;
  static constexpr int B_SFULL = B_KVEMPTY + NSTAGE;
  static constexpr int B_PREADY = B_SFULL + NQ;
  static constexpr int B_ODONE = B_PREADY + NQ;
  static constexpr int B_DRAIN = B_ODONE + NQ;
  static constexpr int NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base
  static constexpr int NTHREADS = 320;
  static constexpr int TMEM_COLS = 512;
  static constexpr int T_S = 0;     // S_q at q * 128
  static constexpr int T_O = 256;   // O_q at 256 + q * DP
  static_assert(T_O + NQ * DP <= TMEM_COLS, "TMEM column budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  // Teardown wait for our own copies / MMAs in flight; ignores the abort flag.
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return false;
  }
  return true;
}

template <int DP, bool F16>
__global__ void __launch_bounds__(320, 1)
    accel_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, void *__restrict__ Ov, int out16,
                     float *__restrict__ LSE, int BH, int L, int Lk_rows, int D, int causal,
                     int off0, float scale_log2, unsigned int *err, unsigned long long timeout_ns,
                     int fault, int G, const int *__restrict__ kv_len, int H, int br) {
  using C = FwdCfg<DP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Heads run in groups of G whose K and V fit in L2 together: all query blocks
  // of a group's heads are scheduled before the next group, so every key tile
  // of a head is read from HBM about once. Within a group the heaviest causal
  // query blocks (largest qb) go first, heads alternating.
  const int nqb = (L + 255) / 256;
  const long long per_group = static_cast<long long>(G) * nqb;
  const int grp = static_cast<int>(blockIdx.x / per_group);
  const int r_in = static_cast<int>(blockIdx.x - grp * per_group);
  const int h0 = grp * G;
  const int Gg = min(G, BH - h0);  // the last group may hold fewer heads
  const int qb = nqb - 1 - r_in / Gg;
  const int bh = h0 + r_in % Gg;
  const int q0 = qb * 256;
  // this head's keys: Lk (all rows, or the batch element's padded length);
  // causal: query i sees key j iff j <= i + off
  const MgKeys keys = mg_keys(kv_len, bh, H, L, Lk_rows, off0, br);
  const int Lk = keys.len, off = keys.off;
  const int nkt = (Lk + C::BN - 1) / C::BN;
  int nT[2];
  for (int q = 0; q < 2; ++q) {
    const int last = min(q0 + (q + 1) * C::BM, L) - 1 + off;  // last key the tile's rows see
    nT[q] = !causal ? nkt : (last < 0 ? 0 : min(nkt, last / C::BN + 1));
  }
  const int nmax = max(nT[0], nT[1]);

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 256) {
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i >= C::B_PREADY && i < C::B_PREADY + C::NQ) cnt = 128;
      mbar_init(bar(i), cnt);
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmQ);
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
      int issued = 0, skipped = -1;
      mbar_arrive_expect_tx(bar(C::B_QFULL), C::NQ * C::Q_TILE);
      for (int q = 0; q < C::NQ; ++q)
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(sbase + C::OFF_Q + q * C::Q_TILE + c * C::BOX_Q, &tmQ, c * 64,
                      q0 + q * C::BM, bh, bar(C::B_QFULL));
      for (int j = 0; j < nmax; ++j) {
        const int s = j % C::NSTAGE;
        if (j >= C::NSTAGE &&
            !mbar_wait(bar(C::B_KVEMPTY + s), ((j / C::NSTAGE) - 1) & 1, ab))
          break;
        if (fault == 1 && j == 1) {
          // Injected fault (tests only): key tile 1 is never loaded, so the
          // MMA issuer's bounded wait on it must expire and report a timeout.
          skipped = j;
        } else {
          mbar_arrive_expect_tx(bar(C::B_KFULL + s), C::KV_TILE);
          for (int c = 0; c < C::NCHUNK; ++c)
            tma_load_3d(sbase + C::OFF_K + s * C::KV_TILE + c * C::BOX_KV, &tmK, c * 64,
                        j * C::BN, bh, bar(C::B_KFULL + s));
        }
        mbar_arrive_expect_tx(bar(C::B_VFULL + s), C::KV_TILE);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(sbase + C::OFF_V + s * C::KV_TILE + c * C::BOX_KV, &tmV, c * 64,
                      j * C::BN, bh, bar(C::B_VFULL + s));
        issued = j + 1;
      }
      // Wait for our own copies in flight before the CTA can exit.
      drain_wait(bar(C::B_QFULL), 0, 2000000000ull);
      for (int j = max(0, issued - C::NSTAGE); j < issued; ++j) {
        const int s = j % C::NSTAGE;
        if (j != skipped) drain_wait(bar(C::B_KFULL + s), (j / C::NSTAGE) & 1, 2000000000ull);
        drain_wait(bar(C::B_VFULL + s), (j / C::NSTAGE) & 1, 2000000000ull);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_16_f32(128, C::BN, false, false, F16);
      constexpr uint32_t idO = idesc_16_f32(128, DP, false, true, F16);
      bool ok = mbar_wait(bar(C::B_QFULL), 0, ab);
      // base descriptors; each MMA adds a compile-time byte offset
      const uint32_t sb = opaque_u32(sbase);
      const uint64_t dQ0 = sdesc_sw128(sb + C::OFF_Q, 0, 1024);
      const uint64_t dK0 = sdesc_sw128(sb + C::OFF_K, 0, 1024);
      const uint64_t dV0 = sdesc_sw128(sb + C::OFF_V, C::BOX_KV, 1024);
      int kwaited = -1;
      auto wait_k = [&](int j) -> bool {
        if (kwaited >= j) return true;
        kwaited = j;
        return mbar_wait(bar(C::B_KFULL + j % C::NSTAGE), (j / C::NSTAGE) & 1, ab);
      };
      auto issue_S = [&](int q, int j) -> bool {
        if (!wait_k(j)) return false;
        tc_fence_after();
        const uint64_t dq = opaque_u64(sdesc_add(dQ0, q * C::Q_TILE));
        const uint64_t dk = opaque_u64(sdesc_add(dK0, (j % C::NSTAGE) * C::KV_TILE));
        const uint32_t dS = tmem + C::T_S + q * 128;
#pragma unroll
        for (int kk = 0; kk < DP / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::BOX_Q + (kk & 3) * 32;
          const uint32_t offk = (kk >> 2) * C::BOX_KV + (kk & 3) * 32;
          mma_ss(dS, sdesc_add(dq, off), sdesc_add(dk, offk), idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::B_SFULL + q));
        return true;
      };
      auto issue_PV = [&](int q, int j) -> bool {
        if (!mbar_wait(bar(C::B_PREADY + q), j & 1, ab)) return false;
        if (!mbar_wait(bar(C::B_VFULL + j % C::NSTAGE), (j / C::NSTAGE) & 1, ab)) return false;
        tc_fence_after();
        const uint64_t dv = opaque_u64(sdesc_add(dV0, (j % C::NSTAGE) * C::KV_TILE));
        const uint32_t dO = tmem + C::T_O + q * DP, aP = tmem + C::T_S + q * 128;
        const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          mma_ts(dO, aP + kk * 8, sdesc_add(dv, kk * 2048), idO, kk > 0 ? 1u : acc0);
        mma_commit(bar(C::B_ODONE + q));
        return true;
      };
      if (ok && nT[0] > 0) ok = issue_S(0, 0);
      if (ok && nT[1] > 0) ok = issue_S(1, 0);
      for (int j = 0; ok && j < nmax; ++j) {
        if (j < nT[0]) {
          ok = issue_PV(0, j);
          if (ok && j + 1 < nT[0]) ok = issue_S(0, j + 1);
        }
        if (ok) ok = issue_PV(1, j);
        if (ok) mma_commit(bar(C::B_KVEMPTY + j % C::NSTAGE));
        if (ok && j + 1 < nT[1]) ok = issue_S(1, j + 1);
      }
      // Drain every MMA this thread issued before TMEM and smem are released.
      mma_commit(bar(C::B_DRAIN));
      drain_wait(bar(C::B_DRAIN), 0, 2000000000ull);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int q = warp >> 2;
    const int rl = 32 * (warp & 3) + lane;  // row within the query tile = TMEM lane
    const int qrow = q0 + q * C::BM + rl;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_off + C::T_S + q * 128;
    const uint32_t tO = tmem + lane_off + C::T_O + q * DP;
    const int n = nT[q];
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      ok = mbar_wait_warp(bar(C::B_SFULL + q), j & 1, ab);
      if (!ok) break;
      tc_fence_after();
      const int k0 = j * C::BN;
      const bool need_mask =
          (k0 + C::BN > Lk) || (causal && k0 + C::BN - 1 > q0 + q * C::BM + off);
      // last allowed key of this row (negative: none)
      const int lim = causal ? min(Lk - 1, qrow + off) : (Lk - 1);
      // One pass: all 128 scores of the row in flight, a single wait.
      uint32_t r[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * c));
      tmem_wait_ld();
      if (need_mask) {
#pragma unroll
        for (int e = 0; e < 128; ++e)
          if (k0 + e > lim) r[e] = __float_as_uint(-INFINITY);
      }
      // row maximum as eight independent chains (three-input maxima at D = 128:
      // about 68 instructions on a 10-step dependent path, not 127 on a 127-step one)
      float m8[8];
      if constexpr (DP == 128) {
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = fmaxf(__uint_as_float(r[i]), __uint_as_float(r[8 + i]));
#pragma unroll
        for (int e = 16; e < 128; e += 16) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            m8[i] = fmax3(m8[i], __uint_as_float(r[e + i]), __uint_as_float(r[e + 8 + i]));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = __uint_as_float(r[i]);
#pragma unroll
        for (int e = 8; e < 128; e += 8) {
#pragma unroll
          for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], __uint_as_float(r[e + i]));
        }
      }
      const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      const float mx2 = mx * scale_log2;
      const bool need = mx2 > m_ref + 8.f;
      const bool warp_need = __any_sync(0xffffffffu, need);
      const float m_new = warp_need ? fmaxf(m_ref, mx2) : m_ref;
      // a row that has seen no allowed key yet keeps m = -inf; its P is 0
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      // P = exp2(s * scale * log2e - m_new), packed to 16 bits (masked scores are
      // -inf -> 0). At D = 128 in pairs: one packed FMA per two exponents' arguments
      // and one packed add per two terms of the row sum (measured 3% faster there;
      // at D = 64 the pairs cost registers and the scalar form is kept)
      uint32_t pk[64];
      float rs;
      if constexpr (DP == 128) {
        const uint64_t sc2 = f2pack(scale_log2, scale_log2), nm2 = f2pack(-m_use, -m_use);
        uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const float2 t = f2unpack(
              f2fma(f2pack(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1])), sc2, nm2));
          const float p0 = ex2(t.x), p1 = ex2(t.y);
          rs2[e & 3] = f2add(rs2[e & 3], f2pack(p0, p1));
          pk[e] = pack16<F16>(p0, p1);
        }
        const float2 ra = f2unpack(f2add(rs2[0], rs2[1])), rb = f2unpack(f2add(rs2[2], rs2[3]));
        rs = (ra.x + ra.y) + (rb.x + rb.y);
      } else {
        float rs4[4] = {0.f, 0.f, 0.f, 0.f};  // row sum as four independent chains
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const float p0 = ex2(fmaf(__uint_as_float(r[2 * e]), scale_log2, -m_use));
          const float p1 = ex2(fmaf(__uint_as_float(r[2 * e + 1]), scale_log2, -m_use));
          rs4[e & 3] += p0 + p1;
          pk[e] = pack16<F16>(p0, p1);
        }
        rs = (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
      }
      if (warp_need) {
        const float alpha = m_new == -INFINITY ? 1.f : ex2(m_ref - m_new);
        if (j > 0) {
          // O holds the sum up to tile j-1: wait for that P V, then rescale.
          ok = mbar_wait_warp(bar(C::B_ODONE + q), (j - 1) & 1, ab);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < DP / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + 32 * c, o);
          }
        }
        l *= alpha;
        m_ref = m_new;
      }
      // P over the first 64 columns of S (all of S has been read)
      tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(pk));
      tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
      l += rs;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::B_PREADY + q));
    }
    if (ok && n > 0) ok = mbar_wait_warp(bar(C::B_ODONE + q), (n - 1) & 1, ab);
    if (ok && n == 0 && qrow < L) {
      // no key tile at all for this query tile: every row has an empty softmax
      const size_t o0 = (static_cast<size_t>(bh) * L + qrow) * D;
      for (int c = 0; c < D; c += 4) {
        if (out16)
          *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(Ov) + o0 + c) = make_uint2(0u, 0u);
        else
          *reinterpret_cast<float4 *>(static_cast<float *>(Ov) + o0 + c) =
              make_float4(0.f, 0.f, 0.f, 0.f);
      }
      LSE[static_cast<size_t>(bh) * L + qrow] = -INFINITY;
    }
    if (ok && n > 0) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;  // l = 0: no allowed key, O = 0
      const bool valid = qrow < L;
      const size_t o0 = (static_cast<size_t>(bh) * L + (valid ? qrow : 0)) * D;
#pragma unroll
      for (int c = 0; c < DP / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tO + 32 * c, r);
        tmem_wait_ld();
        if (valid && 32 * c < D) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float a = __uint_as_float(r[e]) * inv, b = __uint_as_float(r[e + 1]) * inv;
            const float cc = __uint_as_float(r[e + 2]) * inv, d = __uint_as_float(r[e + 3]) * inv;
            if (out16)
              *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(Ov) + o0 + 32 * c + e) =
                  pack16x4<F16>(a, b, cc, d);
            else
              *reinterpret_cast<float4 *>(static_cast<float *>(Ov) + o0 + 32 * c + e) =
                  make_float4(a, b, cc, d);
          }
        }
      }
      if (valid)
        LSE[static_cast<size_t>(bh) * L + qrow] = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
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

// Test hook: MG_FAULT_INJECT=skip_k_tile makes the forward's producer skip one
// key-tile load (read once per process; off unless the variable is set).
int fault_mode() {
  static int v = [] {
    const char *e = getenv("MG_FAULT_INJECT");
    return (e && strcmp(e, "skip_k_tile") == 0) ? 1 : 0;
  }();
  return v;
}

template <int DP, bool F16>
cudaError_t launch(const void *Q, const void *K, const void *V, void *O, float *LSE,
                   const MgProblem &p, unsigned int *err, cudaStream_t st) {
  using C = FwdCfg<DP>;
  const int BH = p.B * p.H;
  CUtensorMap tq, tk, tv;
  cudaError_t e;
  if ((e = mg_tmap_16(&tq, Q, p.D, p.L, BH, C::BM, F16)) != cudaSuccess) return e;
  if ((e = mg_tmap_16(&tk, K, p.D, p.Lk, BH, C::BN, F16)) != cudaSuccess) return e;
  if ((e = mg_tmap_16(&tv, V, p.D, p.Lk, BH, C::BN, F16)) != cudaSuccess) return e;
  auto kern = accel_fwd_kernel<DP, F16>;
  if ((e = mg_set_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM_BYTES,
                            (DP == 64 ? 6 : 7) + (F16 ? 12 : 0))) != cudaSuccess)
    return e;
  const int nqb = (p.L + 255) / 256;
  const long long grid = static_cast<long long>(nqb) * BH;
  // heads per group: K and V of a group (bf16) within 32 MB of the 129 MB L2
  const long long kv_head = 2LL * p.Lk * p.D * 2;
  const int G = static_cast<int>(std::max(1LL, std::min<long long>(BH, (32LL << 20) / kv_head)));
  kern<<<static_cast<unsigned>(grid), C::NTHREADS, C::SMEM_BYTES, st>>>(
      tq, tk, tv, O, p.out16, LSE, BH, p.L, p.Lk, p.D, p.causal, p.off, p.scale * kLog2e, err,
      mg_wait_limit_ns(), fault_mode(), G, p.kv_len, p.H, p.br);
  return cudaGetLastError();
}

}  // namespace

cudaError_t mg_launch_accel_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                const MgProblem &p, unsigned int *err, cudaStream_t st) {
  if (p.f16) {
    if (p.D <= 64) return launch<64, true>(Q, K, V, O, LSE, p, err, st);
    return launch<128, true>(Q, K, V, O, LSE, p, err, st);
  }
  if (p.D <= 64) return launch<64, false>(Q, K, V, O, LSE, p, err, st);
  return launch<128, false>(Q, K, V, O, LSE, p, err, st);
}
