// strict_common.cuh -- device helpers of the STRICT_F32 kernels: cp.async
// staging of f32 row tiles into padded shared memory, warp-shuffle row
// reductions. Plain sm_80+ instructions; no tensor-core path is used here.
#pragma once

#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

namespace mg_strict {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, int src_bytes) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Stage rows [r0, r0 + NROWS) of a row-major [L][D] f32 matrix into shared
// memory with a row stride of `stride` floats. Rows at or beyond L are
// zero-filled (the copy reads nothing from global memory for them).
template <int D, int NROWS, int NT>
__device__ __forceinline__ void stage_rows(float *s, int stride, const float *g, int r0, int L,
                                           int tid) {
  constexpr int C = D / 4;  // 16-byte chunks per row
  static_assert((NROWS * C) % NT == 0, "tile must split evenly over the block");
#pragma unroll
  for (int it = 0; it < (NROWS * C) / NT; ++it) {
    const int idx = tid + it * NT;
    const int r = idx / C, c = idx % C;
    const int gr = r0 + r;
    const bool ok = gr < L;
    const float *src = g + static_cast<size_t>(ok ? gr : 0) * D + c * 4;
    cp_async16(s + r * stride + c * 4, src, ok ? 16 : 0);
  }
}

// Stage NV (<= NT) consecutive floats v[r0 .. r0+NV) (zero past L).
template <int NV>
__device__ __forceinline__ void stage_vec(float *s, const float *g, int r0, int L, int tid) {
  static_assert(NV % 4 == 0, "vector tile is staged in 16-byte chunks");
  if (tid < NV / 4) {
    const int r = r0 + tid * 4;
    // L is not a multiple of 4 in general: copy only the valid floats.
    int valid = L - r;
    valid = valid < 0 ? 0 : (valid > 4 ? 4 : valid);
    if (valid == 4 && ((reinterpret_cast<uintptr_t>(g + r) & 15) == 0)) {
      cp_async16(s + tid * 4, g + r, 16);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) s[tid * 4 + e] = (e < valid) ? g[r + e] : 0.f;
    }
  }
}

template <int WIDTH>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = WIDTH / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
template <int WIDTH>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = WIDTH / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int VW>
struct VecT;
template <>
struct VecT<4> {
  using T = float4;
};
template <>
struct VecT<2> {
  using T = float2;
};

__device__ __forceinline__ float vget(const float4 &v, int c) {
  return c == 0 ? v.x : (c == 1 ? v.y : (c == 2 ? v.z : v.w));
}
__device__ __forceinline__ float vget(const float2 &v, int c) { return c == 0 ? v.x : v.y; }

}  // namespace mg_strict
