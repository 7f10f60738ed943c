// tmap.cu -- TMA tensor-map encoding (see tmap.h).
#include <mutex>

#include "tmap.h"

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

cudaError_t encode(CUtensorMap *m, CUtensorMapDataType dt, int elem_bytes, const void *ptr, int D,
                   int L, int BH, int box_cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * elem_bytes,
                                 static_cast<cuuint64_t>(L) * D * elem_bytes};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols),
                             static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, dt, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t mg_tmap_bf16(CUtensorMap *m, const void *ptr, int D, int L, int BH, int box_rows) {
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, D, L, BH, 64, box_rows);
}

cudaError_t mg_tmap_16(CUtensorMap *m, const void *ptr, int D, int L, int BH, int box_rows,
                       bool f16) {
  return encode(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                ptr, D, L, BH, 64, box_rows);
}

cudaError_t mg_tmap_f32(CUtensorMap *m, const void *ptr, int D, int L, int BH, int box_rows) {
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, D, L, BH, 32, box_rows);
}

cudaError_t mg_tmap_16_4d(CUtensorMap *m, const void *ptr, const long long dims[4],
                          const long long strides_bytes[3], const int box[4], bool f16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t d[4], st[3];
  cuuint32_t b[4];
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  for (int i = 0; i < 4; ++i) {
    if (dims[i] < 1 || box[i] < 1 || box[i] > 256) return cudaErrorInvalidValue;
    d[i] = static_cast<cuuint64_t>(dims[i]);
    b[i] = static_cast<cuuint32_t>(box[i]);
  }
  for (int i = 0; i < 3; ++i) st[i] = static_cast<cuuint64_t>(strides_bytes[i]);
  CUresult r = fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                  const_cast<void *>(ptr), d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t mg_tmap_f32_nd(CUtensorMap *m, const void *ptr, int rank, const long long *dims,
                           const long long *strides_bytes, const int *box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  if (rank < 2 || rank > 5 || box[0] != 32) return cudaErrorInvalidValue;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], estr[5];
  for (int i = 0; i < rank; ++i) {
    if (dims[i] < 1 || box[i] < 1 || box[i] > 256) return cudaErrorInvalidValue;
    d[i] = static_cast<cuuint64_t>(dims[i]);
    b[i] = static_cast<cuuint32_t>(box[i]);
    estr[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) st[i] = static_cast<cuuint64_t>(strides_bytes[i]);
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, const_cast<void *>(ptr), d, st, b,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
