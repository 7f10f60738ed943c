// tmap.h -- host-side TMA tensor-map encoding for the ACCEL kernels.
//
// Every [B][H][L][D] tensor is described as a 3-D tensor (D, L, B*H) so that
// rows at or past L of one head read as zeros instead of the next head's rows.
// cuTensorMapEncodeTiled is reached through the runtime's driver entry-point
// query, so the library does not link libcuda directly. Encoding is host-only
// work on a caller-owned struct: no device allocation.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

// bf16 tensor, boxes of 64 columns x box_rows rows, 128-byte swizzle.
cudaError_t mg_tmap_bf16(CUtensorMap *m, const void *ptr, int D, int L, int BH, int box_rows);
// bf16 (f16 = false) or f16 tensor, boxes of 64 columns x box_rows rows,
// 128-byte swizzle.
cudaError_t mg_tmap_16(CUtensorMap *m, const void *ptr, int D, int L, int BH, int box_rows,
                       bool f16);
// f32 tensor, boxes of 32 columns x box_rows rows, 128-byte swizzle (dQ reduce).
cudaError_t mg_tmap_f32(CUtensorMap *m, const void *ptr, int D, int L, int BH, int box_rows);
// 16-bit 4-D tensor (dims[0] innermost, contiguous; strides in bytes of dims
// 1..3, multiples of 16), boxes of 64 x box1 x box2 x box3 elements, 128-byte
// swizzle, zero fill out of bounds (channels-last convolution operands).
cudaError_t mg_tmap_16_4d(CUtensorMap *m, const void *ptr, const long long dims[4],
                          const long long strides_bytes[3], const int box[4], bool f16);
// f32 tensor of rank 3 or 4 (dims[0] innermost, contiguous; strides in bytes of
// dims 1.., multiples of 16), boxes of 32 x box[1] x ... elements, 128-byte
// swizzle (accumulator tiles staged in shared memory and stored or add-reduced).
cudaError_t mg_tmap_f32_nd(CUtensorMap *m, const void *ptr, int rank, const long long *dims,
                           const long long *strides_bytes, const int *box);
