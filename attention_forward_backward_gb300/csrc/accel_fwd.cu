// placeholder: replaced by the tcgen05 forward
#include "internal.h"
cudaError_t mg_launch_accel_fwd(const __nv_bfloat16 *, const __nv_bfloat16 *, const __nv_bfloat16 *, float *, float *, const MgProblem &, unsigned int *, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t mg_launch_accel_dkdv(const __nv_bfloat16 *, const __nv_bfloat16 *, const __nv_bfloat16 *, const __nv_bfloat16 *, const float *, const float *, float *, float *, float *, const MgProblem &, unsigned int *, cudaStream_t) { return cudaErrorNotSupported; }
