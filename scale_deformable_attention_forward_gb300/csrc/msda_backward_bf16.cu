// Backward kernels for bf16 value tensors.
#include "msda_launch.cuh"

namespace msda {
template cudaError_t launch_backward<__nv_bfloat16>(const Params &, bool, int, int, const __nv_bfloat16 *, const __nv_bfloat16 *,
                                          const float *, const float *, float *, float *, float *, int,
                                          cudaStream_t);
}  // namespace msda
