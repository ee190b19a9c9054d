// Forward kernels for bf16 value tensors.
#include "msda_launch.cuh"

namespace msda {
template cudaError_t launch_forward<__nv_bfloat16>(const Params &, bool, int, int, const __nv_bfloat16 *, const float *,
                                         const float *, __nv_bfloat16 *, cudaStream_t);
}  // namespace msda
