// Forward kernels: bf16 value tensors, vector path.
#include "msda_launch.cuh"

namespace msda {
template cudaError_t launch_forward_path<__nv_bfloat16, true>(const Params &, int, int, const __nv_bfloat16 *, const float *,
                                                     const float *, __nv_bfloat16 *, cudaStream_t);
}  // namespace msda
