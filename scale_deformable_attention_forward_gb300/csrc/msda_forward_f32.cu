// Forward kernels for f32 value tensors.
#include "msda_launch.cuh"

namespace msda {
template cudaError_t launch_forward<float>(const Params &, bool, int, int, const float *, const float *,
                                         const float *, float *, cudaStream_t);
}  // namespace msda
