// Forward kernels: f32 value tensors, scalar path.
#include "msda_launch.cuh"

namespace msda {
template cudaError_t launch_forward_path<float, false>(const Params &, int, int, const float *, const float *,
                                                     const float *, float *, cudaStream_t);
}  // namespace msda
