// Forward kernels: f32 value tensors, vector path.
#include "msda_launch.cuh"

namespace msda {
template cudaError_t launch_forward_path<float, true>(const Params &, int, int, const float *, const float *,
                                                     const float *, float *, cudaStream_t);
}  // namespace msda
