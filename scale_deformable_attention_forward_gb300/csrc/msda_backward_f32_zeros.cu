// Backward kernels: f32 value tensors, vector path, zeros padding.
#include "msda_launch.cuh"

namespace msda {
template cudaError_t launch_backward_pad<float, 0>(const Params &, int, int, const float *,
                                                          const float *, const float *, const float *,
                                                          const BwdBuffers &, cudaStream_t);
}  // namespace msda
