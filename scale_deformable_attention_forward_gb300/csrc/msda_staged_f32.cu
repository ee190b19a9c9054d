// Staged-level forward and backward kernels: binary32 value.
#include "msda_staged_launch.cuh"

namespace msda {
template cudaError_t launch_forward_staged<float>(const Params &, StagePlan, const CUtensorMap &, size_t, int, int,
                                              const float *, const float *, const float *, float *,
                                              unsigned int *, cudaStream_t);
template cudaError_t launch_backward_staged<float>(const Params &, StagePlan, size_t, int, int, const float *,
                                                const float *, const float *, const float *, float *, float *,
                                                float *, cudaStream_t);
}  // namespace msda
