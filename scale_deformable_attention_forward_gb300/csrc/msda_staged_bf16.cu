// Staged-level forward and backward kernels: bfloat16 value.
#include "msda_staged_launch.cuh"

namespace msda {
template cudaError_t launch_forward_staged<__nv_bfloat16>(const Params &, StagePlan, const CUtensorMap &, size_t, int, int,
                                              const __nv_bfloat16 *, const float *, const float *, __nv_bfloat16 *,
                                              unsigned int *, cudaStream_t);
template cudaError_t launch_backward_staged<__nv_bfloat16>(const Params &, StagePlan, size_t, int, int, const __nv_bfloat16 *,
                                                const __nv_bfloat16 *, const float *, const float *, float *, float *,
                                                float *, cudaStream_t);
}  // namespace msda
