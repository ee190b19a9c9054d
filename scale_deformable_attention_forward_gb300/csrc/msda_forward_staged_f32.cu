// Staged-level forward kernels: binary32 value.
#include "msda_forward_staged.cuh"

namespace msda {
template cudaError_t launch_forward_staged<float>(const Params &, StagePlan, const CUtensorMap &, size_t, int, int,
                                              const float *, const float *, const float *, float *,
                                              unsigned int *, cudaStream_t);
}  // namespace msda
