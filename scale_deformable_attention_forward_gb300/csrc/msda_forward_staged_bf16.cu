// Staged-level forward kernels: bfloat16 value.
#include "msda_forward_staged.cuh"

namespace msda {
template cudaError_t launch_forward_staged<__nv_bfloat16>(const Params &, StagePlan, const CUtensorMap &, size_t, int, int,
                                              const __nv_bfloat16 *, const float *, const float *, __nv_bfloat16 *,
                                              unsigned int *, cudaStream_t);
}  // namespace msda
