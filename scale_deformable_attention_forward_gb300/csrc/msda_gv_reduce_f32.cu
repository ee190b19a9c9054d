// Cell-sorted grad_value reduction kernels: f32 grad_output, vector and scalar paths.
#include "msda_launch.cuh"

namespace msda {
template cudaError_t launch_gv_reduce<float, true>(const Params &, int, int, const float *, const BwdBuffers &,
                                                  cudaStream_t);
template cudaError_t launch_gv_reduce<float, false>(const Params &, int, int, const float *, const BwdBuffers &,
                                                   cudaStream_t);
}  // namespace msda
