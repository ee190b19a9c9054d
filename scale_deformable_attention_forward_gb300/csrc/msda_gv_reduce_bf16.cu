// Cell-sorted grad_value reduction kernels: bf16 grad_output, vector and scalar paths.
#include "msda_launch.cuh"

namespace msda {
template cudaError_t launch_gv_reduce<__nv_bfloat16, true>(const Params &, int, int, const __nv_bfloat16 *, const BwdBuffers &,
                                                  cudaStream_t);
template cudaError_t launch_gv_reduce<__nv_bfloat16, false>(const Params &, int, int, const __nv_bfloat16 *, const BwdBuffers &,
                                                   cudaStream_t);
}  // namespace msda
