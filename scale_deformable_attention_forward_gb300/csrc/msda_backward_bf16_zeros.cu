// Backward kernels: bf16 value tensors, vector path, zeros padding.
#include "msda_launch.cuh"

namespace msda {
template cudaError_t launch_backward_pad<__nv_bfloat16, 0>(const Params &, int, int, const __nv_bfloat16 *,
                                                          const __nv_bfloat16 *, const float *, const float *,
                                                          const BwdBuffers &, cudaStream_t);
}  // namespace msda
