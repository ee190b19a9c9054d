// Tile-sorted grad_value reduction kernels: bf16 grad_output (vector path).
#include "msda_launch.cuh"

namespace msda {
template cudaError_t launch_tile_reduce<__nv_bfloat16, true>(const Params &, int, int, const __nv_bfloat16 *, const BwdBuffers &,
                                                    cudaStream_t);
}  // namespace msda
