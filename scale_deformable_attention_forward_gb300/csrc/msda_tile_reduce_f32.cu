// Tile-sorted grad_value reduction kernels: f32 grad_output (vector path).
#include "msda_launch.cuh"

namespace msda {
template cudaError_t launch_tile_reduce<float, true>(const Params &, int, int, const float *, const BwdBuffers &,
                                                    cudaStream_t);
}  // namespace msda
