// msda_staged_launch.cuh -- launchers of the staged-level forward and backward (one
// instantiation of each per value dtype, in its own translation unit).
#pragma once

#include "msda_launch.cuh"
#include "msda_staged.cuh"

namespace msda {

constexpr int kStageMinRows = 32;  // queries a block serves at least: one per group of a 256-thread block

// Blocks per (b, h) and queries per block for a staged kernel with per_sm
// resident blocks per SM.
inline void staged_grid(const Params &p, int per_sm, StagePlan &sp) {
    const uint64_t pairs = p.rows / (uint32_t)p.N_q;  // B * N_h
    const uint64_t slots = (uint64_t)(per_sm > 0 ? per_sm : 1) * (uint64_t)(p.n_sm > 0 ? p.n_sm : 1);
    // blocks per (b, h): the fewest that minimise (waves of the grid) x (queries per block), the
    // critical path when every block's queries cost about the same
    const int64_t most = (p.N_q + kStageMinRows - 1) / kStageMinRows;
    int64_t bpb = 1;
    uint64_t best = UINT64_MAX;
    for (int64_t k = 1; k <= most; ++k) {
        const uint64_t waves = (pairs * (uint64_t)k + slots - 1) / slots;
        const uint64_t cost = waves * (uint64_t)((p.N_q + k - 1) / k);
        if (cost < best) {
            best = cost;
            bpb = k;
        }
    }
    sp.bpb = (int)bpb;
    sp.rpb = (int)((p.N_q + bpb - 1) / bpb);
}

template <typename T, int V, int GG, int NN, int PAD>
cudaError_t staged_launch(const Params &p, StagePlan sp, const CUtensorMap &tmap, size_t smem, const T *value,
                          const float *loc, const float *attn, T *out, unsigned int *timeouts, cudaStream_t stream) {
    auto kernel = msda_forward_staged_kernel<T, V, GG, NN, PAD>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    staged_grid(p, resident_blocks(kernel, kThreads, smem), sp);
    const uint64_t pairs = p.rows / (uint32_t)p.N_q;
    kernel<<<(unsigned)(pairs * (uint64_t)sp.bpb), kThreads, smem, stream>>>(p, sp, tmap, value, loc, attn, out,
                                                                             timeouts);
    return cudaGetLastError();
}

template <typename T, int V, int GG, int NN, int PAD>
cudaError_t staged_bwd_launch(const Params &p, StagePlan sp, size_t smem, const T *grad_out, const T *value,
                              const float *loc, const float *attn, float *gv_acc, float *grad_loc, float *grad_attn,
                              cudaStream_t stream) {
    auto kernel = msda_backward_staged_kernel<T, V, GG, NN, PAD>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    staged_grid(p, resident_blocks(kernel, kThreads, smem), sp);
    const uint64_t pairs = p.rows / (uint32_t)p.N_q;
    kernel<<<(unsigned)(pairs * (uint64_t)sp.bpb), kThreads, smem, stream>>>(p, sp, grad_out, value, loc, attn,
                                                                             gv_acc, grad_loc, grad_attn);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_forward_staged(const Params &p, StagePlan sp, const CUtensorMap &tmap, size_t smem, int G, int NCH,
                                  const T *value, const float *loc, const float *attn, T *out,
                                  unsigned int *timeouts, cudaStream_t stream) {
    if (p.rows == 0) return cudaSuccess;
    constexpr int V = VecWidth<T>::value;
#define MSDA_STAGED_CASE(GG, NN)                                                                  \
    if constexpr (reachable(GG, NN, MSDA_FWD_LANES) && specialised_shape(GG, NN)) {               \
        if (G == GG && NCH == NN)                                                                 \
            return p.padding == 0                                                                 \
                       ? staged_launch<T, V, GG, NN, 0>(p, sp, tmap, smem, value, loc, attn, out, timeouts, stream) \
                       : staged_launch<T, V, GG, NN, 1>(p, sp, tmap, smem, value, loc, attn, out, timeouts, stream); \
    }
    MSDA_SHAPES(MSDA_STAGED_CASE)
#undef MSDA_STAGED_CASE
    return cudaErrorInvalidConfiguration;
}

template <typename T>
cudaError_t launch_backward_staged(const Params &p, StagePlan sp, size_t smem, int G, int NCH, const T *grad_out,
                                   const T *value, const float *loc, const float *attn, float *gv_acc,
                                   float *grad_loc, float *grad_attn, cudaStream_t stream) {
    if (p.rows == 0) return cudaSuccess;
    constexpr int V = BwdVecWidth<T>::value;
#define MSDA_STAGED_BWD_CASE(GG, NN)                                                              \
    if constexpr (reachable(GG, NN, MSDA_BWD_LANES) && specialised_shape(GG, NN)) {               \
        if (G == GG && NCH == NN)                                                                 \
            return p.padding == 0 ? staged_bwd_launch<T, V, GG, NN, 0>(p, sp, smem, grad_out, value, loc, attn, \
                                                                       gv_acc, grad_loc, grad_attn, stream) \
                                  : staged_bwd_launch<T, V, GG, NN, 1>(p, sp, smem, grad_out, value, loc, attn, \
                                                                       gv_acc, grad_loc, grad_attn, stream); \
    }
    MSDA_SHAPES(MSDA_STAGED_BWD_CASE)
#undef MSDA_STAGED_BWD_CASE
    return cudaErrorInvalidConfiguration;
}

}  // namespace msda
