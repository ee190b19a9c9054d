// msda_launch.cuh -- host-side launchers: pick the kernel instantiation for
// (vector width, lanes per sample G, channel chunks per lane NCH).
#pragma once

#include "msda_kernels.cuh"

namespace msda {

template <typename T> struct VecWidth;
template <> struct VecWidth<float> { static constexpr int value = 4; };          // 16-byte loads
template <> struct VecWidth<__nv_bfloat16> { static constexpr int value = 8; };  // 16-byte loads

inline unsigned grid_for_rows(uint32_t rows) { return (rows + (kThreads / 32) - 1) / (kThreads / 32); }

// Instantiated combinations: vector path G in {1..32} with NCH 1, G = 32 with
// NCH in {2,4,8}; scalar path G = 32 with NCH in {1,2,4,8}.
#define MSDA_VECTOR_CASES(X) X(1, 1) X(2, 1) X(4, 1) X(8, 1) X(16, 1) X(32, 1) X(32, 2) X(32, 4) X(32, 8)
#define MSDA_SCALAR_CASES(X) X(32, 1) X(32, 2) X(32, 4) X(32, 8)

template <typename T>
cudaError_t launch_forward(const Params &p, bool vec, int G, int NCH, const T *value, const float *loc,
                           const float *attn, T *out, cudaStream_t stream) {
    if (p.rows == 0) return cudaSuccess;
    const dim3 grid(grid_for_rows(p.rows)), block(kThreads);
    constexpr int V = VecWidth<T>::value;
#define MSDA_FWD_V(GG, NN)                                                                        \
    if (vec && G == GG && NCH == NN) {                                                            \
        msda_forward_kernel<T, V, GG, NN><<<grid, block, 0, stream>>>(p, value, loc, attn, out);  \
        return cudaGetLastError();                                                                \
    }
#define MSDA_FWD_S(GG, NN)                                                                        \
    if (!vec && G == GG && NCH == NN) {                                                           \
        msda_forward_kernel<T, 1, GG, NN><<<grid, block, 0, stream>>>(p, value, loc, attn, out);  \
        return cudaGetLastError();                                                                \
    }
    MSDA_VECTOR_CASES(MSDA_FWD_V)
    MSDA_SCALAR_CASES(MSDA_FWD_S)
#undef MSDA_FWD_V
#undef MSDA_FWD_S
    return cudaErrorInvalidConfiguration;
}

template <typename T>
cudaError_t launch_backward(const Params &p, bool vec, int G, int NCH, const T *grad_out, const T *value,
                            const float *loc, const float *attn, float *gv_acc, float *grad_loc,
                            float *grad_attn, int flags, cudaStream_t stream) {
    if (p.rows == 0) return cudaSuccess;
    const dim3 grid(grid_for_rows(p.rows)), block(kThreads);
    constexpr int V = VecWidth<T>::value;
#define MSDA_BWD_V(GG, NN)                                                                        \
    if (vec && G == GG && NCH == NN) {                                                            \
        msda_backward_kernel<T, V, GG, NN><<<grid, block, 0, stream>>>(                           \
            p, grad_out, value, loc, attn, gv_acc, grad_loc, grad_attn, flags);                   \
        return cudaGetLastError();                                                                \
    }
#define MSDA_BWD_S(GG, NN)                                                                        \
    if (!vec && G == GG && NCH == NN) {                                                           \
        msda_backward_kernel<T, 1, GG, NN><<<grid, block, 0, stream>>>(                           \
            p, grad_out, value, loc, attn, gv_acc, grad_loc, grad_attn, flags);                   \
        return cudaGetLastError();                                                                \
    }
    MSDA_VECTOR_CASES(MSDA_BWD_V)
    MSDA_SCALAR_CASES(MSDA_BWD_S)
#undef MSDA_BWD_V
#undef MSDA_BWD_S
    return cudaErrorInvalidConfiguration;
}

}  // namespace msda
