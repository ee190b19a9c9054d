// msda_launch.cuh -- host-side launchers: pick the kernel instantiation for
// (vector width, lanes per row G, channel chunks per lane NCH, padding,
// backward outputs, grad_value path) and size the grids.
#pragma once

#include "msda_kernels.cuh"
#include "msda_shape.cuh"

namespace msda {

#define MSDA_SHAPES(X)                                                                            \
    X(1, 1) X(2, 1) X(2, 2) X(2, 4) X(2, 8) X(4, 1) X(4, 2) X(4, 4) X(4, 8) X(8, 1) X(8, 2) X(8, 4) \
    X(8, 8) X(16, 1) X(16, 2) X(16, 4) X(16, 8) X(32, 1) X(32, 2) X(32, 4) X(32, 8)

// Blocks of a kernel that fit on one multiprocessor at once (0 if unknown).
template <typename K>
int resident_blocks(K kernel, int threads, size_t smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess) return 0;
    return n;
}

// Row kernels (one group of G lanes per row): as many blocks as fit on the GPU
// at once (fewer when the rows do not fill them); the blocks sweep the rows
// with a grid stride.
template <typename K>
unsigned row_grid(K kernel, int G, const Params &p) {
    const unsigned gpb = kThreads / G;  // rows a block works on at once
    uint64_t blocks = (((uint64_t)p.rows << p.split_log2) + gpb - 1) / gpb;  // work items: rows x parts
    const int per_sm = resident_blocks(kernel, kThreads, 0);
    if (per_sm > 0 && p.n_sm > 0 && (uint64_t)per_sm * p.n_sm < blocks) blocks = (uint64_t)per_sm * p.n_sm;
    if (blocks < 1) blocks = 1;
    return (unsigned)blocks;
}

// SPLIT: the kernel with the row split (p.split_log2 > 0, small problems);
// the others run whole rows (their launches see split_log2 = 0).
template <typename T, int V, int GG, int NN, int PAD, bool GEN, bool SPLIT, bool FULL = false>
cudaError_t fwd_launch(const Params &p, const T *value, const float *loc, const float *attn, T *out,
                       cudaStream_t stream) {
    Params q = p;
    if (!SPLIT) q.split_log2 = 0;
    auto kernel = msda_forward_kernel<T, V, GG, NN, PAD, GEN, SPLIT, FULL>;
    const unsigned blocks = row_grid(kernel, GG, q);
    kernel<<<blocks, kThreads, 0, stream>>>(q, value, loc, attn, out);
    return cudaGetLastError();
}

// The forward always runs the instantiation with the row split compiled in:
// with split_log2 = 0 it takes whole rows, and unlike the split-free
// instantiation (its batch loop with a constant step) it compiles without
// spills for one and two chunks a lane (binary32 and bfloat16).
#ifndef MSDA_FWD_FULL
#define MSDA_FWD_FULL 1
#endif
template <typename T, int V, int GG, int NN, int PAD, bool GEN>
cudaError_t fwd_split(const Params &p, const T *value, const float *loc, const float *attn, T *out,
                      cudaStream_t stream) {
    // full rows (no partial batch, no masked lane): the guard-free instantiation
    if constexpr (MSDA_FWD_FULL && !GEN) {
        if (p.NLP > 0 && p.NLP % GG == 0 && p.chunks == GG * NN)
            return fwd_launch<T, V, GG, NN, PAD, GEN, true, true>(p, value, loc, attn, out, stream);
    }
    return fwd_launch<T, V, GG, NN, PAD, GEN, true>(p, value, loc, attn, out, stream);
}

template <typename T, int V, int GG, int NN>
cudaError_t fwd_shape(const Params &p, const T *value, const float *loc, const float *attn, T *out,
                      cudaStream_t stream) {
    if constexpr (V > 1 && specialised_shape(GG, NN)) {
        const bool gen = p.loc_dt != 0 || p.logits != 0;
        if (p.padding == 0)
            return gen ? fwd_split<T, V, GG, NN, 0, true>(p, value, loc, attn, out, stream)
                       : fwd_split<T, V, GG, NN, 0, false>(p, value, loc, attn, out, stream);
        return gen ? fwd_split<T, V, GG, NN, 1, true>(p, value, loc, attn, out, stream)
                   : fwd_split<T, V, GG, NN, 1, false>(p, value, loc, attn, out, stream);
    } else {
        return fwd_launch<T, V, GG, NN, -1, true, false>(p, value, loc, attn, out, stream);
    }
}

// Forward kernels of the vector (VECTOR = true) or scalar path; each
// (dtype, path) pair is instantiated in its own translation unit.
template <typename T, bool VECTOR>
cudaError_t launch_forward_path(const Params &p, int G, int NCH, const T *value, const float *loc,
                                const float *attn, T *out, cudaStream_t stream) {
    constexpr int V = VECTOR ? VecWidth<T>::value : 1;
#define MSDA_FWD_CASE(GG, NN)                                                                     \
    if constexpr (reachable(GG, NN, MSDA_FWD_LANES)) {                                            \
        if (G == GG && NCH == NN) return fwd_shape<T, V, GG, NN>(p, value, loc, attn, out, stream); \
    }
    MSDA_SHAPES(MSDA_FWD_CASE)
#undef MSDA_FWD_CASE
    return cudaErrorInvalidConfiguration;
}

// The warp-aggregated grad_value scatter (msda_backward_kernel, AGG) serves
// the 32-channel-row shape (8 lanes, one 4-element chunk a lane) whenever the
// kernel adds grad_value and p.aggregate is set (the default; the environment
// variable MSDA_BWD_AGGREGATE=0 selects the plain per-corner atomics).
template <typename T, int V, int GG, int NN, int PAD, int FL, bool SPLIT, bool AGG, bool FULL>
cudaError_t bwd_launch_full(const Params &q, const T *grad_out, const T *value, const float *loc, const float *attn,
                            const BwdBuffers &bb, cudaStream_t stream) {
    auto kernel = msda_backward_kernel<T, V, GG, NN, PAD, FL, SPLIT, AGG, FULL>;
    const unsigned blocks = row_grid(kernel, GG, q);
    kernel<<<blocks, kThreads, 0, stream>>>(q, grad_out, value, loc, attn, bb.gv_acc, bb.grad_loc, bb.grad_attn);
    return cudaGetLastError();
}

// Full rows (every batch G samples, every lane all NCH chunks): the
// guard-free instantiation, for the padding-specialised whole-row kernels with
// the aggregated scatter or without grad_value (measured faster: encoder32 1-2%,
// hires16 6%, encoder16 1.5%); the plain-scatter and row-split kernels keep the
// guards (measured no faster without them).
#ifndef MSDA_BWD_FULL
#define MSDA_BWD_FULL 1
#endif
template <typename T, int V, int GG, int NN, int PAD, int FL, bool SPLIT, bool AGG>
cudaError_t bwd_launch_agg(const Params &q, const T *grad_out, const T *value, const float *loc, const float *attn,
                           const BwdBuffers &bb, cudaStream_t stream) {
    if constexpr (MSDA_BWD_FULL && PAD >= 0 && !SPLIT && (AGG || FL == (kGradLoc | kGradAttn))) {
        if (q.NLP > 0 && q.NLP % GG == 0 && q.chunks == GG * NN)
            return bwd_launch_full<T, V, GG, NN, PAD, FL, SPLIT, AGG, true>(q, grad_out, value, loc, attn, bb, stream);
    }
    return bwd_launch_full<T, V, GG, NN, PAD, FL, SPLIT, AGG, false>(q, grad_out, value, loc, attn, bb, stream);
}

template <typename T, int V, int GG, int NN, int PAD, int FL, bool SPLIT>
cudaError_t bwd_launch(const Params &p, const T *grad_out, const T *value, const float *loc, const float *attn,
                       const BwdBuffers &bb, cudaStream_t stream) {
    Params q = p;
    if (!SPLIT) q.split_log2 = 0;
    constexpr bool CAN_AGG = GG == 8 && NN == 1 && V == 4 && PAD >= 0 && !SPLIT && FL != (kGradLoc | kGradAttn);
    if constexpr (CAN_AGG) {
        if (q.aggregate) return bwd_launch_agg<T, V, GG, NN, PAD, FL, SPLIT, true>(q, grad_out, value, loc, attn, bb, stream);
    }
    return bwd_launch_agg<T, V, GG, NN, PAD, FL, SPLIT, false>(q, grad_out, value, loc, attn, bb, stream);
}

// p.flags: the outputs this launch produces (without kGradValue when the
// tile-sorted grad_value does that part).
template <typename T, int V, int GG, int NN, int PAD>
cudaError_t bwd_flags(const Params &p, const T *grad_out, const T *value, const float *loc, const float *attn,
                      const BwdBuffers &bb, cudaStream_t stream) {
    constexpr int ALL = kGradValue | kGradLoc | kGradAttn;
#define MSDA_BWD(FL, SPLIT) return bwd_launch<T, V, GG, NN, PAD, FL, SPLIT>(p, grad_out, value, loc, attn, bb, stream)
#define MSDA_BWD_S(FL)            \
    {                             \
        if (p.split_log2 > 0)     \
            MSDA_BWD(FL, true);   \
        MSDA_BWD(FL, false);      \
    }
    if constexpr (PAD < 0 || !specialised_shape(GG, NN)) {
        MSDA_BWD(-1, false);
    } else {
        if (!(p.flags & kGradValue)) MSDA_BWD_S(kGradLoc | kGradAttn);
        if (p.flags == ALL) MSDA_BWD_S(ALL);
        if (p.flags == kGradValue) MSDA_BWD_S(kGradValue);
        MSDA_BWD(-1, false);
    }
#undef MSDA_BWD_S
#undef MSDA_BWD
}

// Backward kernels for one padding specialisation, each (dtype, PAD) pair
// instantiated in its own translation unit so the library builds in parallel:
//   PAD 0 / 1: vector path, zeros / border, specialised shapes (wide shapes are
//              passed on to PAD -2);
//   PAD -2   : vector path, wide shapes, padding and outputs read at run time;
//   PAD -1   : scalar path (unaligned pointers or C_h not a multiple of 4).
template <typename T, int PAD>
cudaError_t launch_backward_pad(const Params &p, int G, int NCH, const T *grad_out, const T *value,
                                const float *loc, const float *attn, const BwdBuffers &bb, cudaStream_t stream) {
    constexpr int V = PAD == -1 ? 1 : BwdVecWidth<T>::value;
#define MSDA_BWD_CASE(GG, NN)                                                                     \
    if constexpr (reachable(GG, NN, MSDA_BWD_LANES)) {                                            \
        if (G == GG && NCH == NN) {                                                               \
            if constexpr (PAD == -1 || (PAD == -2) != specialised_shape(GG, NN))                  \
                return bwd_flags<T, V, GG, NN, PAD>(p, grad_out, value, loc, attn, bb, stream);   \
            else if constexpr (PAD >= 0)                                                          \
                return launch_backward_pad<T, -2>(p, G, NCH, grad_out, value, loc, attn, bb,      \
                                                  stream);                                        \
            else                                                                                  \
                return cudaErrorInvalidConfiguration;                                             \
        }                                                                                         \
    }
    MSDA_SHAPES(MSDA_BWD_CASE)
#undef MSDA_BWD_CASE
    return cudaErrorInvalidConfiguration;
}

// Tile-sorted grad_value, step 5: one block per chunk of a tile's samples.
template <typename T, bool VECTOR>
cudaError_t launch_tile_reduce(const Params &p, int G, int NCH, const T *grad_out, const BwdBuffers &bb,
                               cudaStream_t stream) {
    if (p.nbins == 0) return cudaSuccess;
    constexpr int V = VECTOR ? BwdVecWidth<T>::value : 1;
    // chunks <= tiles + samples / kChunk (a tile's last chunk may be partial)
    const uint64_t blocks = (uint64_t)p.nbins + ((uint64_t)p.rows * p.NLP) / kChunk + 1;
#define MSDA_RED_CASE(GG, NN)                                                                     \
    if constexpr (reachable(GG, NN, MSDA_BWD_LANES)) {                                            \
        if (G == GG && NCH == NN) {                                                               \
            auto kernel = msda_tile_reduce_kernel<T, V, GG, NN>;                                  \
            const cudaError_t e =                                                                 \
                cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTileReduceSmem); \
            if (e != cudaSuccess) return e;                                                       \
            kernel<<<(unsigned)blocks, 256, kTileReduceSmem, stream>>>(p, grad_out, bb.offsets, bb.chunks, \
                                                                       bb.entries, bb.gv_acc);   \
            return cudaGetLastError();                                                            \
        }                                                                                         \
    }
    MSDA_SHAPES(MSDA_RED_CASE)
#undef MSDA_RED_CASE
    return cudaErrorInvalidConfiguration;
}

}  // namespace msda
