// msda_staged.cuh -- the forward with staged coarse levels.
//
// The direct forward gathers every corner row through L1.  Here each block
// serves a run of queries of one (b, h) and first copies the whole coarsest
// levels of that head (as many as fit a shared-memory budget) into shared
// memory with TMA tensor copies; samples on those levels gather from shared
// memory, samples on the finer levels from global memory as before.  A coarse
// level is small and hot (encoder32: level 3 of one head is 273 pixels, read
// by about 30 corner lookups per pixel within one block), so the copy is paid
// once per block and the gathers on it no longer depend on L1 hits.  The
// arithmetic (cell, weights, order of the products and sums) is that of
// msda_forward_kernel, so the two give bit-identical outputs.
#pragma once

#include <cuda.h>

#include "msda_kernels.cuh"

namespace msda {

#ifndef MSDA_STAGED_MIN_BLOCKS
#define MSDA_STAGED_MIN_BLOCKS 3  // 85 registers: the direct kernel's loop plus the staging state
#endif

constexpr int kStageBox = 32;                  // pixels per TMA box
constexpr uint32_t kStageWaitLimit = 1u << 22;  // mbarrier polls before the block gives up on the copy

// Staged levels ls..N_l-1 of one head: pixel i of level l sits at shared
// pixel sp[l] + i (each level's region a whole number of boxes), C_h elements
// per pixel.  The grid is B*N_h*bpb blocks; block k of (b, h) serves queries
// [k*rpb, min(N_q, (k+1)*rpb)).
struct StagePlan {
    int ls;    // first staged level (N_l: none)
    int bpb;   // blocks per (b, h)
    int rpb;   // queries per block
    int boxes; // TMA boxes per block
    uint32_t bytes;  // bytes the boxes bring (the mbarrier's transaction count)
    int layout;      // 0: value (B, L, N_h, C_h); 1: (B, N_h, L, C_h) -- the tensor map's dimension order
    int rot;         // backward: channel-chunk rotation mask of the shared accumulator (0: none)
    int sp[kMaxLevels];
};

template <typename T, int VEC> struct ShIO;
template <> struct ShIO<float, 4> {
    static __device__ __forceinline__ void load(uint32_t a, float (&o)[4]) {
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(o[0]), "=f"(o[1]), "=f"(o[2]), "=f"(o[3])
                     : "r"(a));
    }
};
template <> struct ShIO<__nv_bfloat16, 4> {
    static __device__ __forceinline__ void load(uint32_t a, float (&o)[4]) {
        uint32_t x, y;
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(x), "=r"(y) : "r"(a));
        o[0] = __uint_as_float(x << 16);
        o[1] = __uint_as_float(x & 0xffff0000u);
        o[2] = __uint_as_float(y << 16);
        o[3] = __uint_as_float(y & 0xffff0000u);
    }
};

__device__ __forceinline__ bool stage_wait(uint32_t bar, uint32_t phase) {
    for (uint32_t it = 0; it < kStageWaitLimit; ++it) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(bar), "r"(phase)
            : "memory");
        if (done) return true;
    }
    return false;
}

// One block: stage, then the forward of its queries (the direct kernel's
// loop -- cell records in shared memory, the next batch's locations loaded
// ahead -- binary32 weights, specialised padding).  A block whose copy has not
// landed after kStageWaitLimit polls counts itself in timeouts[0] and gathers
// every level from global memory (same results), then waits for the copy
// again (bounded) before it exits, counting itself in timeouts[1] if that
// wait runs out too.
template <typename T, int VEC, int G, int NCH, int PAD>
__global__ void __launch_bounds__(kThreads, MSDA_STAGED_MIN_BLOCKS)
msda_forward_staged_kernel(const __grid_constant__ Params p, const __grid_constant__ StagePlan sp,
                           const __grid_constant__ CUtensorMap tmap, const T *__restrict__ value,
                           const float *__restrict__ loc, const float *__restrict__ attn, T *__restrict__ out,
                           unsigned int *__restrict__ timeouts) {
    // dynamic shared memory: the staged pixels, from a 128-byte boundary (128 bytes of slack allocated)
    extern __shared__ __align__(128) unsigned char stage_raw[];
    __shared__ __align__(8) uint64_t bar_mem;
    __shared__ LevelTables lt;
    __shared__ int sps[kMaxLevels];
    __shared__ int4 rec_o[kThreads];
    __shared__ float4 rec_w[kThreads];
    if (threadIdx.x < (unsigned)p.N_l) sps[threadIdx.x] = sp.sp[threadIdx.x];
    load_level_tables(p, lt);  // (ends with __syncthreads)

    const uint32_t bh = blockIdx.x / (uint32_t)sp.bpb;
    const int q0 = (int)(blockIdx.x - bh * (uint32_t)sp.bpb) * sp.rpb;
    const int q1 = min(p.N_q, q0 + sp.rpb);
    if (q0 >= q1) return;  // uniform over the block
    const uint32_t b = p.div_h.div(bh), h = bh - b * (uint32_t)p.N_h;

    // stage: one thread arms the barrier with the boxes' bytes and issues them
    const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&bar_mem);
    const uint32_t sbase = ((uint32_t)__cvta_generic_to_shared(stage_raw) + 127u) & ~127u;
    const bool staging = sp.ls < p.N_l;
    if (staging && threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(1) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(sp.bytes) : "memory");
        const uint32_t box_bytes = (uint32_t)(kStageBox * p.C_h * (int)sizeof(T));
        for (int l = sp.ls; l < p.N_l; ++l) {
            const int npx = lt.H[l] * lt.W[l];
            for (int i = 0; i * kStageBox < npx; ++i) {
                const int px = lt.start[l] + i * kStageBox;  // first pixel of the box
                const uint32_t dst = sbase + (uint32_t)(sps[l] + i * kStageBox) * (box_bytes / kStageBox);
                // coordinates, innermost first: (channel, head, pixel, batch) or (channel, pixel, head, batch)
                const int c1 = sp.layout == 0 ? (int)h : px, c2 = sp.layout == 0 ? px : (int)h;
                asm volatile(
                    "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                    " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
                    "l"(reinterpret_cast<uint64_t>(&tmap)), "r"(0), "r"(c1), "r"(c2), "r"((int)b), "r"(bar)
                    : "memory");
            }
        }
    }
    __syncthreads();  // the barrier is initialised before anyone polls it
    const bool landed = staging ? stage_wait(bar, 0) : true;
    const bool ok = __syncthreads_and(landed);
    if (staging && !ok && threadIdx.x == 0) atomicAdd(timeouts, 1u);  // counted for msda_staged_timeouts()
    const int lsj = (ok ? sp.ls : p.N_l) * p.N_p;  // samples j >= lsj gather from shared memory

    constexpr int GPB = kThreads / G;
    const int lane = threadIdx.x & 31;
    const int r = lane & (G - 1);
    const int base = lane & ~(G - 1);
    const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << base);
    const int sP = p.v_sP, sJ = p.l_sJ, sXY = p.l_sXY, NLP = p.NLP, C = p.C_h;
    int nk = 0;
#pragma unroll
    for (int k = 0; k < NCH; ++k) nk += (k * G + r < p.chunks);
    const T *vbh = value + b * p.v_sB + (int64_t)h * p.v_sH + r * VEC;
    const uint32_t sbr = sbase + (uint32_t)(r * VEC * (int)sizeof(T));  // this lane's channels of shared pixel 0
    int4 *wo = rec_o + (threadIdx.x & ~31);  // the warp's cell records, as in the direct kernel
    float4 *ww = rec_w + (threadIdx.x & ~31);
    const int mypos = rec_pos<G>(lane / G, r);

    // items as in the direct kernel: part `part` of query q takes its batches part, part + S, ...
    const int jstep = G << p.split_log2;
    for (int item = (q0 << p.split_log2) + (int)threadIdx.x / G; item < (q1 << p.split_log2); item += GPB) {
        const int q = item >> p.split_log2;
        const int part = item & ((1 << p.split_log2) - 1);
        const uint32_t bqh = (b * (uint32_t)p.N_q + (uint32_t)q) * (uint32_t)p.N_h + h;
        const int64_t lo = b * p.l_sB + (int64_t)(((uint32_t)q * (uint32_t)p.N_h + h) * (uint32_t)NLP) * sJ;
        const int64_t ao = (int64_t)bqh * NLP;
        float acc[NCH][VEC];
#pragma unroll
        for (int k = 0; k < NCH; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[k][e] = 0.0f;

        // the next batch's location and weight are loaded before this batch is consumed
        float nu = 0.0f, nv = 0.0f, nA = 0.0f;
        {
            const int jf = part * G + r;
            if (jf < NLP) {
                nu = ldl(loc, lo + jf * sJ, 0);
                nv = ldl(loc, lo + jf * sJ + sXY, 0);
                nA = ldl(attn, ao + jf, 0);
            }
        }
        for (int j0 = part * G; j0 < NLP; j0 += jstep) {
            // owner phase: the sample's record; staged samples get offsets into
            // shared memory (pixel stride C_h), the others into value
            const int j = j0 + r;
            const float u = nu, v = nv, A = nA;
            {
                const int jn = j + jstep;
                if (jn < NLP) {
                    nu = ldl(loc, lo + jn * sJ, 0);
                    nv = ldl(loc, lo + jn * sJ + sXY, 0);
                    nA = ldl(attn, ao + jn, 0);
                }
            }
            if (j < NLP) {
                const int l = (int)p.div_p.div((uint32_t)j);
                const int W = lt.W[l], H = lt.H[l];
                const Cell c = make_cell<PAD>(u, v, lt.sx[l], lt.sy[l], p.off, W, H, p.padding);
                const Corners cr =
                    j >= lsj ? corners_of(c, A, W, H, sps[l], C) : corners_of(c, A, W, H, lt.start[l], sP);
                wo[mypos] = make_int4(cr.o[0], cr.o[1], cr.o[2], cr.o[3]);
                ww[mypos] = make_float4(cr.w[0], cr.w[1], cr.w[2], cr.w[3]);
            } else {  // past the row's last sample: weight 0 at value offset 0
                wo[mypos] = make_int4(0, 0, 0, 0);
                ww[mypos] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
            __syncwarp(gmask);
            const int ns = min(G, NLP - j0);
            constexpr int S2 = (G >= 2 && NCH * VEC <= 4) ? 2 : 1;  // two samples in flight for one chunk a lane
#pragma unroll
            for (int s = 0; s < G; s += S2) {
                if (s < ns) {
                    int o[S2][4];
                    float w[S2][4];
                    float x[S2][4][NCH][VEC];
#pragma unroll
                    for (int h2 = 0; h2 < S2; ++h2) {
                        const int qp = rec_pos<G>(lane / G, s + h2);
                        const int4 o4 = wo[qp];
                        const float4 w4 = ww[qp];
                        o[h2][0] = o4.x;
                        o[h2][1] = o4.y;
                        o[h2][2] = o4.z;
                        o[h2][3] = o4.w;
                        w[h2][0] = w4.x;
                        w[h2][1] = w4.y;
                        w[h2][2] = w4.z;
                        w[h2][3] = w4.w;
                        // the same for every lane of the warp; a sample past the row's last
                        // (weight 0, offset 0) reads global memory, as in the direct kernel
                        const bool st = j0 + s + h2 >= lsj && j0 + s + h2 < NLP;
                        if (st) {
#pragma unroll
                            for (int i = 0; i < 4; ++i)
#pragma unroll
                                for (int k = 0; k < NCH; ++k)
                                    if (k < nk)
                                        ShIO<T, VEC>::load(sbr + (uint32_t)(o[h2][i] + k * G * VEC) * (uint32_t)sizeof(T),
                                                           x[h2][i][k]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 4; ++i)
#pragma unroll
                                for (int k = 0; k < NCH; ++k)
                                    if (k < nk) VecIO<T, VEC>::load(vbh + o[h2][i] + k * G * VEC, x[h2][i][k]);
                        }
                    }
#pragma unroll
                    for (int h2 = 0; h2 < S2; ++h2)
#pragma unroll
                        for (int i = 0; i < 4; ++i)
#pragma unroll
                            for (int k = 0; k < NCH; ++k)
                                if (k < nk) axpy<VEC>(acc[k], w[h2][i], x[h2][i][k]);
                }
            }
            __syncwarp(gmask);  // records are rewritten by the next batch
        }
        sum_parts<G, NCH, VEC>(acc, p.split_log2, lane);
        T *dst = out + (int64_t)bqh * C + r * VEC;
        if (part == 0) {
#pragma unroll
            for (int k = 0; k < NCH; ++k)
                if (k < nk) VecIO<T, VEC>::store(dst + k * G * VEC, acc[k]);
        }
    }
    // a copy that had not landed must not write into shared memory the next
    // block owns: wait for it again (bounded); if it still has not landed, the
    // block exits with the copy in flight and counts itself in timeouts[1]
    // (msda_staged_timeouts then reports MSDA_ERR_STAGE_COPY)
    if (staging && !ok) {
        const bool landed_late = __syncthreads_and(stage_wait(bar, 0));
        if (!landed_late && threadIdx.x == 0) atomicAdd(timeouts + 1, 1u);
    }
}

// ---------------------------------------------------------------- staged backward
// The backward with a per-level shared-memory grad_value accumulator (the
// alternative to direct atomics for the coarse levels): each block serves a
// run of queries of one (b, h) and keeps a binary32 accumulator for the
// staged levels of that head in shared memory.  Samples on those levels add
// their four corner contributions there (red.shared.add.f32), samples on
// finer levels straight into the global accumulator as in
// msda_backward_kernel; at the end the block adds its shared rows into the
// global accumulator (red.global.add.v4.f32, rows that stayed zero skipped).
// grad_sampling_locations and grad_attention_weights are the direct kernel's
// (the same record exchange, gathers and reductions), so they are
// bit-identical to msda_backward's.  Channel chunk c of staged pixel x sits
// at chunk (c + (x & rot)) & (chunks - 1) of the pixel's row (chunks a power
// of two; rot = 0 otherwise), so that the groups of a warp, usually on
// different pixels, spread over the banks.
__device__ __forceinline__ void red_shared_add(uint32_t a, float v) {
    asm volatile("red.shared.add.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

template <typename T, int VEC, int G, int NCH, int PAD>
__global__ void __launch_bounds__(kThreads, NCH == 1 ? MSDA_BWD_MIN_BLOCKS : 2)
msda_backward_staged_kernel(const __grid_constant__ Params p, const __grid_constant__ StagePlan sp,
                            const T *__restrict__ grad_out, const T *__restrict__ value,
                            const float *__restrict__ loc, const float *__restrict__ attn,
                            float *__restrict__ gv_acc, float *__restrict__ grad_loc, float *__restrict__ grad_attn) {
    extern __shared__ __align__(16) float acc_s[];  // staged pixels x C_h, binary32
    __shared__ LevelTables lt;
    __shared__ int4 rec_o[kThreads];
    __shared__ float4 rec_w[kThreads];
    __shared__ int4 rec_s[kThreads];  // staged samples: the corners' staged pixel indices
    __shared__ int sps[kMaxLevels];
    if (threadIdx.x < (unsigned)p.N_l) sps[threadIdx.x] = sp.sp[threadIdx.x];
    load_level_tables(p, lt);

    const uint32_t bh = blockIdx.x / (uint32_t)sp.bpb;
    const int q0 = (int)(blockIdx.x - bh * (uint32_t)sp.bpb) * sp.rpb;
    const int q1 = min(p.N_q, q0 + sp.rpb);
    if (q0 >= q1) return;  // uniform over the block
    const uint32_t b = p.div_h.div(bh), h = bh - b * (uint32_t)p.N_h;
    const int C = p.C_h, npix = sp.boxes * kStageBox;
    for (int i = threadIdx.x; i < npix * C; i += kThreads) acc_s[i] = 0.0f;
    __syncthreads();

    constexpr int GPB = kThreads / G;
    const int flags = p.flags;
    const bool want_gl = flags & kGradLoc, want_ga = flags & kGradAttn;
    const bool need_v = want_gl || want_ga;
    const int lane = threadIdx.x & 31;
    const int r = lane & (G - 1);
    const int grp = lane / G;
    const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane & ~(G - 1)));
    int4 *wo = rec_o + (threadIdx.x & ~31);
    float4 *ww = rec_w + (threadIdx.x & ~31);
    int4 *wsx = rec_s + (threadIdx.x & ~31);
    const int mypos = rec_pos<G>(grp, r);
    const int sP = p.v_sP, sJ = p.l_sJ, sXY = p.l_sXY, NLP = p.NLP;
    const int lsj = sp.ls * p.N_p;  // samples j >= lsj accumulate in shared memory
    int nk = 0;
#pragma unroll
    for (int k = 0; k < NCH; ++k) nk += (k * G + r < p.chunks);
    const int64_t bhoff = b * p.v_sB + (int64_t)h * p.v_sH;
    const T *vbh = value + bhoff + r * VEC;
    float *gbh = gv_acc + bhoff + r * VEC;
    const uint32_t sacc = (uint32_t)__cvta_generic_to_shared(acc_s);

    for (int q = q0 + (int)threadIdx.x / G; q < q1; q += GPB) {
        const uint32_t bqh = (b * (uint32_t)p.N_q + (uint32_t)q) * (uint32_t)p.N_h + h;
        const int64_t lrow = b * p.l_sB + (int64_t)(((uint32_t)q * (uint32_t)p.N_h + h) * (uint32_t)NLP) * sJ;
        const int64_t ao = (int64_t)bqh * NLP;
        float g[NCH][VEC];
        {
            const T *src = grad_out + (int64_t)bqh * C + r * VEC;
#pragma unroll
            for (int k = 0; k < NCH; ++k) {
                if (k < nk) {
                    VecIO<T, VEC>::load(src + k * G * VEC, g[k]);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) g[k][e] = 0.0f;
                }
            }
        }
        for (int j0 = 0; j0 < NLP; j0 += G) {
            const int j = j0 + r;
            const bool live = j < NLP;
            int l = 0;
            float A = 0.0f;
            Cell c;
            {
                Corners cr = {{0, 0, 0, 0}, {0.0f, 0.0f, 0.0f, 0.0f}};
                float u = 0.0f, v = 0.0f;
                if (live) {
                    l = (int)p.div_p.div((uint32_t)j);
                    u = ldl(loc, lrow + j * sJ, p.loc_dt);
                    v = ldl(loc, lrow + j * sJ + sXY, p.loc_dt);
                    A = ldl(attn, ao + j, p.loc_dt);
                }
                const int W = lt.W[l], H = lt.H[l];
                c = make_cell<PAD>(u, v, lt.sx[l], lt.sy[l], p.off, W, H, p.padding);
                if (live) cr = corners_of(c, A, W, H, lt.start[l], sP);
                wo[mypos] = make_int4(cr.o[0], cr.o[1], cr.o[2], cr.o[3]);
                ww[mypos] = make_float4(cr.w[0], cr.w[1], cr.w[2], cr.w[3]);
                if (live && j >= lsj) {  // the same corners as staged pixel indices (stride 1)
                    const Corners cs = corners_of(c, A, W, H, sps[l], 1);
                    wsx[mypos] = make_int4(cs.o[0], cs.o[1], cs.o[2], cs.o[3]);
                }
            }
            __syncwarp(gmask);
            const int ns = min(G, NLP - j0);
            float pd[4][G <= 8 ? G : 1];
            float dt[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int s = 0; s < G; ++s) {
                float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                if (s < ns) {
                    const int qp = rec_pos<G>(grp, s);
                    const int4 o4 = wo[qp];
                    const int oo[4] = {o4.x, o4.y, o4.z, o4.w};
                    if (need_v) {
                        float x[4][NCH][VEC];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
#pragma unroll
                            for (int k = 0; k < NCH; ++k)
                                if (k < nk) VecIO<T, VEC>::load(vbh + oo[i] + k * G * VEC, x[i][k]);
                        // the direct kernel's summation: even / odd channel partial sums, chunk by chunk
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            float2 dp = make_float2(0.0f, 0.0f);
#pragma unroll
                            for (int k = 0; k < NCH; ++k)
                                if (k < nk) dot_acc<VEC>(dp, g[k], x[i][k]);
                            d[i] = dp.x + dp.y;
                        }
                    }
                    const float4 w4 = ww[qp];
                    const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
                    if (j0 + s >= lsj) {  // staged level (the same for every lane of the warp)
                        const int4 s4 = wsx[qp];
                        const int px[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (wv[i] != 0.0f)
#pragma unroll
                                for (int k = 0; k < NCH; ++k)
                                    if (k < nk) {
                                        const int ck = ((k * G + r) + (px[i] & sp.rot)) & (p.chunks - 1);
                                        const int cc = sp.rot ? ck : k * G + r;
                                        const uint32_t a = sacc + (uint32_t)((px[i] * C + cc * VEC) * 4);
#pragma unroll
                                        for (int e = 0; e < VEC; ++e) red_shared_add(a + 4 * e, wv[i] * g[k][e]);
                                    }
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (wv[i] != 0.0f)
#pragma unroll
                                for (int k = 0; k < NCH; ++k)
                                    if (k < nk) RedIO<VEC>::add(gbh + oo[i] + k * G * VEC, g[k], wv[i]);
                    }
                }
                if constexpr (G <= 8) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) pd[i][s] = d[i];
                } else if (need_v) {
#pragma unroll
                    for (int o = 1; o < G; o <<= 1)
#pragma unroll
                        for (int i = 0; i < 4; ++i) d[i] += __shfl_xor_sync(gmask, d[i], o);
                    if (r == s) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) dt[i] = d[i];
                    }
                }
            }
            __syncwarp(gmask);
            if (need_v) {
                if constexpr (G <= 8) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) dt[i] = reduce_scatter<G>(pd[i], r, gmask);
                }
                if (live) {
                    const float gx = 1.0f - c.fx, gy = 1.0f - c.fy;
                    const float w[4] = {gx * gy, c.fx * gy, gx * c.fy, c.fx * c.fy};
                    const float dwx[4] = {-gy, gy, -c.fy, c.fy};
                    const float dwy[4] = {-gx, -c.fx, gx, c.fx};
                    float ga = 0.0f, tx = 0.0f, ty = 0.0f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float di = (c.valid & (1u << i)) ? dt[i] : 0.0f;
                        ga = fmaf(w[i], di, ga);
                        tx = fmaf(dwx[i], di, tx);
                        ty = fmaf(dwy[i], di, ty);
                    }
                    if (want_ga) stl(grad_attn, ao + j, ga, p.loc_dt);
                    if (want_gl) {
                        stl(grad_loc, lrow + j * sJ, A * tx * (lt.sx[l] * c.kx), p.loc_dt);
                        stl(grad_loc, lrow + j * sJ + sXY, A * ty * (lt.sy[l] * c.ky), p.loc_dt);
                    }
                }
            }
        }
    }
    // flush: each group adds staged pixels' rows into the global accumulator
    __syncthreads();
    for (int l = sp.ls; l < p.N_l; ++l) {
        const int n = lt.H[l] * lt.W[l];
        for (int pl = (int)threadIdx.x / G; pl < n; pl += GPB) {
            const int px = sps[l] + pl;
#pragma unroll
            for (int k = 0; k < NCH; ++k)
                if (k < nk) {
                    const int ck = ((k * G + r) + (px & sp.rot)) & (p.chunks - 1);
                    const int cc = sp.rot ? ck : k * G + r;
                    float v[VEC];
                    bool any = false;
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        v[e] = acc_s[px * C + cc * VEC + e];
                        any |= v[e] != 0.0f;
                    }
                    if (any) RedIO<VEC>::add_sum(gbh + (lt.start[l] + pl) * sP + k * G * VEC, v);
                }
        }
    }
}

// Host side (msda_staged_{f32,bf16}.cu): pick the kernel for (G, NCH,
// padding), size the grid (blocks per (b, h) from the occupancy at `smem`
// bytes) and launch.
template <typename T>
cudaError_t launch_forward_staged(const Params &p, StagePlan sp, const CUtensorMap &tmap, size_t smem, int G, int NCH,
                                  const T *value, const float *loc, const float *attn, T *out,
                                  unsigned int *timeouts, cudaStream_t stream);
template <typename T>
cudaError_t launch_backward_staged(const Params &p, StagePlan sp, size_t smem, int G, int NCH, const T *grad_out,
                                   const T *value, const float *loc, const float *attn, float *gv_acc,
                                   float *grad_loc, float *grad_attn, cudaStream_t stream);

}  // namespace msda
