// msda_kernels.cuh -- sm_103a kernels for multi-scale deformable attention.
//
// Operation ("MS Deformable Attention Kernel API Reference", Background,
// Parameters, Returns; "MS Deformable Attention Backward Kernel API
// Reference", Background, Returns, Notes): every (batch b, query q, head h)
// row samples N_l pyramid levels at N_p learned normalised locations each,
// interpolates the head-h value map bilinearly (align_corners mapping, zeros
// or border padding), weights each sample by its attention weight and sums
// into out[b, q, h*C_h : (h+1)*C_h].  The backward recomputes the same
// bilinear cells and produces grad_value (scatter-add), the location gradient
// and the attention-weight gradient.
//
// Work decomposition (both directions): one warp per row.  A row's
// N_l*N_p samples are processed S = 32/G at a time: lanes form S groups of G
// lanes, each group owns one sample, and inside a group every lane owns
// VEC*NCH channels (128-bit loads when C_h allows).  The value map is read
// through the read-only path and is meant to stay L1/L2 resident; nothing is
// staged in shared memory.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace msda {

constexpr int kMaxLevels = 16;
constexpr int kThreads = 256;  // 8 warps per block, one row per warp

// Everything a kernel needs, passed by value (kernel parameter space).
struct Params {
    uint32_t rows;      // B * N_q * N_h
    int N_q, N_h, C_h, NLP;  // NLP = N_l * N_p
    uint64_t np_div;    // floor(j / N_p) = (j * np_div) >> 32, np_div = ceil(2^32 / N_p)
    int chunks;         // vector chunks per channel row: C_h / VEC
    int row_order_bhq;  // 1: row = (b*N_h + h)*N_q + q; 0: row = (b*N_q + q)*N_h + h
    int padding;        // 0 zeros, 1 border
    // value (and grad_value / accumulator) element strides
    int64_t v_sB;
    int v_sH, v_sP;
    // sampling_locations (and its gradient) element strides: batch, sample, x->y
    int64_t l_sB;
    int l_sJ, l_sXY;
    // per level
    int H[kMaxLevels], W[kMaxLevels], start[kMaxLevels];
    float sx[kMaxLevels], sy[kMaxLevels];  // pixels per unit of normalised coordinate
    float off;                             // -0.5 (align_corners = 0) or 0 (align_corners = 1)
};

// ---------------------------------------------------------------- element access
template <typename T, int VEC> struct VecIO;

template <> struct VecIO<float, 4> {
    static __device__ __forceinline__ void load(const float *p, float (&o)[4]) {
        const float4 x = __ldg(reinterpret_cast<const float4 *>(p));
        o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w;
    }
    static __device__ __forceinline__ void store(float *p, const float (&o)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(o[0], o[1], o[2], o[3]);
    }
};

template <> struct VecIO<float, 1> {
    static __device__ __forceinline__ void load(const float *p, float (&o)[1]) { o[0] = __ldg(p); }
    static __device__ __forceinline__ void store(float *p, const float (&o)[1]) { *p = o[0]; }
};

template <> struct VecIO<__nv_bfloat16, 8> {
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float (&o)[8]) {
        const uint4 x = __ldg(reinterpret_cast<const uint4 *>(p));
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // bf16 -> f32 is exact: the bits move up 16 places
            o[2 * i] = __uint_as_float(w[i] << 16);
            o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float (&o)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 t = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t *>(&t);
        }
        *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

template <> struct VecIO<__nv_bfloat16, 1> {
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float (&o)[1]) {
        o[0] = __bfloat162float(__ldg(p));
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float (&o)[1]) {
        *p = __float2bfloat16_rn(o[0]);
    }
};

// Fire-and-forget binary32 atomic adds in L2 (no return value).
__device__ __forceinline__ void red_add(float *p, float a) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(a) : "memory");
}
__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

template <int VEC> struct RedIO;
template <> struct RedIO<1> {
    static __device__ __forceinline__ void add(float *p, const float (&v)[1], float s) { red_add(p, s * v[0]); }
};
template <> struct RedIO<4> {
    static __device__ __forceinline__ void add(float *p, const float (&v)[4], float s) {
        red_add_v4(p, s * v[0], s * v[1], s * v[2], s * v[3]);
    }
};
template <> struct RedIO<8> {
    static __device__ __forceinline__ void add(float *p, const float (&v)[8], float s) {
        red_add_v4(p, s * v[0], s * v[1], s * v[2], s * v[3]);
        red_add_v4(p + 4, s * v[4], s * v[5], s * v[6], s * v[7]);
    }
};

// ---------------------------------------------------------------- row / sample geometry
struct Row {
    int b, q, h;
    uint32_t bqh;  // (b*N_q + q)*N_h + h: row of out / grad_output / attention_weights
};

__device__ __forceinline__ Row decode_row(const Params &p, uint32_t row) {
    Row r;
    if (p.row_order_bhq) {
        const uint32_t t = row / (uint32_t)p.N_q;
        r.q = (int)(row - t * (uint32_t)p.N_q);
        r.b = (int)(t / (uint32_t)p.N_h);
        r.h = (int)(t - (uint32_t)r.b * (uint32_t)p.N_h);
    } else {
        const uint32_t t = row / (uint32_t)p.N_h;
        r.h = (int)(row - t * (uint32_t)p.N_h);
        r.b = (int)(t / (uint32_t)p.N_q);
        r.q = (int)(t - (uint32_t)r.b * (uint32_t)p.N_q);
    }
    r.bqh = ((uint32_t)r.b * (uint32_t)p.N_q + (uint32_t)r.q) * (uint32_t)p.N_h + (uint32_t)r.h;
    return r;
}

__device__ __forceinline__ int level_of(const Params &p, int j) {
    return (int)(((uint64_t)(uint32_t)j * p.np_div) >> 32);
}

// The bilinear cell of one sample on level l: element offsets (relative to
// the (b, h) value slice) of the four corners (y0,x0), (y0,x0+1),
// (y0+1,x0), (y0+1,x0+1), their weights, which of them read the map, and
// the fractional position.
struct Cell {
    int off[4];
    float w[4];
    float fx, fy;
    unsigned valid;  // bit i: corner i reads the map
};

__device__ __forceinline__ Cell make_cell(const Params &p, int l, float u, float v) {
    Cell c;
    const int H = p.H[l], W = p.W[l];
    // Pixel coordinate with one rounding (align_corners mapping).
    float x = __fmaf_rn(u, p.sx[l], p.off);
    float y = __fmaf_rn(v, p.sy[l], p.off);
    // Clamping to [-2, size+1] changes no result: every corner of a cell
    // beyond it lies outside the map ("zeros") or clamps onto the same edge
    // pixel ("border"); it keeps the integer conversion in range.
    x = fminf(fmaxf(x, -2.0f), (float)W + 1.0f);
    y = fminf(fmaxf(y, -2.0f), (float)H + 1.0f);
    const float x0f = floorf(x), y0f = floorf(y);
    c.fx = x - x0f;
    c.fy = y - y0f;
    int x0 = (int)x0f, y0 = (int)y0f, x1 = x0 + 1, y1 = y0 + 1;
    const float gx = 1.0f - c.fx, gy = 1.0f - c.fy;
    c.w[0] = gx * gy;
    c.w[1] = c.fx * gy;
    c.w[2] = gx * c.fy;
    c.w[3] = c.fx * c.fy;
    if (p.padding == 0) {
        const bool ix0 = (unsigned)x0 < (unsigned)W, ix1 = (unsigned)x1 < (unsigned)W;
        const bool iy0 = (unsigned)y0 < (unsigned)H, iy1 = (unsigned)y1 < (unsigned)H;
        c.valid = (unsigned)(ix0 && iy0) | ((unsigned)(ix1 && iy0) << 1) | ((unsigned)(ix0 && iy1) << 2) |
                  ((unsigned)(ix1 && iy1) << 3);
    } else {
        c.valid = 0xfu;
    }
    // Addresses are formed only from clamped indices.
    x0 = min(max(x0, 0), W - 1);
    x1 = min(max(x1, 0), W - 1);
    y0 = min(max(y0, 0), H - 1);
    y1 = min(max(y1, 0), H - 1);
    const int r0 = p.start[l] + y0 * W, r1 = p.start[l] + y1 * W;
    c.off[0] = (r0 + x0) * p.v_sP;
    c.off[1] = (r0 + x1) * p.v_sP;
    c.off[2] = (r1 + x0) * p.v_sP;
    c.off[3] = (r1 + x1) * p.v_sP;
    return c;
}

// ---------------------------------------------------------------- forward
template <typename T, int VEC, int G, int NCH>
__global__ void __launch_bounds__(kThreads)
msda_forward_kernel(const Params p, const T *__restrict__ value, const float *__restrict__ loc,
                    const float *__restrict__ attn, T *__restrict__ out) {
    constexpr int S = 32 / G;
    const int lane = threadIdx.x & 31, grp = lane / G, r = lane % G;
    const uint32_t row = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (row >= p.rows) return;  // the whole warp leaves together
    const Row rw = decode_row(p, row);
    const T *vbh = value + rw.b * p.v_sB + (int64_t)rw.h * p.v_sH;
    const float *lrow = loc + rw.b * p.l_sB +
                        (int64_t)(((uint32_t)rw.q * (uint32_t)p.N_h + (uint32_t)rw.h) * (uint32_t)p.NLP) * p.l_sJ;
    const float *arow = attn + (int64_t)rw.bqh * p.NLP;

    float acc[NCH][VEC];
#pragma unroll
    for (int k = 0; k < NCH; ++k)
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[k][e] = 0.0f;

    for (int j = grp; j < p.NLP; j += S) {
        const int l = level_of(p, j);
        const float A = __ldg(arow + j);
        const float u = __ldg(lrow + j * p.l_sJ), v = __ldg(lrow + j * p.l_sJ + p.l_sXY);
        const Cell c = make_cell(p, l, u, v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (c.valid & (1u << i)) {
                const float aw = A * c.w[i];
                const T *src = vbh + c.off[i];
#pragma unroll
                for (int k = 0; k < NCH; ++k) {
                    const int kc = k * G + r;
                    if (kc < p.chunks) {
                        float x[VEC];
                        VecIO<T, VEC>::load(src + kc * VEC, x);
#pragma unroll
                        for (int e = 0; e < VEC; ++e) acc[k][e] = fmaf(aw, x[e], acc[k][e]);
                    }
                }
            }
        }
    }
    // Sum the S groups' partial rows.
#pragma unroll
    for (int o = G; o < 32; o <<= 1)
#pragma unroll
        for (int k = 0; k < NCH; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[k][e] += __shfl_xor_sync(0xffffffffu, acc[k][e], o);
    if (grp == 0) {
        T *dst = out + (int64_t)rw.bqh * p.C_h;
#pragma unroll
        for (int k = 0; k < NCH; ++k) {
            const int kc = k * G + r;
            if (kc < p.chunks) VecIO<T, VEC>::store(dst + kc * VEC, acc[k]);
        }
    }
}

// ---------------------------------------------------------------- backward
enum : int { kGradValue = 1, kGradLoc = 2, kGradAttn = 4 };

template <typename T, int VEC, int G, int NCH>
__global__ void __launch_bounds__(kThreads)
msda_backward_kernel(const Params p, const T *__restrict__ grad_out, const T *__restrict__ value,
                     const float *__restrict__ loc, const float *__restrict__ attn,
                     float *__restrict__ gv_acc, float *__restrict__ grad_loc,
                     float *__restrict__ grad_attn, const int flags) {
    constexpr int S = 32 / G;
    const int lane = threadIdx.x & 31, grp = lane / G, r = lane % G;
    const uint32_t row = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (row >= p.rows) return;  // the whole warp leaves together
    const bool want_gv = flags & kGradValue, want_gl = flags & kGradLoc, want_ga = flags & kGradAttn;
    const bool need_v = want_gl || want_ga;  // value is read only for these two
    const bool need_a = want_gv || want_gl;  // attention is read only for these two

    const Row rw = decode_row(p, row);
    const int64_t bh = rw.b * p.v_sB + (int64_t)rw.h * p.v_sH;
    const T *vbh = value + bh;
    float *gbh = gv_acc + bh;
    const int64_t lrow = rw.b * p.l_sB +
                         (int64_t)(((uint32_t)rw.q * (uint32_t)p.N_h + (uint32_t)rw.h) * (uint32_t)p.NLP) * p.l_sJ;
    const float *arow = attn + (int64_t)rw.bqh * p.NLP;

    float g[NCH][VEC];
    {
        const T *src = grad_out + (int64_t)rw.bqh * p.C_h;
#pragma unroll
        for (int k = 0; k < NCH; ++k) {
            const int kc = k * G + r;
            if (kc < p.chunks) {
                VecIO<T, VEC>::load(src + kc * VEC, g[k]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) g[k][e] = 0.0f;
            }
        }
    }

    for (int j0 = 0; j0 < p.NLP; j0 += S) {  // uniform trip count: shuffles below need all lanes
        const int j = j0 + grp;
        const bool active = j < p.NLP;
        float dA = 0.0f, dX = 0.0f, dY = 0.0f, A = 0.0f;
        int l = 0;
        if (active) {
            l = level_of(p, j);
            if (need_a) A = __ldg(arow + j);
            const float u = __ldg(loc + lrow + j * p.l_sJ), v = __ldg(loc + lrow + j * p.l_sJ + p.l_sXY);
            const Cell c = make_cell(p, l, u, v);
            if (need_v) {
                // d[i] = this lane's part of <g, value(corner i)>
                float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (c.valid & (1u << i)) {
                        const T *src = vbh + c.off[i];
#pragma unroll
                        for (int k = 0; k < NCH; ++k) {
                            const int kc = k * G + r;
                            if (kc < p.chunks) {
                                float x[VEC];
                                VecIO<T, VEC>::load(src + kc * VEC, x);
#pragma unroll
                                for (int e = 0; e < VEC; ++e) d[i] = fmaf(g[k][e], x[e], d[i]);
                            }
                        }
                    }
                }
                const float gx = 1.0f - c.fx, gy = 1.0f - c.fy;
                dA = c.w[0] * d[0] + c.w[1] * d[1] + c.w[2] * d[2] + c.w[3] * d[3];
                dX = gy * (d[1] - d[0]) + c.fy * (d[3] - d[2]);  // d(sample)/d(pixel x), dotted with g
                dY = gx * (d[2] - d[0]) + c.fx * (d[3] - d[1]);  // d(sample)/d(pixel y), dotted with g
            }
            if (want_gv) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (c.valid & (1u << i)) {
                        const float aw = A * c.w[i];
                        float *dst = gbh + c.off[i];
#pragma unroll
                        for (int k = 0; k < NCH; ++k) {
                            const int kc = k * G + r;
                            if (kc < p.chunks) RedIO<VEC>::add(dst + kc * VEC, g[k], aw);
                        }
                    }
                }
            }
        }
        if (need_v) {
#pragma unroll
            for (int o = 1; o < G; o <<= 1) {
                dA += __shfl_xor_sync(0xffffffffu, dA, o);
                dX += __shfl_xor_sync(0xffffffffu, dX, o);
                dY += __shfl_xor_sync(0xffffffffu, dY, o);
            }
            if (active && r == 0) {
                if (want_ga) grad_attn[(int64_t)rw.bqh * p.NLP + j] = dA;
                if (want_gl) {
                    float *gl = grad_loc + lrow + j * p.l_sJ;
                    gl[0] = A * dX * p.sx[l];
                    gl[p.l_sXY] = A * dY * p.sy[l];
                }
            }
        }
    }
}

// ---------------------------------------------------------------- helpers
// Zero n floats (grid-stride; 16-byte stores when the pointer allows).
__global__ void msda_zero_f32_kernel(float *__restrict__ p, int64_t n);
// grad_value (bf16) = round-to-nearest-even(acc) for n elements.
__global__ void msda_f32_to_bf16_kernel(const float *__restrict__ acc, __nv_bfloat16 *__restrict__ out,
                                        int64_t n);

// Launchers (return cudaGetLastError() after the launch).
template <typename T>
cudaError_t launch_forward(const Params &p, bool vec, int G, int NCH, const T *value, const float *loc,
                           const float *attn, T *out, cudaStream_t stream);
template <typename T>
cudaError_t launch_backward(const Params &p, bool vec, int G, int NCH, const T *grad_out, const T *value,
                            const float *loc, const float *attn, float *gv_acc, float *grad_loc,
                            float *grad_attn, int flags, cudaStream_t stream);
cudaError_t launch_zero_f32(float *p, int64_t n, cudaStream_t stream);
cudaError_t launch_f32_to_bf16(const float *acc, __nv_bfloat16 *out, int64_t n, cudaStream_t stream);

}  // namespace msda
