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
// Work decomposition (both directions): a group of G lanes owns one row and
// walks its N_l*N_p samples in order; a warp therefore serves 32/G rows at
// once, rows ordered (b, h, q) so that the rows of a warp and of a block are
// neighbouring queries of one head (their samples reuse value lines in L1).
// Inside a group, lane r owns the 16-byte channel chunks r, r+G, r+2G, ...
// (NCH of them, VEC elements each), so each load instruction of a group reads
// G*16 contiguous bytes of a corner's channel row.  The G lanes of a group
// compute the sample's bilinear cell redundantly: that costs fewer
// instructions than distributing it, and the forward needs no cross-lane
// communication at all.  The backward reduces its three per-sample dot
// products over the G lanes with shuffles and scatters grad_value with
// vector atomics (red.global.add.v4.f32).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace msda {

constexpr int kMaxLevels = 16;
constexpr int kThreads = 256;

// Unsigned division by a runtime constant d >= 1, exact for every 32-bit n:
// n / d = (umulhi(n, mul) + n) >> shift, with shift = ceil(log2 d) and
// mul = floor(2^32 (2^shift - d) / d) + 1 (the sum is formed in 64 bits).
struct FastDiv {
    uint32_t d, mul, shift;
    __device__ __forceinline__ uint32_t div(uint32_t n) const {
        const uint64_t t = (uint64_t)__umulhi(n, mul) + n;
        return (uint32_t)(t >> shift);
    }
};

// Everything a kernel needs, passed by value (kernel parameter space).
struct Params {
    uint32_t rows;  // B * N_h * N_q, ordered (b, h, q)
    int N_q, N_h, C_h, N_l, N_p, NLP;
    int chunks;     // C_h / VEC: channel chunks per row
    FastDiv div_q, div_h, div_p;  // by N_q, N_h, N_p
    int padding;    // 0 zeros, 1 border (used when the kernel is not specialised)
    int flags;      // kGradValue | kGradLoc | kGradAttn (backward)
    // value (and grad_value / accumulator) element strides
    int64_t v_sB;
    int v_sH, v_sP;
    // sampling_locations (and its gradient): batch stride, per-sample stride, x -> y distance
    int64_t l_sB;
    int l_sJ, l_sXY;
    // per level
    int H[kMaxLevels], W[kMaxLevels], start[kMaxLevels];
    float sx[kMaxLevels], sy[kMaxLevels];  // pixels per unit of normalised coordinate
    float off;                             // -0.5 (align_corners = 0) or 0 (align_corners = 1)
    // backward: queries per block, and the levels accumulated in shared memory
    int q_chunk;
    int priv_start[kMaxLevels];  // first shared-memory pixel of a privatised level, -1 if not
    int priv_pixels;             // privatised pixels in total (C_h floats each)
    int swizzle;                 // rotate channels by pixel within 32-float runs (C_h % 32 == 0)
    int n_sm;                    // multiprocessors of the device (grid sizing)
};

enum : int { kGradValue = 1, kGradLoc = 2, kGradAttn = 4 };

// ---------------------------------------------------------------- element access
// Two binary32 values -> one register of two bfloat16 (round to nearest
// even), `lo` in the low half (the lower address).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

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
        *reinterpret_cast<uint4 *>(p) = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                                                   pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7]));
    }
};

template <> struct VecIO<__nv_bfloat16, 4> {
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float (&o)[4]) {
        const uint2 x = __ldg(reinterpret_cast<const uint2 *>(p));
        o[0] = __uint_as_float(x.x << 16);
        o[1] = __uint_as_float(x.x & 0xffff0000u);
        o[2] = __uint_as_float(x.y << 16);
        o[3] = __uint_as_float(x.y & 0xffff0000u);
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float (&o)[4]) {
        *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
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

// ---------------------------------------------------------------- geometry
struct Row {
    uint32_t b, q, h;
    uint32_t bqh;  // (b*N_q + q)*N_h + h: row of out / grad_output / attention_weights
};

__device__ __forceinline__ Row decode_row(const Params &p, uint32_t row) {
    Row r;
    const uint32_t bh = p.div_q.div(row);
    r.q = row - bh * (uint32_t)p.N_q;
    r.b = p.div_h.div(bh);
    r.h = bh - r.b * (uint32_t)p.N_h;
    r.bqh = (r.b * (uint32_t)p.N_q + r.q) * (uint32_t)p.N_h + r.h;
    return r;
}

// The bilinear cell of one sample on a level of W x H pixels.
//
// (x0, y0) is the corner of the cell; the corners are (y0,x0), (y0,x0+1),
// (y0+1,x0), (y0+1,x0+1) with weights (1-fx)(1-fy), fx(1-fy), (1-fx)fy,
// fx*fy; bit i of `valid` says corner i reads the map.
//   zeros : a corner outside the map reads 0 (its bit is clear).
//   border: corner indices clamp onto the map.  The cell is rewritten so
//           that every corner it reads is inside: along an axis where both
//           corners would clamp onto the same edge pixel, the cell moves onto
//           that pixel with fraction 0 (same values and same grad_value), and
//           kx / ky = 0 record that the sample does not move along that axis
//           (its location derivative there is 0).
// The pixel coordinate is first clamped to [-2, size+1]: every cell beyond
// that reads nothing ("zeros") or the same edge pixel ("border"), and the
// integer conversion stays in range for any input, NaN included.
struct Cell {
    int x0, y0;
    float fx, fy, kx, ky;
    unsigned valid;
};

template <int PAD>
__device__ __forceinline__ Cell make_cell(float u, float v, float sx, float sy, float off, int W, int H,
                                          int pad_runtime) {
    Cell c;
    float x = __fmaf_rn(u, sx, off);  // one rounding, as the reference mapping is linear
    float y = __fmaf_rn(v, sy, off);
    x = fminf(fmaxf(x, -2.0f), (float)W + 1.0f);
    y = fminf(fmaxf(y, -2.0f), (float)H + 1.0f);
    const float xf = floorf(x), yf = floorf(y);
    c.fx = x - xf;
    c.fy = y - yf;
    c.x0 = (int)xf;
    c.y0 = (int)yf;
    const bool border = PAD == 1 || (PAD < 0 && pad_runtime == 1);
    c.kx = 1.0f;
    c.ky = 1.0f;
    if (border) {
        if (c.x0 < 0 || c.x0 >= W - 1) {
            c.x0 = c.x0 < 0 ? 0 : W - 1;
            c.fx = 0.0f;
            c.kx = 0.0f;
        }
        if (c.y0 < 0 || c.y0 >= H - 1) {
            c.y0 = c.y0 < 0 ? 0 : H - 1;
            c.fy = 0.0f;
            c.ky = 0.0f;
        }
    }
    const bool ix0 = (unsigned)c.x0 < (unsigned)W, ix1 = (unsigned)(c.x0 + 1) < (unsigned)W;
    const bool iy0 = (unsigned)c.y0 < (unsigned)H, iy1 = (unsigned)(c.y0 + 1) < (unsigned)H;
    c.valid = (unsigned)(ix0 & iy0) | ((unsigned)(ix1 & iy0) << 1) | ((unsigned)(ix0 & iy1) << 2) |
              ((unsigned)(ix1 & iy1) << 3);
    return c;
}

// ---------------------------------------------------------------- forward
// Level tables copied to shared memory once per block: lanes of a warp look
// up different levels at the same time, which shared memory serves in one
// pass (the kernel parameter space would serialise distinct addresses).
struct LevelTables {
    int W[kMaxLevels], H[kMaxLevels], start[kMaxLevels], priv[kMaxLevels];
    float sx[kMaxLevels], sy[kMaxLevels];
};

__device__ __forceinline__ void load_level_tables(const Params &p, LevelTables &t) {
    if (threadIdx.x < (unsigned)p.N_l) {
        const int l = threadIdx.x;
        t.W[l] = p.W[l];
        t.H[l] = p.H[l];
        t.start[l] = p.start[l];
        t.priv[l] = p.priv_start[l];
        t.sx[l] = p.sx[l];
        t.sy[l] = p.sy[l];
    }
    __syncthreads();
}

// Corner offsets and weights of one sample, as the consumers of a group read
// them: corner i reads value at element offset off[i] (relative to the
// (b, h) slice) with weight w[i].  A corner that reads nothing ("zeros"
// padding outside the map) gets weight 0 and an offset clamped onto the map,
// so every corner can be loaded without a branch.  Non-finite numbers stored
// at such a clamped pixel would reach the sum as 0 * inf; the pages leave
// non-finite inputs unspecified.
struct alignas(16) CornerRec {
    int off[4];
    float w[4];
};

__device__ __forceinline__ void corner_offsets(const Cell &c, int W, int H, int start, int sP, int (&off)[4]) {
    const int xa = min(max(c.x0, 0), W - 1), xb = min(max(c.x0 + 1, 0), W - 1);
    const int ya = min(max(c.y0, 0), H - 1), yb = min(max(c.y0 + 1, 0), H - 1);
    const int ra = start + ya * W, rb = start + yb * W;
    off[0] = (ra + xa) * sP;
    off[1] = (ra + xb) * sP;
    off[2] = (rb + xa) * sP;
    off[3] = (rb + xb) * sP;
}

// A group of G lanes owns one row at a time.  Its samples are taken G at a
// time: lane r computes the bilinear cell of sample j0 + r (the cell
// arithmetic is done once per sample) and writes the sample's CornerRec to
// shared memory; then the group walks the G samples together, reads each
// record with two 16-byte shared loads and loads every corner's channel row
// with one instruction, two samples' corners before their multiply-adds.
// Blocks stay resident and loop over rows; while a group works on a row the
// locations and weights of its next row are already being fetched.
// PAD: 0 zeros, 1 border, -1 read p.padding at run time.
template <typename T, int VEC, int G, int NCH, int PAD>
__global__ void __launch_bounds__(kThreads, 3)
msda_forward_kernel(const Params p, const T *__restrict__ value, const float *__restrict__ loc,
                    const float *__restrict__ attn, T *__restrict__ out) {
    __shared__ LevelTables lt;
    __shared__ CornerRec recs[kThreads];  // one record per lane: [warp][s][group]
    load_level_tables(p, lt);
    constexpr int GPB = kThreads / G;  // groups (rows in flight) per block
    const int lane = threadIdx.x & 31;
    const int r = lane & (G - 1);
    const int grp = lane / G;
    const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane & ~(G - 1)));
    CornerRec *wrec = recs + (threadIdx.x & ~31);  // sample s of group g at s * (32 / G) + g
    CornerRec &mine = wrec[r * (32 / G) + grp];
    const int sP = p.v_sP, sJ = p.l_sJ, sXY = p.l_sXY;
    int nk = 0;  // chunks this lane owns: k*G + r < chunks
#pragma unroll
    for (int k = 0; k < NCH; ++k) nk += (k * G + r < p.chunks);
    constexpr int PF = 2;  // samples of a row whose inputs are prefetched per lane (batches 0 and 1)
    static_assert(PF == 2, "the owner phase below selects between two prefetched samples");
    const uint64_t stride = (uint64_t)gridDim.x * GPB;

    // inputs of this lane's first PF samples of a row
    auto fetch = [&](uint64_t row64, float (&u)[PF], float (&v)[PF], float (&A)[PF]) {
        if (row64 < p.rows) {
            const Row rw = decode_row(p, (uint32_t)row64);
            const float *lp = loc + rw.b * p.l_sB +
                              (int64_t)((rw.q * (uint32_t)p.N_h + rw.h) * (uint32_t)p.NLP) * sJ;
            const float *ap = attn + (int64_t)rw.bqh * p.NLP;
#pragma unroll
            for (int t = 0; t < PF; ++t) {
                const int j = r + t * G;
                if (j < p.NLP) {
                    u[t] = __ldg(lp + j * sJ);
                    v[t] = __ldg(lp + j * sJ + sXY);
                    A[t] = __ldg(ap + j);
                }
            }
        }
    };
    float nu[PF], nv[PF], nA[PF];
    uint64_t row64 = (uint64_t)blockIdx.x * GPB + threadIdx.x / G;
    fetch(row64, nu, nv, nA);
    for (; row64 < p.rows; row64 += stride) {
        float cu[PF], cv[PF], cA[PF];
#pragma unroll
        for (int t = 0; t < PF; ++t) {
            cu[t] = nu[t];
            cv[t] = nv[t];
            cA[t] = nA[t];
        }
        fetch(row64 + stride, nu, nv, nA);
        const Row rw = decode_row(p, (uint32_t)row64);
        const T *vbh = value + rw.b * p.v_sB + (int64_t)rw.h * p.v_sH + r * VEC;
        const float *lp = loc + rw.b * p.l_sB + (int64_t)((rw.q * (uint32_t)p.N_h + rw.h) * (uint32_t)p.NLP) * sJ;
        const float *ap = attn + (int64_t)rw.bqh * p.NLP;

        float acc[NCH][VEC];
#pragma unroll
        for (int k = 0; k < NCH; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[k][e] = 0.0f;

        for (int j0 = 0, t = 0; j0 < p.NLP; j0 += G, ++t) {
            // owner phase: this lane's sample
            {
                CornerRec rec;
                const int j = j0 + r;
                if (j < p.NLP) {
                    const int l = (int)p.div_p.div((uint32_t)j);
                    const int W = lt.W[l], H = lt.H[l];
                    float u, v, A;
                    if (t < PF) {  // prefetched
                        u = t == 0 ? cu[0] : cu[PF - 1];
                        v = t == 0 ? cv[0] : cv[PF - 1];
                        A = t == 0 ? cA[0] : cA[PF - 1];
                    } else {
                        u = __ldg(lp + j * sJ);
                        v = __ldg(lp + j * sJ + sXY);
                        A = __ldg(ap + j);
                    }
                    const Cell c = make_cell<PAD>(u, v, lt.sx[l], lt.sy[l], p.off, W, H, p.padding);
                    const float ax = A - A * c.fx, bx = A * c.fx;  // A(1-fx), A fx
                    const float gy = 1.0f - c.fy;
                    rec.w[0] = (c.valid & 1u) ? ax * gy : 0.0f;
                    rec.w[1] = (c.valid & 2u) ? bx * gy : 0.0f;
                    rec.w[2] = (c.valid & 4u) ? ax * c.fy : 0.0f;
                    rec.w[3] = (c.valid & 8u) ? bx * c.fy : 0.0f;
                    corner_offsets(c, W, H, lt.start[l], sP, rec.off);
                } else {  // past the last sample: four zero-weight reads of pixel 0
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        rec.off[i] = 0;
                        rec.w[i] = 0.0f;
                    }
                }
                mine = rec;
            }
            __syncwarp(gmask);
            // consume phase: the group's G samples, two at a time
            // two samples' corners in flight when a lane's share of a corner is
            // at most 4 floats, else one (register budget)
            constexpr int S2 = (G >= 2 && NCH * VEC <= 4) ? 2 : 1;
#pragma unroll
            for (int s = 0; s < G; s += S2) {
                CornerRec rec[S2];
                float x[S2][4][NCH][VEC];
#pragma unroll
                for (int h2 = 0; h2 < S2; ++h2) {
                    rec[h2] = wrec[(s + h2) * (32 / G) + grp];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const T *src = vbh + rec[h2].off[i];
#pragma unroll
                        for (int k = 0; k < NCH; ++k)
                            if (k < nk) VecIO<T, VEC>::load(src + k * G * VEC, x[h2][i][k]);
                    }
                }
#pragma unroll
                for (int h2 = 0; h2 < S2; ++h2)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int k = 0; k < NCH; ++k)
                            if (k < nk)
#pragma unroll
                                for (int e = 0; e < VEC; ++e)
                                    acc[k][e] = fmaf(rec[h2].w[i], x[h2][i][k][e], acc[k][e]);
            }
            __syncwarp(gmask);  // records are rewritten by the next batch
        }
        T *dst = out + (int64_t)rw.bqh * p.C_h + r * VEC;
#pragma unroll
        for (int k = 0; k < NCH; ++k)
            if (k < nk) VecIO<T, VEC>::store(dst + k * G * VEC, acc[k]);
    }
}

// ---------------------------------------------------------------- backward
constexpr int kBwdThreads = 512;

// Sum each of a lane's G per-sample partials over the G lanes of its group so
// that lane r ends with the total of sample r (a transposed butterfly: at
// each step a lane keeps half of its entries and sends the other half to its
// partner, G-1 shuffles in all).
template <int G>
__device__ __forceinline__ float reduce_scatter(float (&v)[G], int r, unsigned gmask) {
#pragma unroll
    for (int o = G / 2; o >= 1; o >>= 1) {
        const bool up = (r & o) != 0;
#pragma unroll
        for (int t = 0; t < o; ++t) {
            const float send = up ? v[t] : v[t + o];
            const float keep = up ? v[t + o] : v[t];
            v[t] = keep + __shfl_xor_sync(gmask, send, o);
        }
    }
    return v[0];
}

// Shared-memory index of channel c of privatised pixel px.  With C_h a
// multiple of 32 the channels of a pixel are rotated by the pixel index
// inside each run of 32 floats, so the groups of a warp that add to
// different pixels at once spread over the banks.
__device__ __forceinline__ int priv_index(int px, int c, int C_h, int swz) {
    return px * C_h + (swz ? ((c & ~31) | ((c + px) & 31)) : c);
}

// What the consumers of a group need of one sample in the backward: the
// pixels of its four corners (clamped onto the map when a corner reads
// nothing), the bilinear weights w (0 for such corners) and their derivatives
// with respect to the pixel coordinates (dwx, dwy; also 0 for such corners),
// the attention weight, and pdelta = (shared-memory pixel - pixel) when the
// sample's level is accumulated in shared memory (kNoPriv otherwise).
constexpr int kNoPriv = -2147483647 - 1;
struct alignas(16) BwdRec {
    int pix[4];
    float w[4], dwx[4], dwy[4];
    float A;
    int pdelta;
    int pad_[2];
};

// A block owns one (b, h) and the queries [q0, q0 + q_chunk); a group of G
// lanes owns one query row at a time and walks its samples G at a time, as in
// the forward: lane r computes sample j0 + r's cell and writes its BwdRec to
// shared memory, and the group reads each record back and loads each
// corner's channel row with one instruction.  Per sample and lane it forms
// the partial dot products d_i of g with the four corners, then
// <g, S> = sum w_i d_i (grad_attention) and <g, dS/dx> = sum dwx_i d_i,
// <g, dS/dy> = sum dwy_i d_i (grad_location); a transposed butterfly leaves
// lane r with sample r's totals, which it stores.  grad_value receives
// A*w_i*g per corner: into a block-private binary32 copy in shared memory for
// the privatised (small) levels when PRIV, flushed with vector atomics at the
// end, else straight into the accumulator with red.global.add.v4.f32.
// FL: kGradValue|kGradLoc|kGradAttn or kGradValue (exactly these outputs),
// kGradLoc|kGradAttn (no grad_value; the two others as p.flags says), or -1
// (everything from p.flags at run time).  PAD as in the forward.
template <typename T, int VEC, int G, int NCH, int PAD, int FL, bool PRIV>
__global__ void __launch_bounds__(kBwdThreads)
msda_backward_kernel(const Params p, const T *__restrict__ grad_out, const T *__restrict__ value,
                     const float *__restrict__ loc, const float *__restrict__ attn,
                     float *__restrict__ gv_acc, float *__restrict__ grad_loc,
                     float *__restrict__ grad_attn) {
    extern __shared__ float s_acc[];
    __shared__ LevelTables lt;
    __shared__ BwdRec recs[kBwdThreads];  // one record per lane: [warp][s][group]
    load_level_tables(p, lt);
    const int flags = FL < 0 ? p.flags : (FL == (kGradLoc | kGradAttn) ? (p.flags & FL) : FL);
    const bool want_gv = flags & kGradValue, want_gl = flags & kGradLoc, want_ga = flags & kGradAttn;
    const bool need_v = want_gl || want_ga;  // value is read only for these two
    const bool need_a = want_gv || want_gl;  // attention is read only for these two
    if constexpr (PRIV) {
        for (int i = threadIdx.x; i < p.priv_pixels * p.C_h; i += kBwdThreads) s_acc[i] = 0.0f;
        __syncthreads();
    }

    const int lane = threadIdx.x & 31;
    const int r = lane & (G - 1);
    const int grp = lane / G;
    const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane & ~(G - 1)));
    BwdRec *wrec = recs + (threadIdx.x & ~31);
    BwdRec &mine = wrec[r * (32 / G) + grp];
    const uint32_t bhi = blockIdx.x;  // b * N_h + h
    const uint32_t b = p.div_h.div(bhi), h = bhi - b * (uint32_t)p.N_h;
    const uint32_t q0 = blockIdx.y * (uint32_t)p.q_chunk;
    const uint32_t q1 = min((uint32_t)p.N_q, q0 + (uint32_t)p.q_chunk);
    const int64_t bhoff = b * p.v_sB + (int64_t)h * p.v_sH;
    const T *vbh = value + bhoff + r * VEC;
    float *gbh = gv_acc + bhoff + r * VEC;
    const int sP = p.v_sP, sJ = p.l_sJ, sXY = p.l_sXY;
    int nk = 0;  // chunks this lane owns: k*G + r < chunks
#pragma unroll
    for (int k = 0; k < NCH; ++k) nk += (k * G + r < p.chunks);

    for (uint32_t q = q0 + threadIdx.x / G; q < q1; q += kBwdThreads / G) {
        const uint32_t bqh = (b * (uint32_t)p.N_q + q) * (uint32_t)p.N_h + h;
        const int64_t lrow = b * p.l_sB + (int64_t)((q * (uint32_t)p.N_h + h) * (uint32_t)p.NLP) * sJ;
        const float *lp = loc + lrow;
        float *glp = grad_loc + lrow;
        const float *ap = attn + (int64_t)bqh * p.NLP;
        float *gap = grad_attn + (int64_t)bqh * p.NLP;
        float g[NCH][VEC];
        {
            const T *src = grad_out + (int64_t)bqh * p.C_h + r * VEC;
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

        for (int j0 = 0; j0 < p.NLP; j0 += G) {
            // owner phase: this lane's sample
            const int j = j0 + r;
            float A = 0.0f, sxk = 0.0f, syk = 0.0f;
            {
                BwdRec rec;
                rec.pdelta = kNoPriv;
                if (j < p.NLP) {
                    const int l = (int)p.div_p.div((uint32_t)j);
                    const int W = lt.W[l], H = lt.H[l];
                    const float u = __ldg(lp + j * sJ), v = __ldg(lp + j * sJ + sXY);
                    if (need_a) A = __ldg(ap + j);
                    const Cell c = make_cell<PAD>(u, v, lt.sx[l], lt.sy[l], p.off, W, H, p.padding);
                    const int xa = min(max(c.x0, 0), W - 1), xb = min(max(c.x0 + 1, 0), W - 1);
                    const int ya = min(max(c.y0, 0), H - 1), yb = min(max(c.y0 + 1, 0), H - 1);
                    const int ra = lt.start[l] + ya * W, rb = lt.start[l] + yb * W;
                    rec.pix[0] = ra + xa;
                    rec.pix[1] = ra + xb;
                    rec.pix[2] = rb + xa;
                    rec.pix[3] = rb + xb;
                    const float gx = 1.0f - c.fx, gy = 1.0f - c.fy;
                    const float w[4] = {gx * gy, c.fx * gy, gx * c.fy, c.fx * c.fy};
                    const float dwx[4] = {-gy, gy, -c.fy, c.fy};
                    const float dwy[4] = {-gx, -c.fx, gx, c.fx};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const bool ok = c.valid & (1u << i);
                        rec.w[i] = ok ? w[i] : 0.0f;
                        rec.dwx[i] = ok ? dwx[i] : 0.0f;
                        rec.dwy[i] = ok ? dwy[i] : 0.0f;
                    }
                    rec.A = A;
                    if constexpr (PRIV) rec.pdelta = lt.priv[l] >= 0 ? lt.priv[l] - lt.start[l] : kNoPriv;
                    sxk = lt.sx[l] * c.kx;
                    syk = lt.sy[l] * c.ky;
                } else {  // past the last sample: zero-weight reads of pixel 0
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        rec.pix[i] = 0;
                        rec.w[i] = rec.dwx[i] = rec.dwy[i] = 0.0f;
                    }
                    rec.A = 0.0f;
                }
                mine = rec;
            }
            __syncwarp(gmask);
            float pa[G], px[G], py[G];
            // consume phase: the group's G samples, in order
#pragma unroll
            for (int s = 0; s < G; ++s) {
                const BwdRec &rec = wrec[s * (32 / G) + grp];
                int pix[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) pix[i] = rec.pix[i];
                pa[s] = px[s] = py[s] = 0.0f;
                if (need_v) {
                    float d[4];  // this lane's part of <g, corner i>
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        d[i] = 0.0f;
                        const T *src = vbh + pix[i] * sP;
#pragma unroll
                        for (int k = 0; k < NCH; ++k) {
                            if (k < nk) {
                                float x[VEC];
                                VecIO<T, VEC>::load(src + k * G * VEC, x);
#pragma unroll
                                for (int e = 0; e < VEC; ++e) d[i] = fmaf(g[k][e], x[e], d[i]);
                            }
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        pa[s] = fmaf(rec.w[i], d[i], pa[s]);
                        px[s] = fmaf(rec.dwx[i], d[i], px[s]);
                        py[s] = fmaf(rec.dwy[i], d[i], py[s]);
                    }
                    if constexpr (G > 8) {  // wide groups: reduce per sample, the owner stores
                        float ta = pa[s], tx = px[s], ty = py[s];
#pragma unroll
                        for (int o = 1; o < G; o <<= 1) {
                            ta += __shfl_xor_sync(gmask, ta, o);
                            tx += __shfl_xor_sync(gmask, tx, o);
                            ty += __shfl_xor_sync(gmask, ty, o);
                        }
                        if (r == s && j < p.NLP) {
                            if (want_ga) gap[j] = ta;
                            if (want_gl) {
                                glp[j * sJ] = A * tx * sxk;
                                glp[j * sJ + sXY] = A * ty * syk;
                            }
                        }
                    }
                }
                if (want_gv) {
                    const float As = rec.A;
                    const int pdelta = PRIV ? rec.pdelta : kNoPriv;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float aw = As * rec.w[i];
                        if (aw != 0.0f) {
                            if (PRIV && pdelta != kNoPriv) {
                                const int pxi = pix[i] + pdelta;
#pragma unroll
                                for (int k = 0; k < NCH; ++k)
                                    if (k < nk)
#pragma unroll
                                        for (int e = 0; e < VEC; ++e)
                                            atomicAdd(&s_acc[priv_index(pxi, (k * G + r) * VEC + e, p.C_h, p.swizzle)],
                                                      aw * g[k][e]);
                            } else {
                                float *dst = gbh + pix[i] * sP;
#pragma unroll
                                for (int k = 0; k < NCH; ++k)
                                    if (k < nk) RedIO<VEC>::add(dst + k * G * VEC, g[k], aw);
                            }
                        }
                    }
                }
            }
            __syncwarp(gmask);  // records are rewritten by the next batch
            if constexpr (G <= 8) {
                if (need_v) {
                    const float ta = reduce_scatter<G>(pa, r, gmask);
                    const float tx = reduce_scatter<G>(px, r, gmask);
                    const float ty = reduce_scatter<G>(py, r, gmask);
                    if (j < p.NLP) {
                        if (want_ga) gap[j] = ta;
                        if (want_gl) {
                            glp[j * sJ] = A * tx * sxk;
                            glp[j * sJ + sXY] = A * ty * syk;
                        }
                    }
                }
            }
        }
    }

    if constexpr (PRIV) {
        // Add the block's private levels into the accumulator: one 16-byte
        // atomic per 4 channels of a pixel, skipping pixels this block never
        // touched.
        __syncthreads();
        const int c4n = p.C_h / 4;
        float *gb = gv_acc + bhoff;
        for (int idx = threadIdx.x; idx < p.priv_pixels * c4n; idx += kBwdThreads) {
            const int pxi = idx / c4n, c = (idx - pxi * c4n) * 4;
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = s_acc[priv_index(pxi, c + e, p.C_h, p.swizzle)];
            if (v[0] != 0.0f || v[1] != 0.0f || v[2] != 0.0f || v[3] != 0.0f) {
                int l = 0;
                while (!(lt.priv[l] >= 0 && pxi >= lt.priv[l] && pxi < lt.priv[l] + lt.W[l] * lt.H[l])) ++l;
                const int gpix = lt.start[l] + (pxi - lt.priv[l]);
                red_add_v4(gb + (int64_t)gpix * sP + c, v[0], v[1], v[2], v[3]);
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
template <typename T, bool VECTOR>
cudaError_t launch_forward_path(const Params &p, int G, int NCH, const T *value, const float *loc,
                                const float *attn, T *out, cudaStream_t stream);
template <typename T>
inline cudaError_t launch_forward(const Params &p, bool vec, int G, int NCH, const T *value, const float *loc,
                                  const float *attn, T *out, cudaStream_t stream) {
    if (p.rows == 0) return cudaSuccess;
    return vec ? launch_forward_path<T, true>(p, G, NCH, value, loc, attn, out, stream)
               : launch_forward_path<T, false>(p, G, NCH, value, loc, attn, out, stream);
}
template <typename T, int PAD>
cudaError_t launch_backward_pad(const Params &p, int G, int NCH, bool priv, const T *grad_out, const T *value,
                                const float *loc, const float *attn, float *gv_acc, float *grad_loc,
                                float *grad_attn, cudaStream_t stream);
// Dispatch on vector path / padding to the launch_backward_pad instantiations.
template <typename T>
inline cudaError_t launch_backward(const Params &p, bool vec, int G, int NCH, bool priv, const T *grad_out,
                                   const T *value, const float *loc, const float *attn, float *gv_acc,
                                   float *grad_loc, float *grad_attn, cudaStream_t stream) {
    if (p.rows == 0) return cudaSuccess;
    if (!vec)
        return launch_backward_pad<T, -1>(p, G, NCH, false, grad_out, value, loc, attn, gv_acc, grad_loc,
                                          grad_attn, stream);
    if (p.padding == 0)
        return launch_backward_pad<T, 0>(p, G, NCH, priv, grad_out, value, loc, attn, gv_acc, grad_loc,
                                         grad_attn, stream);
    return launch_backward_pad<T, 1>(p, G, NCH, priv, grad_out, value, loc, attn, gv_acc, grad_loc, grad_attn,
                                     stream);
}
cudaError_t launch_zero_f32(float *p, int64_t n, cudaStream_t stream);
cudaError_t launch_f32_to_bf16(const float *acc, __nv_bfloat16 *out, int64_t n, cudaStream_t stream);

}  // namespace msda
