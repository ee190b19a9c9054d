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
// Inside a group, lane r owns the channel chunks r, r+G, r+2G, ... (NCH of
// them, VEC elements each), so each load instruction of a group reads one
// contiguous piece of a corner's channel row.  The samples are taken G at a
// time: lane r computes sample j0 + r's bilinear cell once and hands it to
// the group through swizzled shared-memory records (wide forward rows: by
// shuffles).  The backward sums its per-sample dot products over
// the G lanes with a transposed butterfly and scatters grad_value with vector
// atomics (red.global.add.v4.f32) -- for 32-channel rows after merging the
// contributions of a warp's four rows that land on one pixel -- or, for
// grad_value-only calls on dense problems, through the tile-sorted path
// further down.  The staged variants (coarse levels in shared memory) are in
// msda_staged.cuh.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
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

// Everything a kernel needs, passed by value (kernel parameter space; the
// kernels take it as __grid_constant__, so per-level entries indexed by a
// warp-uniform level are read from the constant bank without a local copy).
struct Params {
    uint32_t rows;  // B * N_h * N_q, ordered (b, h, q)
    int N_q, N_h, C_h, N_l, N_p, NLP;
    int chunks;     // C_h / VEC: channel chunks per row
    FastDiv div_q, div_h, div_p, div_nlp;  // by N_q, N_h, N_p, N_l * N_p
    int padding;    // 0 zeros, 1 border (used when the kernel is not specialised)
    int flags;      // kGradValue | kGradLoc | kGradAttn (backward)
    int logits;     // 1: `attention_weights` holds logits; A = softmax over the row's N_l*N_p of them
    int loc_dt;     // dtype of locations, weights and their gradients: 0 binary32, 1 bfloat16, 2 binary16
    int split_log2; // row kernels: each row's samples split over 2^split_log2 groups (see block_rows)
    int aggregate;  // backward: warp-aggregated grad_value scatter where the kernel shape has one
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
    int n_sm;                              // multiprocessors of the device (grid sizing)
    // tile-sorted grad_value (see the partition and reduction kernels below)
    int NB;                     // tiles (kTileCells x kTileCells cells) of one (b, h)
    int bst[kMaxLevels];        // first tile of level l inside a (b, h)
    int BX[kMaxLevels];         // tiles per tile row of level l
    uint32_t nbins;             // B * N_h * NB
    uint32_t parts;             // partition blocks (counts are kept per tile and block)
    uint32_t part_rows;         // rows of one partition block
    int span;                   // most (b, h) pairs one partition block's rows touch
    uint32_t capacity;          // entries the workspace holds (= samples)
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
    static __device__ __forceinline__ void add_sum(float *p, const float (&v)[1]) { red_add(p, v[0]); }
};
// s * v with packed binary32 products (rounded as the scalar products would be)
__device__ __forceinline__ void red_add_scaled4(float *p, const float *v, float s) {
    const float2 ss = make_float2(s, s);
    const float2 lo = __fmul2_rn(ss, make_float2(v[0], v[1]));
    const float2 hi = __fmul2_rn(ss, make_float2(v[2], v[3]));
    red_add_v4(p, lo.x, lo.y, hi.x, hi.y);
}
template <> struct RedIO<4> {
    static __device__ __forceinline__ void add(float *p, const float (&v)[4], float s) { red_add_scaled4(p, v, s); }
    static __device__ __forceinline__ void add_sum(float *p, const float (&v)[4]) {
        red_add_v4(p, v[0], v[1], v[2], v[3]);
    }
};
template <> struct RedIO<8> {
    static __device__ __forceinline__ void add(float *p, const float (&v)[8], float s) {
        red_add_scaled4(p, v, s);
        red_add_scaled4(p + 4, v + 4, s);
    }
    static __device__ __forceinline__ void add_sum(float *p, const float (&v)[8]) {
        red_add_v4(p, v[0], v[1], v[2], v[3]);
        red_add_v4(p + 4, v[4], v[5], v[6], v[7]);
    }
};

// Packed binary32 arithmetic (sm_100 and later): one instruction applies an
// FMA or a product to two lanes of data; each element is rounded exactly as
// fmaf / a binary32 product would round it, so results are unchanged.
// acc[e] += w * x[e] for the VEC elements of a chunk.
template <int VEC>
__device__ __forceinline__ void axpy(float (&acc)[VEC], float w, const float (&x)[VEC]) {
    if constexpr (VEC % 2 == 0) {
        const float2 ww = make_float2(w, w);
#pragma unroll
        for (int e = 0; e < VEC; e += 2) {
            const float2 r = __ffma2_rn(ww, make_float2(x[e], x[e + 1]), make_float2(acc[e], acc[e + 1]));
            acc[e] = r.x;
            acc[e + 1] = r.y;
        }
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] = fmaf(w, x[e], acc[e]);
    }
}

// dp += the products g[e] x[e] of one chunk, even channels into dp.x and odd
// ones into dp.y (packed FMAs); <g, x> over a lane's chunks is dp.x + dp.y.
template <int VEC>
__device__ __forceinline__ void dot_acc(float2 &dp, const float (&g)[VEC], const float (&x)[VEC]) {
    if constexpr (VEC % 2 == 0) {
#pragma unroll
        for (int e = 0; e < VEC; e += 2)
            dp = __ffma2_rn(make_float2(g[e], g[e + 1]), make_float2(x[e], x[e + 1]), dp);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) dp.x = fmaf(g[e], x[e], dp.x);
    }
}

// Locations, attention weights and their gradients in their storage dtype
// (dt: 0 binary32, 1 bfloat16, 2 binary16), addressed by element index from
// the tensor's base; arithmetic is binary32, stores round to nearest even.
__device__ __forceinline__ float ldl(const float *base, int64_t i, int dt) {
    if (dt == 0) return __ldg(base + i);
    const unsigned short bits = __ldg(reinterpret_cast<const unsigned short *>(base) + i);
    if (dt == 1) return __uint_as_float((uint32_t)bits << 16);  // bfloat16 -> binary32 is exact
    return __half2float(__ushort_as_half(bits));
}
// The same for an element this thread wrote earlier in the kernel (not
// through the read-only path).
// Both coordinates of a sample: one 8-byte read when they are adjacent binary32
// values at an 8-byte aligned address (pair), else two reads.
__device__ __forceinline__ void ld_uv(const float *base, int64_t i, int sXY, int dt, bool pair, float &u, float &v) {
    if (pair) {
        const float2 t = __ldg(reinterpret_cast<const float2 *>(base + i));
        u = t.x;
        v = t.y;
    } else {
        u = ldl(base, i, dt);
        v = ldl(base, i + sXY, dt);
    }
}
__device__ __forceinline__ float ldl_own(const float *base, int64_t i, int dt) {
    if (dt == 0) return base[i];
    const unsigned short bits = reinterpret_cast<const unsigned short *>(base)[i];
    if (dt == 1) return __uint_as_float((uint32_t)bits << 16);
    return __half2float(__ushort_as_half(bits));
}
__device__ __forceinline__ void stl(float *base, int64_t i, float v, int dt) {
    if (dt == 0) base[i] = v;
    else if (dt == 1) reinterpret_cast<__nv_bfloat16 *>(base)[i] = __float2bfloat16_rn(v);
    else reinterpret_cast<__half *>(base)[i] = __float2half_rn(v);
}
// The store counterpart of ld_uv.
__device__ __forceinline__ void st_uv(float *base, int64_t i, int sXY, int dt, bool pair, float x, float y) {
    if (pair) {
        *reinterpret_cast<float2 *>(base + i) = make_float2(x, y);
    } else {
        stl(base, i, x, dt);
        stl(base, i + sXY, y, dt);
    }
}

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

// ---------------------------------------------------------------- shared by the row kernels
// Level tables copied to shared memory once per block: the lanes of a warp
// look up different levels at once, which shared memory serves in one pass.
struct LevelTables {
    int W[kMaxLevels], H[kMaxLevels], start[kMaxLevels], bst[kMaxLevels], BX[kMaxLevels];
    float sx[kMaxLevels], sy[kMaxLevels];
    float4 geo[kMaxLevels];  // (sx, sy, W, H) of a level in one 16-byte read (W, H as int bits)
};
__device__ __forceinline__ void load_level_tables(const Params &p, LevelTables &t) {
    if (threadIdx.x < (unsigned)p.N_l) {
        const int l = threadIdx.x;
        t.W[l] = p.W[l];
        t.H[l] = p.H[l];
        t.start[l] = p.start[l];
        t.bst[l] = p.bst[l];
        t.BX[l] = p.BX[l];
        t.sx[l] = p.sx[l];
        t.sy[l] = p.sy[l];
        t.geo[l] = make_float4(p.sx[l], p.sy[l], __int_as_float(p.W[l]), __int_as_float(p.H[l]));
    }
    __syncthreads();
}

// Corner reads and weights of one sample.  o[i] is the element offset
// (relative to the (b, h) slice of value) of corner i = (0,0), (0,1), (1,0),
// (1,1) (row, column) of the cell, clamped onto the map, so that every corner
// can be loaded without a branch; w[i] is the bilinear weight times A, 0 for
// a corner outside the map ("zeros").  (Non-finite numbers stored at such a
// clamped pixel would reach the sum as 0 * inf; the pages leave non-finite
// inputs unspecified.)  The weights are formed as ay_i * ax_k with
// ax0 = A(1-fx), ax1 = A fx, ay0 = 1-fy, ay1 = fy.
struct Corners {
    int o[4];
    float w[4];
};

__device__ __forceinline__ Corners corners_of(const Cell &c, float A, int W, int H, int start, int sP) {
    const int xa = min(max(c.x0, 0), W - 1), xb = min(max(c.x0 + 1, 0), W - 1);
    const int ya = min(max(c.y0, 0), H - 1), yb = min(max(c.y0 + 1, 0), H - 1);
    Corners k;
    const int ra = start + ya * W, rb = start + yb * W;
    k.o[0] = (ra + xa) * sP;
    k.o[1] = (ra + xb) * sP;
    k.o[2] = (rb + xa) * sP;
    k.o[3] = (rb + xb) * sP;
    const float A1 = A * c.fx;
    const float ax0 = A - A1, ax1 = A1, ay0 = 1.0f - c.fy, ay1 = c.fy;
    k.w[0] = (c.valid & 1u) ? ay0 * ax0 : 0.0f;
    k.w[1] = (c.valid & 2u) ? ay0 * ax1 : 0.0f;
    k.w[2] = (c.valid & 4u) ? ay1 * ax0 : 0.0f;
    k.w[3] = (c.valid & 8u) ? ay1 * ax1 : 0.0f;
    return k;
}

// Per-warp exchange of sample records through shared memory.  A group of G
// lanes owns one row; lane r computes the record of the row's sample j0 + r
// and the group then reads the G records back one sample at a time.  Records
// are two 16-byte halves kept in two arrays; record (group g, sample s) sits
// at position g*G + (s ^ f(g)) of the warp's 32, with f chosen so that the
// groups of a warp reading sample s at the same time hit distinct 16-byte
// bank slots (one wavefront per read), while each group's stores fill its own
// G positions (contiguous, one wavefront per 128 bytes).
template <int G> __device__ __forceinline__ int rec_pos(int g, int s) {
    if constexpr (G >= 8) return g * G + (s ^ g);
    else if constexpr (G == 4) return g * G + (s ^ ((g >> 1) & 3));
    else return g * G + s;
}

// Work items of a block: the blocks (as many as fit on the GPU at once) sweep
// the items together, GPB consecutive items per block and step, so at any
// time the whole GPU works on one window of neighbouring queries: value lines
// are shared in L2 by the multiprocessors and in L1 by a block's groups.
// (Giving each block its own contiguous run of rows measured slower.)  An
// item is one part of a row: with S = 2^split_log2 parts (chosen > 1 only when
// the rows alone would leave most of the GPU idle), item t is part t % S of
// row t / S, and part k takes the row's sample batches k, k + S, k + 2S, ...
// The S parts of a row are neighbouring groups of one warp, so the forward
// sums their partial outputs with shuffles; the row's dependent chain of
// loads is S times shorter.
struct RowRange {
    uint32_t beg, end, step;
};
template <int GPB>
__device__ __forceinline__ RowRange block_rows(const Params &p, int split_log2) {
    RowRange rr;
    rr.beg = blockIdx.x * GPB;
    rr.end = p.rows << split_log2;
    rr.step = gridDim.x * GPB;
    return rr;
}

// Sum a row's S part accumulators over its S groups (lanes G, 2G, ... apart;
// `lane` is the caller's lane in the warp); every part ends with the total.
template <int G, int NCH, int VEC>
__device__ __forceinline__ void sum_parts(float (&acc)[NCH][VEC], int split_log2, int lane) {
    if (split_log2 == 0) return;
    const int span = G << split_log2;  // lanes of the row (<= 32)
    const unsigned pmask = span >= 32 ? 0xffffffffu : (((1u << span) - 1u) << (lane & ~(span - 1)));
    for (int o = G; o < span; o <<= 1)
#pragma unroll
        for (int k = 0; k < NCH; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[k][e] += __shfl_xor_sync(pmask, acc[k][e], o);
}

// Softmax of one row's N_l*N_p attention logits (the attention weights the
// workloads are built from), over the G lanes of its group: every lane ends
// with the row maximum m and 1 / sum_j exp(x_j - m), and the weight of sample
// j is then exp(x_j - m) times the latter.
template <int G>
__device__ __forceinline__ float2 row_softmax_stats(const float *attn, int64_t ao, int NLP, int r, unsigned gmask,
                                                    int dt) {
    float m = -INFINITY;
    for (int j = r; j < NLP; j += G) m = fmaxf(m, ldl(attn, ao + j, dt));
#pragma unroll
    for (int o = G / 2; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(gmask, m, o));
    float sum = 0.0f;
    for (int j = r; j < NLP; j += G) sum += expf(ldl(attn, ao + j, dt) - m);
#pragma unroll
    for (int o = G / 2; o >= 1; o >>= 1) sum += __shfl_xor_sync(gmask, sum, o);
    return make_float2(m, 1.0f / sum);
}

// ---------------------------------------------------------------- forward
#ifndef MSDA_FWD_INFLIGHT
#define MSDA_FWD_INFLIGHT 2
#endif
#ifndef MSDA_FWD_MIN_BLOCKS
#define MSDA_FWD_MIN_BLOCKS 4
#endif
#ifndef MSDA_BWD_MIN_BLOCKS
#define MSDA_BWD_MIN_BLOCKS 3
#endif
// Blocks per SM the row kernels are compiled for: for one 4-element chunk a
// lane the forward 4 (64 registers a thread: more warps to hide the gather
// latency) and the backward 3 (85 registers: its per-sample partials and
// reduction need them); for two chunks the forward 3 and the backward 2; 2
// (128 registers) for the wide-row kernels (one block per SM for the widest
// backward rows removes their spill but measured slower).
__host__ __device__ constexpr int row_min_blocks(int elems, bool fwd) {
    return elems <= 4 ? (fwd ? MSDA_FWD_MIN_BLOCKS : MSDA_BWD_MIN_BLOCKS) : (elems <= 8 && fwd) ? 3 : 2;
}

// One sample's cell in the form the lanes of a group exchange by six 32-bit
// shuffles (rows wider than four chunks a lane, and the staged forward; the
// others use the shared-memory records of Corners): o0 is the element offset
// (relative to the (b, h) slice of value)
// of the top-left corner read, with bit 31 set when the right-hand corners
// read the next pixel to the right (clear when both columns clamp onto the
// same pixel; offsets are below 2^31), o1 the offset of the bottom-left
// corner read, and w the four corner weights ay_i * ax_k with ax0 = A(1-fx),
// ax1 = A fx, ay0 = 1-fy, ay1 = fy, a factor 0 when its column or row lies
// outside the map ("zeros").  The owner forms the products once, so the
// group's lanes do not each repeat them.
struct FwdCell {
    int o0, o1;
    float w00, w01, w10, w11;
};

__device__ __forceinline__ FwdCell fwd_cell(const Cell &c, float A, int W, int H, int start, int sP) {
    const int xa = min(max(c.x0, 0), W - 1), xb = min(max(c.x0 + 1, 0), W - 1);
    const int ya = min(max(c.y0, 0), H - 1), yb = min(max(c.y0 + 1, 0), H - 1);
    FwdCell f;
    f.o0 = (int)((unsigned)((start + ya * W + xa) * sP) | ((unsigned)(xb - xa) << 31));
    f.o1 = (start + yb * W + xa) * sP;
    const float A1 = A * c.fx;
    const float ax0 = (c.valid & 5u) ? A - A1 : 0.0f;  // column x0 lies in the map
    const float ax1 = (c.valid & 10u) ? A1 : 0.0f;     // column x0 + 1
    const float ay0 = (c.valid & 3u) ? 1.0f - c.fy : 0.0f;
    const float ay1 = (c.valid & 12u) ? c.fy : 0.0f;
    f.w00 = ay0 * ax0;
    f.w01 = ay0 * ax1;
    f.w10 = ay1 * ax0;
    f.w11 = ay1 * ax1;
    return f;
}

// A group of G lanes owns one row (b, q, h) at a time; a block's groups take
// consecutive rows of its run, so the rows in flight on a multiprocessor are
// neighbouring queries of one head and reuse value lines in L1.  The row's
// samples are taken G at a time: lane r loads sample j0 + r's location and
// weight (coalesced), computes its bilinear cell once and publishes it as a
// record (four corner offsets, four weights) in shared memory, at the
// swizzled position the backward uses; the group then walks the G samples,
// reading each record (two 16-byte loads; rows of more than four chunks a
// lane take the cell by shuffles instead), and loads every corner's channel
// row with one instruction per channel chunk (lane r owns chunks r, r+G, ...),
// two samples' corners in flight; the next batch's location and weight are
// loaded before the current batch is consumed.
// PAD: 0 zeros, 1 border, -1 read p.padding at run time.  GEN: false for
// binary32 weights (p.loc_dt == 0, p.logits == 0, the common case compiled
// without the branches), true reads both at run time (with the backward's
// register budget: the softmax statistics need registers).  FULL: every
// batch holds G samples (N_l*N_p a multiple of G) and every lane owns all NCH
// chunks (C_h = G*NCH*VEC), so the partial-batch and masked-lane guards
// compile away.
template <typename T, int VEC, int G, int NCH, int PAD, bool GEN, bool SPLIT, bool FULL>
__global__ void __launch_bounds__(kThreads, row_min_blocks(NCH *VEC, !GEN))
msda_forward_kernel(const __grid_constant__ Params p, const T *__restrict__ value, const float *__restrict__ loc,
                    const float *__restrict__ attn, T *__restrict__ out) {
    __shared__ LevelTables lt;
    constexpr bool REC = NCH <= 4;  // cell records in shared memory (wide rows: shuffles)
    __shared__ int4 rec_o[REC ? kThreads : 1];
    __shared__ float4 rec_w[REC ? kThreads : 1];
    load_level_tables(p, lt);
    constexpr int GPB = kThreads / G;  // rows in flight per block
    const int lane = threadIdx.x & 31;
    const int r = lane & (G - 1);
    const int base = lane & ~(G - 1);
    const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << base);
    int4 *wo = rec_o + (REC ? (threadIdx.x & ~31) : 0);
    float4 *ww = rec_w + (REC ? (threadIdx.x & ~31) : 0);
    const int mypos = rec_pos<G>(lane / G, r);
    const int sP = p.v_sP, sJ = p.l_sJ, sXY = p.l_sXY, NLP = p.NLP;
    int nk = 0;  // chunks this lane owns: k*G + r < chunks (FULL: all NCH)
#pragma unroll
    for (int k = 0; k < NCH; ++k) nk += (FULL || k * G + r < p.chunks);
    const int slog = SPLIT ? p.split_log2 : 0;  // (SPLIT = false: the whole-row kernel, no split code)
    const RowRange rr = block_rows<GPB>(p, slog);
    const int jstep = G << slog;

    for (uint32_t item = rr.beg + threadIdx.x / G; item < rr.end; item += rr.step) {
        const uint32_t row = item >> slog;
        const int part = (int)(item & ((1u << slog) - 1u));
        const Row rw = decode_row(p, row);
        const T *vbh = value + rw.b * p.v_sB + (int64_t)rw.h * p.v_sH + r * VEC;
        const int64_t lo = rw.b * p.l_sB + (int64_t)((rw.q * (uint32_t)p.N_h + rw.h) * (uint32_t)NLP) * sJ;
        const int64_t ao = (int64_t)rw.bqh * NLP;
        const int ldt = GEN ? p.loc_dt : 0;
        const bool logits = GEN && p.logits;
        const float2 sm = logits ? row_softmax_stats<G>(attn, ao, NLP, r, gmask, ldt) : make_float2(0.0f, 1.0f);

        float acc[NCH][VEC];
#pragma unroll
        for (int k = 0; k < NCH; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[k][e] = 0.0f;

        // LA: the next batch's location and weight are loaded before this batch is
        // consumed (measured 1-9% faster)
        constexpr bool LA = REC;
        // BQHLP2 binary32: (x, y) adjacent at an even index, as aligned as loc
        const bool lpair = sXY == 1 && sJ == 2 && ldt == 0 && !(reinterpret_cast<uintptr_t>(loc) & 7u);
        float nu = 0.0f, nv = 0.0f, nA = 0.0f;
        if constexpr (LA) {
            const int j = part * G + r;
            if (j < NLP) {
                ld_uv(loc, lo + j * sJ, sXY, ldt, lpair, nu, nv);
                nA = ldl(attn, ao + j, ldt);
            }
        }
        for (int j0 = part * G; j0 < NLP; j0 += jstep) {
            // owner phase: this lane's sample (past the last sample: weight 0 at offset 0)
            FwdCell mine = {0, 0, 0.0f, 0.0f, 0.0f, 0.0f};
            const int j = j0 + r;
            float cu = nu, cv = nv, cA = nA;
            if constexpr (LA) {
                const int jn = j + jstep;
                if (jn < NLP) {
                    ld_uv(loc, lo + jn * sJ, sXY, ldt, lpair, nu, nv);
                    nA = ldl(attn, ao + jn, ldt);
                }
            }
            if (FULL || j < NLP) {  // (FULL: every batch the loop reaches is whole)
                const float u = LA ? cu : ldl(loc, lo + j * sJ, ldt), v = LA ? cv : ldl(loc, lo + j * sJ + sXY, ldt);
                float A = LA ? cA : ldl(attn, ao + j, ldt);
                if (logits) A = expf(A - sm.x) * sm.y;
                const int l = (int)p.div_p.div((uint32_t)j);
                const float4 gg = lt.geo[l];
                const int W = __float_as_int(gg.z), H = __float_as_int(gg.w);
                const Cell c = make_cell<PAD>(u, v, gg.x, gg.y, p.off, W, H, p.padding);
                if constexpr (REC) {
                    const Corners cr = corners_of(c, A, W, H, lt.start[l], sP);
                    wo[mypos] = make_int4(cr.o[0], cr.o[1], cr.o[2], cr.o[3]);
                    ww[mypos] = make_float4(cr.w[0], cr.w[1], cr.w[2], cr.w[3]);
                } else {
                    mine = fwd_cell(c, A, W, H, lt.start[l], sP);
                }
            } else if constexpr (REC) {
                wo[mypos] = make_int4(0, 0, 0, 0);
                ww[mypos] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
            if constexpr (REC) __syncwarp(gmask);
            // consume phase: the group's samples in order, corners of two in flight
            const int ns = FULL ? G : min(G, NLP - j0);  // (FULL: every batch has G samples)
            // samples in flight for one chunk a lane (MSDA_FWD_INFLIGHT, a divisor of G)
            constexpr int S2 = (G >= 2 && NCH * VEC <= 4) ? (MSDA_FWD_INFLIGHT < G ? MSDA_FWD_INFLIGHT : G) : 1;
#pragma unroll
            for (int s = 0; s < G; s += S2) {
                if constexpr (NCH > 4) {  // wide rows: the same arithmetic, two chunks' corners at a time
                    if (s < ns) {
                        const int src = base + s;
                        const int o0 = __shfl_sync(gmask, mine.o0, src);
                        const int o1 = __shfl_sync(gmask, mine.o1, src);
                        const float w[4] = {__shfl_sync(gmask, mine.w00, src), __shfl_sync(gmask, mine.w01, src),
                                            __shfl_sync(gmask, mine.w10, src), __shfl_sync(gmask, mine.w11, src)};
                        const int dx = (int)((unsigned)o0 >> 31) * sP;
                        const int o[4] = {o0 & 0x7fffffff, (o0 & 0x7fffffff) + dx, o1, o1 + dx};
#pragma unroll
                        for (int k0 = 0; k0 < NCH; k0 += 2) {
                            float x[4][2][VEC];
#pragma unroll
                            for (int i = 0; i < 4; ++i)
#pragma unroll
                                for (int kk = 0; kk < 2; ++kk)
                                    if (k0 + kk < nk) VecIO<T, VEC>::load(vbh + o[i] + (k0 + kk) * G * VEC, x[i][kk]);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
#pragma unroll
                                for (int kk = 0; kk < 2; ++kk)
                                    if (k0 + kk < nk) axpy<VEC>(acc[k0 + kk], w[i], x[i][kk]);
                        }
                    }
                    continue;
                }
                if (s < ns) {
                    int o[S2][4];
                    float w[S2][4];
                    float x[S2][4][NCH][VEC];
#pragma unroll
                    for (int h2 = 0; h2 < S2; ++h2) {
                        static_assert(REC || NCH > 4, "up to four chunks a lane: the record exchange");
                        const int q = rec_pos<G>(lane / G, s + h2);
                        const int4 o4 = wo[q];
                        const float4 w4 = ww[q];
                        o[h2][0] = o4.x;
                        o[h2][1] = o4.y;
                        o[h2][2] = o4.z;
                        o[h2][3] = o4.w;
                        w[h2][0] = w4.x;
                        w[h2][1] = w4.y;
                        w[h2][2] = w4.z;
                        w[h2][3] = w4.w;
#pragma unroll
                        for (int i = 0; i < 4; ++i)
#pragma unroll
                            for (int k = 0; k < NCH; ++k)
                                if (k < nk) VecIO<T, VEC>::load(vbh + o[h2][i] + k * G * VEC, x[h2][i][k]);
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
            if constexpr (REC) __syncwarp(gmask);  // records are rewritten by the next batch
        }
        if constexpr (SPLIT) sum_parts<G, NCH, VEC>(acc, slog, lane);
        T *dst = out + (int64_t)rw.bqh * p.C_h + r * VEC;
        if (part == 0) {
#pragma unroll
            for (int k = 0; k < NCH; ++k)
                if (k < nk) VecIO<T, VEC>::store(dst + k * G * VEC, acc[k]);
        }
    }
}

// ---------------------------------------------------------------- backward
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

// The steps o = N/2, ..., 1 of reduce_scatter on the N = G/2 values left
// after its first step (o = G/2), which the backward takes as soon as each
// pair of samples t, t + G/2 is done (fewer partials live at once).
template <int N>
__device__ __forceinline__ float reduce_scatter_tail(float (&v)[N], int r, unsigned gmask) {
#pragma unroll
    for (int o = N / 2; o >= 1; o >>= 1) {
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

// Tiles of the tile-sorted grad_value.  A sample's cell (top-left corner
// (y0, x0), y0 in [-1, H-1], x0 in [-1, W-1]) has extended coordinates
// (ey, ex) = (y0 + 1, x0 + 1) on an (H+1) x (W+1) grid, cut into tiles of
// kTileCells x kTileCells cells numbered row-major per level after the tiles
// of the levels before it.  bucket_of returns the tile (within the (b, h))
// and, in *cell, the cell's index inside it; -1 when none of the cell's
// corners lies in the map ("zeros" beyond the edge): such a sample adds
// nothing to grad_value.
constexpr int kTileCells = 16;
__device__ __forceinline__ int bucket_of(const Cell &c, int bst, int BX, int *cell) {
    if (!c.valid) return -1;
    const int ey = c.y0 + 1, ex = c.x0 + 1;
    const int ty = ey / kTileCells, tx = ex / kTileCells;
    *cell = (ey - ty * kTileCells) * kTileCells + (ex - tx * kTileCells);
    return bst + ty * BX + tx;
}

// ---------------------------------------------------------------- warp-aggregated grad_value
// A warp serves four rows (neighbouring queries of one head) a batch of eight
// samples each: 32 samples, up to 128 corner contributions A w_i g_row to
// grad_value.  Neighbouring queries sample overlapping neighbourhoods, so many
// of them land on the same pixel (encoder-ordered Deformable-DETR queries:
// about half).  Instead of one 128-byte reduction line per contribution, the
// warp first merges equal pixels in a table of its own in shared memory,
// keyed by the pixel's element offset in the (b, h) slice and holding per
// slot the summed corner weights of each of the four rows; a group then adds,
// for every distinct pixel, the sum over the four rows of weight times that
// row's grad_output with one red.global.add.v4.f32 per lane.  A contribution
// that finds no slot within kAggProbes linear probes is added directly.  When
// a batch has few repeated pixels (random locations), the warp scatters the
// next kAggBackoff batches directly, as the plain kernel does, and then
// measures again.
constexpr int kAggSlots = 256;   // power of two (128: 3% slower, longer probe runs)
constexpr int kAggProbes = 8;
constexpr int kAggBackoff = 64;  // batches
struct AggTable {
    int key[kAggSlots];           // element offset of the pixel in the (b, h) slice; -1 empty
    float4 w[kAggSlots];          // summed A w_i of rows 0..3 of the warp (x, y, z, w)
    unsigned char list[128];      // slots filled in this batch (at most 128), in fill order
};
__device__ __forceinline__ unsigned agg_hash(int key) {
    return ((unsigned)key * 0x9E3779B1u) >> (32 - 8);  // 8 = log2(kAggSlots)
}
static_assert(kAggSlots == 256, "agg_hash takes the top 8 bits");

// One batch of a warp's merged grad_value scatter (the AGG backward below);
// every lane of the warp calls it.  (o4, w4): this lane's own sample record
// (all weights 0 for no sample); g: chunk r of this lane's row of
// grad_output; bqh / active: this lane's row and whether it has one.
// Returns (contributions << 8) | distinct pixels of the batch.
template <typename T>
__device__ __forceinline__ int agg_scatter(AggTable &tab, int4 o4, float4 w4, int grp, int r, int nk, float *gbh,
                                           const float (&g)[4], const T *grad_out, uint32_t bqh, bool active,
                                           int C_h) {
    const int lane = threadIdx.x & 31;
    const int gbase = lane & ~7;
    const unsigned below = (1u << lane) - 1u;
    const unsigned gmask = 0xffu << gbase;
    const int key4[4] = {o4.x, o4.y, o4.z, o4.w};
    const float wt4[4] = {w4.x, w4.y, w4.z, w4.w};
    // insert the four corners: the table sums each row's weights per pixel;
    // the four first probes go out back to back, collisions probe on after
    int nrec = 0, ncon = 0;
    unsigned ovf = 0;  // corners of this lane that found no slot
    bool want[4];
    unsigned sl[4];
    int old[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        want[i] = wt4[i] != 0.0f;
        sl[i] = agg_hash(key4[i]);
        old[i] = want[i] ? atomicCAS(&tab.key[sl[i]], -1, key4[i]) : -1;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        bool fresh = false;
        if (want[i]) {
            bool placed = old[i] == -1 || old[i] == key4[i];
            fresh = old[i] == -1;
            unsigned s = sl[i];
            for (int t = 1; t < kAggProbes && !placed; ++t) {
                s = (s + 1) & (kAggSlots - 1);
                const int o2 = atomicCAS(&tab.key[s], -1, key4[i]);
                placed = o2 == -1 || o2 == key4[i];
                fresh = o2 == -1;
            }
            sl[i] = s;
            if (placed) atomicAdd(reinterpret_cast<float *>(&tab.w[s]) + grp, wt4[i]);
            else ovf |= 1u << i;
        }
        const unsigned nm = __ballot_sync(0xffffffffu, fresh);
        if (fresh) tab.list[nrec + __popc(nm & below)] = (unsigned char)sl[i];
        nrec += __popc(nm);
        ncon += __popc(__ballot_sync(0xffffffffu, want[i]));
    }
    // contributions that found no slot: their row's group adds them directly
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        unsigned om = (__ballot_sync(0xffffffffu, (ovf >> i) & 1u) >> gbase) & 0xffu;
        while (om) {  // uniform over the group
            const int src = gbase + __ffs(om) - 1;
            om &= om - 1;
            const int key = __shfl_sync(gmask, key4[i], src);
            const float wt = __shfl_sync(gmask, wt4[i], src);
            if (nk) RedIO<4>::add(gbh + key, g, wt);
        }
    }
    // chunk r of the four rows' grad_output (zero for a group without a row)
    float G4[4][4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const uint32_t rb = __shfl_sync(0xffffffffu, bqh, b * 8);
        const bool ab = __shfl_sync(0xffffffffu, (int)active, b * 8) != 0;
        if (ab && nk) {
            VecIO<T, 4>::load(grad_out + (int64_t)rb * C_h + r * 4, G4[b]);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) G4[b][e] = 0.0f;
        }
    }
    __syncwarp();
    // one reduction line per distinct pixel; group grp takes every fourth
    for (int t = grp; t < nrec; t += 4) {
        const int s = tab.list[t];
        const int key = tab.key[s];
        const float4 ws = tab.w[s];
        float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        axpy<4>(a, ws.x, G4[0]);
        axpy<4>(a, ws.y, G4[1]);
        axpy<4>(a, ws.z, G4[2]);
        axpy<4>(a, ws.w, G4[3]);
        if (nk) red_add_v4(gbh + key, a[0], a[1], a[2], a[3]);
    }
    __syncwarp();
    for (int t = lane; t < nrec; t += 32) {  // empty the slots for the next batch
        const int s = tab.list[t];
        tab.key[s] = -1;
        tab.w[s] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    return (ncon << 8) | nrec;
}

// The backward reuses the forward's work split: a group of G lanes per row,
// samples taken G at a time, lane r computing sample j0 + r's cell once and
// publishing its record (corner offsets, weights A w_i).  With grad_output's
// row g in registers (lane r holds its channel chunks), each lane forms, for
// every sample of the batch, its part of d_i = <g, V_i> at the four corners;
// a transposed butterfly leaves lane r with sample r's totals, from which it
// computes, with its own cell's fractions,
//   <g, S>     = sum_i w_i d_i        -> grad_attention_weights
//   <g, dS/dx> = sum_i dw_i/dx d_i     -> grad_sampling_locations.x = A sx <g, dS/dx>
//   <g, dS/dy> = sum_i dw_i/dy d_i     -> grad_sampling_locations.y = A sy <g, dS/dy>
// (corners outside the map read 0: their d_i count as 0).  grad_value, when
// requested here, receives A w_i g at corner i in the binary32 accumulator:
// AGG = false, one red.global.add.v4.f32 per lane and corner; AGG = true
// (four rows a warp, one chunk a lane), merged per warp and batch as above.
// (The tile-sorted grad_value runs this kernel without kGradValue.)
// FL: kGradValue|kGradLoc|kGradAttn or kGradValue (exactly these outputs),
// kGradLoc|kGradAttn (no grad_value; the two others as p.flags says), or -1
// (everything from p.flags at run time).  PAD and FULL as in the forward.
#ifndef MSDA_AGG_MIN_BLOCKS
#define MSDA_AGG_MIN_BLOCKS MSDA_BWD_MIN_BLOCKS
#endif
// Without grad_value a lane keeps no scatter state: with the paired exchange
// one chunk a lane fits 4 blocks per SM (64 registers), measured 6% faster
// than 3 on the bfloat16 workloads and equal on the binary32 one.
#ifndef MSDA_LOCATTN_MIN_BLOCKS
#define MSDA_LOCATTN_MIN_BLOCKS 4
#endif
__host__ __device__ constexpr int bwd_min_blocks(int elems, int fl, bool agg) {
    return agg ? MSDA_AGG_MIN_BLOCKS
               : (fl == (kGradLoc | kGradAttn) && elems <= 4) ? MSDA_LOCATTN_MIN_BLOCKS : row_min_blocks(elems, false);
}
template <typename T, int VEC, int G, int NCH, int PAD, int FL, bool SPLIT, bool AGG, bool FULL>
__global__ void __launch_bounds__(kThreads, bwd_min_blocks(NCH *VEC, FL, AGG))
msda_backward_kernel(const __grid_constant__ Params p, const T *__restrict__ grad_out, const T *__restrict__ value,
                     const float *__restrict__ loc, const float *__restrict__ attn, float *__restrict__ gv_acc,
                     float *__restrict__ grad_loc, float *__restrict__ grad_attn) {
    static_assert(!AGG || (G == 8 && NCH == 1 && VEC == 4 && !SPLIT), "aggregation: four rows a warp, one chunk a lane");
    __shared__ LevelTables lt;
    __shared__ int4 rec_o[kThreads];
    __shared__ float4 rec_w[kThreads];
    __shared__ AggTable agg_tables[AGG ? kThreads / 32 : 1];
    load_level_tables(p, lt);
    constexpr int GPB = kThreads / G;
    const int flags = FL < 0 ? p.flags : (FL == (kGradLoc | kGradAttn) ? (p.flags & FL) : FL);
    const bool want_gv = flags & kGradValue, want_gl = flags & kGradLoc, want_ga = flags & kGradAttn;
    const bool need_v = want_gl || want_ga;  // value is read only for these two
    // attention is read only for these two, and for the logits' gradient
    const bool need_a = want_gv || want_gl || (p.logits && want_ga);
    const bool scatter = want_gv;            // consumers add into grad_value
    const int lane = threadIdx.x & 31;
    const int r = lane & (G - 1);
    const int grp = lane / G;
    const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane & ~(G - 1)));
    int4 *wo = rec_o + (threadIdx.x & ~31);
    float4 *ww = rec_w + (threadIdx.x & ~31);
    const int mypos = rec_pos<G>(grp, r);
    const int sP = p.v_sP, sJ = p.l_sJ, sXY = p.l_sXY, NLP = p.NLP;
    const bool lpair = sXY == 1 && sJ == 2 && p.loc_dt == 0 && !(reinterpret_cast<uintptr_t>(loc) & 7u);
    const bool gpair = sXY == 1 && sJ == 2 && p.loc_dt == 0 && !(reinterpret_cast<uintptr_t>(grad_loc) & 7u);
    int nk = 0;  // chunks this lane owns: k*G + r < chunks (FULL: all NCH)
#pragma unroll
    for (int k = 0; k < NCH; ++k) nk += (FULL || k * G + r < p.chunks);
    // split only without logits (the rewrite below needs whole rows); SPLIT = false: no split code
    const int slog = SPLIT ? p.split_log2 : 0;
    const RowRange rr = block_rows<GPB>(p, slog);
    const int jstep = G << slog;
    AggTable &tab = agg_tables[AGG ? (threadIdx.x >> 5) : 0];
    if constexpr (AGG) {
        for (int i = lane; i < kAggSlots; i += 32) {
            tab.key[i] = -1;
            tab.w[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        __syncwarp();
    }
    int direct_left = 0;  // (AGG) batches the warp still scatters directly

    // AGG: the four groups of a warp run the same iterations (warp-wide
    // exchanges); a group past the last row runs along without samples.
    for (uint32_t lead = rr.beg + (AGG ? (threadIdx.x >> 5) * (32 / G) : threadIdx.x / G); lead < rr.end;
         lead += rr.step) {
        const uint32_t item = AGG ? lead + grp : lead;
        const bool active = !AGG || item < rr.end;
        const uint32_t row = (active ? item : lead) >> slog;
        const int part = (int)(item & ((1u << slog) - 1u));
        const Row rw = decode_row(p, row);
        const int64_t bhoff = rw.b * p.v_sB + (int64_t)rw.h * p.v_sH;
        const T *vbh = value + bhoff + r * VEC;
        float *gbh = gv_acc + bhoff + r * VEC;
        const int64_t lrow = rw.b * p.l_sB + (int64_t)((rw.q * (uint32_t)p.N_h + rw.h) * (uint32_t)NLP) * sJ;
        const int64_t ao = (int64_t)rw.bqh * NLP;  // row of attention_weights and its gradient
        const bool soft = p.logits && need_a;
        const float2 sm =
            soft ? row_softmax_stats<G>(attn, ao, NLP, r, gmask, p.loc_dt) : make_float2(0.0f, 1.0f);
        float sAg = 0.0f;  // (logits) this lane's part of sum_j A_j <g, S_j>
        float g[NCH][VEC];
        {
            const T *src = grad_out + (int64_t)rw.bqh * p.C_h + r * VEC;
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
        // (AGG) the warp's rows share one (b, h) slice, so pixel offsets are
        // comparable keys; a warp straddling two heads scatters directly
        bool merge = false;
        if constexpr (AGG) {
            const uint32_t bh = rw.b * (uint32_t)p.N_h + rw.h;
            const uint32_t bh0 = __shfl_sync(0xffffffffu, bh, 0);  // every lane takes part in the shuffle
            merge = __all_sync(0xffffffffu, !active || bh == bh0) && scatter;
        }

        for (int j0 = part * G; j0 < NLP; j0 += jstep) {
            const bool agg_now = AGG && merge && direct_left == 0;  // uniform over the warp
            // owner phase: this lane's sample
            const int j = j0 + r;
            const bool live = active && (FULL || j < NLP);
            int l = 0;
            float A = 0.0f;
            Cell c;
            {
                Corners cr = {{0, 0, 0, 0}, {0.0f, 0.0f, 0.0f, 0.0f}};
                float u = 0.0f, v = 0.0f;
                if (live) {
                    l = (int)p.div_p.div((uint32_t)j);
                    ld_uv(loc, lrow + j * sJ, sXY, p.loc_dt, lpair, u, v);
                    if (need_a) A = ldl(attn, ao + j, p.loc_dt);
                    if (soft) A = expf(A - sm.x) * sm.y;
                }
                const float4 gg = lt.geo[l];
                const int W = __float_as_int(gg.z), H = __float_as_int(gg.w);
                c = make_cell<PAD>(u, v, gg.x, gg.y, p.off, W, H, p.padding);
                if (live) cr = corners_of(c, A, W, H, lt.start[l], sP);
                wo[mypos] = make_int4(cr.o[0], cr.o[1], cr.o[2], cr.o[3]);
                ww[mypos] = make_float4(cr.w[0], cr.w[1], cr.w[2], cr.w[3]);
            }
            if constexpr (AGG) __syncwarp();
            else __syncwarp(gmask);
            // consume phase: the group's samples, in order or (PAIRED) in pairs
            // t, t + G/2, whose first butterfly exchange is taken at once
            const int ns = active ? (FULL ? G : min(G, NLP - j0)) : 0;
            // (measured: the full backward 6-8% faster; it also lets the kernel
            // without grad_value fit 4 blocks per SM)
            constexpr bool PAIRED = G == 8;
            float pd[4][(G <= 8 && !PAIRED) ? G : 1];  // this lane's part of d_i, per sample of the batch
            float ph[4][PAIRED ? G / 2 : 1];           // (PAIRED) the same after the first exchange
            float dprev[4] = {0.0f, 0.0f, 0.0f, 0.0f}; // (PAIRED) sample t of the pair being formed
            float dt[4] = {0.0f, 0.0f, 0.0f, 0.0f};    // (G > 8) totals of this lane's own sample
#pragma unroll
            for (int u = 0; u < G; ++u) {
                const int s = PAIRED ? ((u >> 1) + (u & 1) * (G / 2)) : u;
                float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                if (s < ns) {
                    const int q = rec_pos<G>(grp, s);
                    const int4 o4 = wo[q];
                    const int oo[4] = {o4.x, o4.y, o4.z, o4.w};
                    if (need_v) {
                        // (wide rows: two chunks' corners at a time; each d_i still sums chunk by chunk)
                        constexpr int KB = NCH > 2 ? 2 : NCH;
                        // d_i in two interleaved partial sums (even and odd channels) by packed FMAs
                        float2 dp[4] = {{0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}};
#pragma unroll
                        for (int k0 = 0; k0 < NCH; k0 += KB) {
                            float x[4][KB][VEC];
#pragma unroll
                            for (int i = 0; i < 4; ++i)
#pragma unroll
                                for (int kk = 0; kk < KB; ++kk)
                                    if (k0 + kk < nk) VecIO<T, VEC>::load(vbh + oo[i] + (k0 + kk) * G * VEC, x[i][kk]);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
#pragma unroll
                                for (int kk = 0; kk < KB; ++kk)
                                    if (k0 + kk < nk) dot_acc<VEC>(dp[i], g[k0 + kk], x[i][kk]);
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) d[i] = dp[i].x + dp[i].y;
                    }
                    if (scatter && !agg_now) {
                        const float4 w4 = ww[q];
                        const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (wv[i] != 0.0f)
#pragma unroll
                                for (int k = 0; k < NCH; ++k)
                                    if (k < nk) RedIO<VEC>::add(gbh + oo[i] + k * G * VEC, g[k], wv[i]);
                    }
                }
                if constexpr (PAIRED) {
                    if (!(u & 1)) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) dprev[i] = d[i];
                    } else if (need_v) {  // reduce_scatter's first step for samples t and t + G/2
                        const int t = u >> 1;
                        const bool up = (r & (G / 2)) != 0;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float send = up ? dprev[i] : d[i];
                            const float keep = up ? d[i] : dprev[i];
                            ph[i][t] = keep + __shfl_xor_sync(gmask, send, G / 2);
                        }
                    }
                } else if constexpr (G <= 8) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) pd[i][s] = d[i];
                } else if (need_v) {  // wide groups: sum per sample, the owner keeps it
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
            if (need_v) {
                if constexpr (PAIRED) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) dt[i] = reduce_scatter_tail<G / 2>(ph[i], r, gmask);
                } else if constexpr (G <= 8) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) dt[i] = reduce_scatter<G>(pd[i], r, gmask);
                }
                if (live) {
                    // weights without A and their derivatives; corners outside the map read 0
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
                    if (want_ga) stl(grad_attn, ao + j, ga, p.loc_dt);  // (logits: <g, S_j>, made d/dlogit below)
                    if (soft) sAg = fmaf(A, ga, sAg);
                    if (want_gl) {
                        const float2 sxy = *reinterpret_cast<const float2 *>(&lt.geo[l]);
                        st_uv(grad_loc, lrow + j * sJ, sXY, p.loc_dt, gpair, A * tx * (sxy.x * c.kx),
                              A * ty * (sxy.y * c.ky));
                    }
                }
            }
            if constexpr (AGG) {
                if (agg_now) {
                    const int nc = agg_scatter<T>(tab, wo[mypos], ww[mypos], grp, r, nk, gbh, g[0], grad_out, rw.bqh,
                                                  active, p.C_h);
                    // nc: (contributions << 8) | distinct pixels of this batch
                    if ((nc & 0xff) * 5 > (nc >> 8) * 4) direct_left = kAggBackoff;  // under 1.25 per pixel
                } else if (direct_left > 0) {
                    --direct_left;
                }
                __syncwarp();  // records are rewritten by the next batch
            } else {
                __syncwarp(gmask);
            }
        }
        if (soft && want_ga && active) {
            // d/dlogit_j = A_j (<g, S_j> - sum_k A_k <g, S_k>); lane r rewrites the
            // samples it stored above
#pragma unroll
            for (int o = G / 2; o >= 1; o >>= 1) sAg += __shfl_xor_sync(gmask, sAg, o);
            for (int j = r; j < NLP; j += G) {
                const float A = expf(ldl(attn, ao + j, p.loc_dt) - sm.x) * sm.y;
                stl(grad_attn, ao + j, A * (ldl_own(grad_attn, ao + j, p.loc_dt) - sAg), p.loc_dt);
            }
        }
    }
}

// ---------------------------------------------------------------- tile-sorted grad_value
// grad_value[pixel] = sum over samples s and corners i of s's cell at that
// pixel of A_s w_i(s) g_{row(s)}.  Scattered one corner at a time this is four
// C_h-wide binary32 reduction lines per sample, and the GPU's reduction rate
// (about 6.7 TB/s of payload, one 128-byte line per ~6 SM cycles) bounds the
// backward.  The tile-sorted path first groups the samples by cell and sums
// each cell's samples in registers, so a cell costs four reduction lines per
// run of its samples instead of four per sample:
//   1. msda_tile_count_kernel   counts[tile][part]: samples of partition block
//                               `part` (a run of rows) in tile `tile`
//                               (kTileCells^2 cells of one level and (b, h)),
//                               counted in shared memory: no global atomics
//   2. scan                     offsets = exclusive prefix sum of the counts in
//                               (tile, part) order: a tile's samples become one
//                               contiguous range, split by partition block
//   3. msda_tile_items_kernel   chunks[tile] = ceil(samples of tile / kChunk),
//      scan                     then chunk offsets
//   4. msda_tile_append_kernel  each partition block writes its samples'
//                               entries (row | cell << 24, A - A fx, A fx, fy) into its
//                               own slots of each tile (shared cursors)
//   5. msda_tile_reduce_kernel  one block per chunk of a tile: counting sort of
//                               the chunk's entries by cell in shared memory;
//                               each group of G lanes sweeps an equal share of
//                               the sorted entries with several grad_output
//                               rows in flight, sums each cell's samples times
//                               its four corner weights in registers and adds
//                               them to the accumulator when the cell changes
//                               (red.global.add.v4.f32).
// It is used for calls whose only output is grad_value: next to the other two
// gradients, the fused row kernel overlaps the direct atomics with the value
// gather and is faster.
// Within a (tile, part) segment entries are in shared-atomic order, so
// grad_value's summation order (not its value) varies from call to call.
#ifndef MSDA_REDUCE_ROWS
#define MSDA_REDUCE_ROWS 6
#endif
constexpr int kChunk = 4096;         // entries of one reduction block
constexpr int kEntryCellShift = 24;  // entry.x = row | cell << 24 (rows < 2^24, cells < 2^8)
static_assert(kTileCells * kTileCells <= (1 << (32 - kEntryCellShift)), "cell index must fit above the row");

// Exclusive prefix sum of n int32 counts, in tiles of kScanTile: pass 1 sums
// each tile, pass 2 scans each tile after the sums of the tiles before it, in
// place (counts become offsets), and writes the grand total to offsets[n].
constexpr int kScanThreads = 1024;
constexpr int kScanPer = 4;
constexpr int kScanTile = kScanThreads * kScanPer;
__global__ void msda_scan_tiles_kernel(const int *__restrict__ counts, uint32_t n, int *__restrict__ tile_sums);
__global__ void msda_scan_apply_kernel(int *__restrict__ offsets, uint32_t n, const int *__restrict__ tile_sums);

// The tile of one sample of row `row` (rows in (b, h, q) order), its cell in
// the tile, and the sample's cell fractions; -1 when it adds nothing.
template <int PAD>
__device__ __forceinline__ int tile_of_sample(const Params &p, const LevelTables &lt, const float *loc, uint32_t row,
                                              int j, int *cell, Cell *cout, uint32_t *bh_out, uint32_t *bqh_out) {
    const Row rw = decode_row(p, row);
    const int64_t lo = rw.b * p.l_sB + (int64_t)((rw.q * (uint32_t)p.N_h + rw.h) * (uint32_t)p.NLP + j) * p.l_sJ;
    const int l = (int)p.div_p.div((uint32_t)j);
    const int W = lt.W[l], H = lt.H[l];
    const Cell c = make_cell<PAD>(ldl(loc, lo, p.loc_dt), ldl(loc, lo + p.l_sXY, p.loc_dt), lt.sx[l], lt.sy[l], p.off,
                                  W, H, p.padding);
    *cout = c;
    *bh_out = rw.b * (uint32_t)p.N_h + rw.h;
    *bqh_out = rw.bqh;
    return bucket_of(c, lt.bst[l], lt.BX[l], cell);
}

// Partition block `part` owns rows [part * part_rows, +part_rows) of the
// (b, h, q) order; their samples fall in the tiles of at most p.span (b, h)
// pairs, the first being (first row) / N_q.  Shared memory: p.span * p.NB ints.
template <int PAD>
__global__ void __launch_bounds__(256)
msda_tile_count_kernel(const __grid_constant__ Params p, const float *__restrict__ loc, int *__restrict__ counts) {
    extern __shared__ int hist[];
    __shared__ LevelTables lt;
    load_level_tables(p, lt);
    const uint32_t part = blockIdx.x;
    const uint32_t r0 = part * p.part_rows;
    const uint32_t r1 = min(p.rows, r0 + p.part_rows);
    if (r0 >= r1) return;  // uniform over the block
    const uint32_t bh0 = p.div_q.div(r0);
    for (int i = threadIdx.x; i < p.span * p.NB; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const uint32_t n = (r1 - r0) * (uint32_t)p.NLP;
    for (uint32_t t = threadIdx.x; t < n; t += blockDim.x) {
        const uint32_t row = r0 + p.div_nlp.div(t);
        const int j = (int)(t - (row - r0) * (uint32_t)p.NLP);
        int cell;
        Cell c;
        uint32_t bh, bqh;
        const int tile = tile_of_sample<PAD>(p, lt, loc, row, j, &cell, &c, &bh, &bqh);
        if (tile >= 0) atomicAdd(hist + (int)(bh - bh0) * p.NB + tile, 1);
    }
    __syncthreads();
    // every (tile, part) count of this block's (b, h) range, zeros included
    const int here = (int)(p.div_q.div(r1 - 1) - bh0 + 1) * p.NB;
    for (int i = threadIdx.x; i < here; i += blockDim.x)
        counts[(size_t)(bh0 * (uint32_t)p.NB + (uint32_t)i) * p.parts + part] = hist[i];
}

// chunks[tile] = ceil(samples of tile / kChunk); offsets are in (tile, part) order.
__global__ void msda_tile_items_kernel(const __grid_constant__ Params p, const int *__restrict__ offsets,
                                       int *__restrict__ chunks);

template <int PAD>
__global__ void __launch_bounds__(256)
msda_tile_append_kernel(const __grid_constant__ Params p, const float *__restrict__ loc,
                        const float *__restrict__ attn, const int *__restrict__ offsets,
                        uint4 *__restrict__ entries) {
    extern __shared__ int cur[];  // p.span * p.NB
    __shared__ LevelTables lt;
    load_level_tables(p, lt);
    const uint32_t part = blockIdx.x;
    const uint32_t r0 = part * p.part_rows;
    const uint32_t r1 = min(p.rows, r0 + p.part_rows);
    if (r0 >= r1) return;
    const uint32_t bh0 = p.div_q.div(r0);
    const int here = (int)(p.div_q.div(r1 - 1) - bh0 + 1) * p.NB;
    for (int i = threadIdx.x; i < here; i += blockDim.x)
        cur[i] = offsets[(size_t)(bh0 * (uint32_t)p.NB + (uint32_t)i) * p.parts + part];
    __syncthreads();
    const uint32_t n = (r1 - r0) * (uint32_t)p.NLP;
    for (uint32_t t = threadIdx.x; t < n; t += blockDim.x) {
        const uint32_t row = r0 + p.div_nlp.div(t);
        const int j = (int)(t - (row - r0) * (uint32_t)p.NLP);
        int cell;
        Cell c;
        uint32_t bh, bqh;
        const int tile = tile_of_sample<PAD>(p, lt, loc, row, j, &cell, &c, &bh, &bqh);
        if (tile >= 0) {
            float A = ldl(attn, (int64_t)bqh * p.NLP + j, p.loc_dt);
            if (p.logits) {  // softmax over the row's logits (recomputed per sample: rows are short)
                float m = -INFINITY, sum = 0.0f;
                for (int k = 0; k < p.NLP; ++k) m = fmaxf(m, ldl(attn, (int64_t)bqh * p.NLP + k, p.loc_dt));
                for (int k = 0; k < p.NLP; ++k) sum += expf(ldl(attn, (int64_t)bqh * p.NLP + k, p.loc_dt) - m);
                A = expf(A - m) * (1.0f / sum);
            }
            const uint32_t slot = (uint32_t)atomicAdd(cur + (int)(bh - bh0) * p.NB + tile, 1);
            if (slot < p.capacity) {
                const float A1 = A * c.fx;  // the x factors of the corner weights, formed once per entry
                entries[slot] = make_uint4(bqh | ((uint32_t)cell << kEntryCellShift), __float_as_uint(A - A1),
                                           __float_as_uint(A1), __float_as_uint(c.fy));
            }
        }
    }
}

// Shared memory of msda_tile_reduce_kernel: the chunk's entries and their order.
constexpr size_t kTileReduceSmem = (size_t)kChunk * sizeof(uint4) + (size_t)kChunk * sizeof(uint16_t);

// 3 blocks per SM (the shared memory allows no more) for one channel chunk a
// lane; fewer for wider rows, whose 4 x NCH x VEC accumulators a lane need the
// registers.
template <typename T, int VEC, int G, int NCH>
__global__ void __launch_bounds__(256, NCH >= 4 ? 1 : NCH == 2 ? 2 : 3)
msda_tile_reduce_kernel(const __grid_constant__ Params p, const T *__restrict__ grad_out,
                        const int *__restrict__ offsets, const int *__restrict__ chunk_start,
                        const uint4 *__restrict__ entries, float *__restrict__ gv_acc) {
    constexpr int GPB = 256 / G;
    constexpr int NCELL = kTileCells * kTileCells;
    extern __shared__ __align__(16) unsigned char smem[];
    uint4 *ent = reinterpret_cast<uint4 *>(smem);
    uint16_t *order = reinterpret_cast<uint16_t *>(ent + kChunk);
    __shared__ int ccount[NCELL];
    __shared__ int s_tile, s_k;

    const int total_items = chunk_start[p.nbins];
    if ((int)blockIdx.x >= total_items) return;  // uniform over the block
    if (threadIdx.x == 0) {  // the tile whose chunks include this block: last tile with chunk_start <= item
        uint32_t lo = 0, hi = p.nbins;  // chunk_start[lo] <= item < chunk_start[hi]
        while (hi - lo > 1) {
            const uint32_t mid = (lo + hi) / 2;
            if (chunk_start[mid] <= (int)blockIdx.x) lo = mid;
            else hi = mid;
        }
        s_tile = (int)lo;
        s_k = (int)blockIdx.x - chunk_start[lo];
    }
    for (int i = threadIdx.x; i < NCELL; i += blockDim.x) ccount[i] = 0;
    __syncthreads();
    const uint32_t tile = (uint32_t)s_tile;
    const int e0 = offsets[(size_t)tile * p.parts] + s_k * kChunk;
    const int ne = min(offsets[(size_t)(tile + 1) * p.parts], e0 + kChunk) - e0;
    // the tile's (b, h), level and position
    const uint32_t bh = tile / (uint32_t)p.NB;
    const int lb = (int)(tile - bh * (uint32_t)p.NB);
    int l = 0;
    while (l + 1 < p.N_l && p.bst[l + 1] <= lb) ++l;
    const int rel = lb - p.bst[l];
    const int ty = rel / p.BX[l], tx = rel - ty * p.BX[l];
    const int W = p.W[l], H = p.H[l];
    const int y_org = ty * kTileCells - 1, x_org = tx * kTileCells - 1;  // pixel of cell (0,0)'s top-left corner

    // counting sort of the chunk's entries by cell
    for (int i = threadIdx.x; i < ne; i += blockDim.x) {
        const uint4 e = __ldg(entries + e0 + i);
        ent[i] = e;
        atomicAdd(ccount + (int)(e.x >> kEntryCellShift), 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {  // exclusive scan of the NCELL counts, NCELL/32 per lane
        int v[NCELL / 32], sum = 0;
#pragma unroll
        for (int i = 0; i < NCELL / 32; ++i) {
            v[i] = ccount[threadIdx.x * (NCELL / 32) + i];
            sum += v[i];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if ((int)threadIdx.x >= o) incl += y;
        }
        int run = incl - sum;
#pragma unroll
        for (int i = 0; i < NCELL / 32; ++i) {
            ccount[threadIdx.x * (NCELL / 32) + i] = run;  // becomes the cell's cursor
            run += v[i];
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < ne; i += blockDim.x)
        order[atomicAdd(ccount + (int)(ent[i].x >> kEntryCellShift), 1)] = (uint16_t)i;
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int r = lane & (G - 1);
    const int grp = threadIdx.x / G;
    int nk = 0;
#pragma unroll
    for (int k = 0; k < NCH; ++k) nk += (k * G + r < p.chunks);
    const T *gbase = grad_out + r * VEC;
    const uint32_t b = p.div_h.div(bh), h = bh - b * (uint32_t)p.N_h;
    float *gb = gv_acc + b * p.v_sB + (int64_t)h * p.v_sH + r * VEC;
    // Each group sweeps an equal share of the cell-sorted entries with U
    // grad_output rows in flight, summing the current cell's samples in
    // registers, and adds the four corner sums to the accumulator when the cell
    // changes.
    const int s_beg = (int)(((int64_t)ne * grp) / GPB), s_end = (int)(((int64_t)ne * (grp + 1)) / GPB);
    float acc[4][NCH][VEC];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int k = 0; k < NCH; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[i][k][e] = 0.0f;
    int cur_cell = -1;
    auto flush = [&]() {  // the current cell's four corner sums, corners in the map only
        if (cur_cell < 0) return;
        const int cy = cur_cell / kTileCells, cx = cur_cell - cy * kTileCells;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int y = y_org + cy + (i >> 1), x = x_org + cx + (i & 1);
            if ((unsigned)y < (unsigned)H && (unsigned)x < (unsigned)W) {
                float *dst = gb + (int64_t)(p.start[l] + y * W + x) * p.v_sP;
#pragma unroll
                for (int k = 0; k < NCH; ++k)
                    if (k < nk) RedIO<VEC>::add_sum(dst + k * G * VEC, acc[i][k]);
            }
#pragma unroll
            for (int k = 0; k < NCH; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[i][k][e] = 0.0f;
        }
    };
    // grad_output rows in flight a group (one chunk a lane: MSDA_REDUCE_ROWS; wider rows: 32 registers of them)
    constexpr int U = NCH >= 8 ? 1 : (NCH == 1 ? MSDA_REDUCE_ROWS : 8 / NCH);
    for (int s0 = s_beg; s0 < s_end; s0 += U) {
        int ei[U];
        float gv[U][NCH][VEC];
#pragma unroll
        for (int t = 0; t < U; ++t) {
            ei[t] = s0 + t < s_end ? (int)order[s0 + t] : -1;
            uint32_t row = ei[t] >= 0 ? (ent[ei[t]].x & ((1u << kEntryCellShift) - 1u)) : 0u;
            if (row >= p.rows) row = 0;  // an entry's row is always < rows
#pragma unroll
            for (int k = 0; k < NCH; ++k)
                if (k < nk) VecIO<T, VEC>::load(gbase + (int64_t)row * p.C_h + k * G * VEC, gv[t][k]);
        }
#pragma unroll
        for (int t = 0; t < U; ++t) {
            if (ei[t] >= 0) {
                const uint4 en = ent[ei[t]];
                const int cell = (int)(en.x >> kEntryCellShift);
                if (cell != cur_cell) {
                    flush();
                    cur_cell = cell;
                }
                const float ax0 = __uint_as_float(en.y), ax1 = __uint_as_float(en.z), fy = __uint_as_float(en.w);
                const float ay0 = 1.0f - fy, ay1 = fy;
                const float w[4] = {ay0 * ax0, ay0 * ax1, ay1 * ax0, ay1 * ax1};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int k = 0; k < NCH; ++k)
                        if (k < nk)
#pragma unroll
                            for (int e = 0; e < VEC; ++e) acc[i][k][e] = fmaf(w[i], gv[t][k][e], acc[i][k][e]);
            }
        }
    }
    flush();
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

// Buffers of the backward: the binary32 grad_value accumulator and, for the
// tile-sorted grad_value, the (tile, part) counts / offsets (nbins * parts + 1),
// the per-tile chunk counts / offsets (nbins + 1), the scans' tile sums and the
// entries (capacity).
struct BwdBuffers {
    float *gv_acc;
    float *grad_loc, *grad_attn;
    int *offsets, *chunks, *tile_sums;
    uint4 *entries;
};
template <typename T, int PAD>
cudaError_t launch_backward_pad(const Params &p, int G, int NCH, const T *grad_out, const T *value,
                                const float *loc, const float *attn, const BwdBuffers &bb, cudaStream_t stream);
// Dispatch on vector path / padding to the launch_backward_pad instantiations.
template <typename T>
inline cudaError_t launch_backward(const Params &p, bool vec, int G, int NCH, const T *grad_out, const T *value,
                                   const float *loc, const float *attn, const BwdBuffers &bb, cudaStream_t stream) {
    if (p.rows == 0) return cudaSuccess;
    if (!vec) return launch_backward_pad<T, -1>(p, G, NCH, grad_out, value, loc, attn, bb, stream);
    if (p.padding == 0) return launch_backward_pad<T, 0>(p, G, NCH, grad_out, value, loc, attn, bb, stream);
    return launch_backward_pad<T, 1>(p, G, NCH, grad_out, value, loc, attn, bb, stream);
}
// Tile-sorted grad_value, steps 1-4 (count, scans, chunks, append) and 5 (reduce).
cudaError_t launch_tile_partition(const Params &p, const float *loc, const float *attn, const BwdBuffers &bb,
                                  cudaStream_t stream);
template <typename T, bool VECTOR>
cudaError_t launch_tile_reduce(const Params &p, int G, int NCH, const T *grad_out, const BwdBuffers &bb,
                               cudaStream_t stream);
cudaError_t launch_zero_f32(float *p, int64_t n, cudaStream_t stream);
cudaError_t launch_f32_to_bf16(const float *acc, __nv_bfloat16 *out, int64_t n, cudaStream_t stream);

}  // namespace msda
