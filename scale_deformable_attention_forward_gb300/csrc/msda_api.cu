// msda_api.cu -- the C ABI declared in include/msda.h: argument validation,
// kernel parameter set-up and dispatch, plus the two small helper kernels
// (accumulator zero-fill and binary32 -> bfloat16 conversion).
#include "msda.h"
#include "msda_entry.h"
#include "msda_kernels.cuh"
#include "msda_shape.cuh"
#include "msda_staged.cuh"

#include <cudaTypedefs.h>
#include <limits.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>

namespace {

using msda::Params;

thread_local int g_last_cuda_error = 0;

constexpr int64_t kIndexLimit = INT32_MAX;  // 32-bit index arithmetic inside the kernels

int record_cuda(cudaError_t e) {
    if (e == cudaSuccess) return MSDA_OK;
    g_last_cuda_error = (int)e;
    return MSDA_ERR_CUDA;
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

size_t value_elem_size(const msda_desc *d) { return d->value_dtype == MSDA_DTYPE_BF16 ? 2 : 4; }
size_t loc_elem_size(const msda_desc *d) { return d->loc_dtype == MSDA_DTYPE_F32 ? 4 : 2; }

// Shape, enum and level checks shared by every entry point ("MS Deformable
// Attention Kernel API Reference", Parameters: spatial_shapes,
// level_start_index; Dimensions: L is the sum of H_i * W_i).
int validate_desc(const msda_desc *d) {
    if (!d) return MSDA_ERR_NULL_POINTER;
    if (d->value_layout != MSDA_LAYOUT_BLNC && d->value_layout != MSDA_LAYOUT_BNLC) return MSDA_ERR_BAD_ENUM;
    if (d->loc_layout != MSDA_LAYOUT_BQHLP2 && d->loc_layout != MSDA_LAYOUT_B2QHLP) return MSDA_ERR_BAD_ENUM;
    if (d->padding_mode != MSDA_PADDING_ZEROS && d->padding_mode != MSDA_PADDING_BORDER) return MSDA_ERR_BAD_ENUM;
    if (d->align_corners != 0 && d->align_corners != 1) return MSDA_ERR_BAD_ENUM;
    if (d->value_dtype != MSDA_DTYPE_F32 && d->value_dtype != MSDA_DTYPE_BF16 && d->value_dtype != MSDA_DTYPE_F16)
        return MSDA_ERR_BAD_ENUM;
    if (d->loc_dtype != MSDA_DTYPE_F32 && d->loc_dtype != MSDA_DTYPE_BF16 && d->loc_dtype != MSDA_DTYPE_F16)
        return MSDA_ERR_BAD_ENUM;
    if (d->B < 0 || d->N_q < 0 || d->N_h < 0 || d->C_h < 0 || d->N_l < 0 || d->N_p < 0 || d->L < 0)
        return MSDA_ERR_BAD_DIM;
    if (d->N_l > MSDA_MAX_LEVELS) return MSDA_ERR_BAD_DIM;
    if (d->N_l > 0 && (!d->spatial_shapes || !d->level_start_index)) return MSDA_ERR_NULL_POINTER;
    int64_t s = 0;
    for (int64_t l = 0; l < d->N_l; ++l) {
        const int64_t H = d->spatial_shapes[2 * l], W = d->spatial_shapes[2 * l + 1];
        if (H < 1 || W < 1 || H > kIndexLimit || W > kIndexLimit) return MSDA_ERR_LEVELS;
        if (d->level_start_index[l] != s) return MSDA_ERR_LEVELS;
        s += H * W;
        if (s > kIndexLimit) return MSDA_ERR_TOO_LARGE;
    }
    if (s != d->L) return MSDA_ERR_LEVELS;
    // 32-bit index limits (stated in msda.h)
    if (d->N_h > 0 && d->C_h > 0 && d->L > kIndexLimit / d->N_h / d->C_h) return MSDA_ERR_TOO_LARGE;
    const int64_t nlp = d->N_l * d->N_p;
    // Corner offsets of cells up to two pixels outside a level are formed in
    // 32-bit arithmetic: (L + 2*max(W) + 4) * N_h * C_h must stay below 2^31.
    int64_t wmax = 0;
    for (int64_t l = 0; l < d->N_l; ++l) wmax = d->spatial_shapes[2 * l + 1] > wmax ? d->spatial_shapes[2 * l + 1] : wmax;
    if (d->N_h > 0 && d->C_h > 0 && d->L + 2 * wmax + 4 > kIndexLimit / d->N_h / d->C_h) return MSDA_ERR_TOO_LARGE;
    if (d->N_q > 0 && d->N_h > 0 && nlp > 0 && d->N_q > kIndexLimit / 2 / d->N_h / nlp) return MSDA_ERR_TOO_LARGE;
    if (d->B > 0 && d->N_q > 0 && d->N_h > 0 && d->B > kIndexLimit / d->N_q / d->N_h) return MSDA_ERR_TOO_LARGE;
    if (d->value_dtype == MSDA_DTYPE_F16) return MSDA_ERR_UNSUPPORTED;  // value: binary32 or bfloat16 only
    return MSDA_OK;
}

// Kernel configuration chosen from C_h, pointer alignment and direction.
struct Config {
    bool vec;
    int G, NCH;
};

// V: elements per vector access; aligned: every value-typed pointer is
// aligned to V elements (and the binary32 accumulator to 16 bytes).
int choose_config(const msda_desc *d, int V, bool aligned_ok, int preferred_lanes, Config *cfg) {
    cfg->vec = aligned_ok && (d->C_h % V == 0);
    const int64_t chunks = cfg->vec ? d->C_h / V : d->C_h;
    if (chunks > 256) return MSDA_ERR_UNSUPPORTED;
    const msda::Shape s = msda::select_shape((int)chunks, preferred_lanes);
    cfg->G = s.G;
    cfg->NCH = s.NCH;
    return MSDA_OK;
}

// n / d in the kernels' FastDiv form (d >= 1).
msda::FastDiv make_fastdiv(uint32_t d) {
    msda::FastDiv f;
    f.d = d < 1 ? 1 : d;
    uint32_t s = 0;
    while (((uint64_t)1 << s) < f.d) ++s;
    f.shift = s;
    f.mul = (uint32_t)((((uint64_t)1 << 32) * (((uint64_t)1 << s) - f.d)) / f.d + 1);
    return f;
}

// Tile partition of the tile-sorted grad_value (see msda_kernels.cuh): per
// level, ceil((H+1)/T) x ceil((W+1)/T) tiles of T x T cells; partition blocks
// of part_rows (about 512) rows each, at most 1024 of them; `usable` when the
// sizes fit the kernels' 32-bit indices and shared-memory tables.
struct TileGeom {
    int64_t NB, bst[msda::kMaxLevels], BX[msda::kMaxLevels];
    int64_t nbins, parts, part_rows, span;
    bool usable;
};

TileGeom tile_geom(const msda_desc *d) {
    TileGeom g;
    memset(&g, 0, sizeof(g));
    const int64_t T = msda::kTileCells;
    for (int64_t l = 0; l < d->N_l; ++l) {
        const int64_t H = d->spatial_shapes[2 * l], W = d->spatial_shapes[2 * l + 1];
        g.bst[l] = g.NB;
        g.BX[l] = (W + 1 + T - 1) / T;
        g.NB += ((H + 1 + T - 1) / T) * g.BX[l];
    }
    const int64_t rows = d->B * d->N_h * d->N_q;
    const int64_t samples = rows * d->N_l * d->N_p;
    g.nbins = d->B * d->N_h * g.NB;
    g.parts = rows > 0 ? (rows + 511) / 512 : 1;
    if (g.parts > 1024) g.parts = 1024;
    g.part_rows = rows > 0 ? (rows + g.parts - 1) / g.parts : 1;
    g.span = d->N_q > 0 ? (g.part_rows + d->N_q - 1) / d->N_q + 1 : 1;
    g.usable = rows > 0 && samples < (int64_t)INT32_MAX && rows < ((int64_t)1 << msda::kEntryCellShift) &&
               g.nbins * g.parts + 1 < (int64_t)INT32_MAX && g.span * g.NB * 4 <= 48 * 1024;
    return g;
}

Params make_params(const msda_desc *d, const Config &cfg, int V_vec) {
    Params p;
    memset(&p, 0, sizeof(p));
    p.rows = (uint32_t)(d->B * d->N_q * d->N_h);
    p.N_q = (int)d->N_q;
    p.N_h = (int)d->N_h;
    p.C_h = (int)d->C_h;
    p.N_l = (int)d->N_l;
    p.N_p = (int)d->N_p;
    p.NLP = (int)(d->N_l * d->N_p);
    const int V = cfg.vec ? V_vec : 1;
    p.chunks = (int)(d->C_h / V);
    p.div_q = make_fastdiv((uint32_t)d->N_q);
    p.div_h = make_fastdiv((uint32_t)d->N_h);
    p.div_p = make_fastdiv((uint32_t)d->N_p);
    p.div_nlp = make_fastdiv((uint32_t)(d->N_l * d->N_p));
    p.padding = d->padding_mode;
    p.loc_dt = d->loc_dtype == MSDA_DTYPE_F32 ? 0 : d->loc_dtype == MSDA_DTYPE_BF16 ? 1 : 2;
    p.flags = 0;
    if (d->value_layout == MSDA_LAYOUT_BLNC) {
        p.v_sB = d->L * d->N_h * d->C_h;
        p.v_sP = (int)(d->N_h * d->C_h);
        p.v_sH = (int)d->C_h;
    } else {
        p.v_sB = d->N_h * d->L * d->C_h;
        p.v_sH = (int)(d->L * d->C_h);
        p.v_sP = (int)d->C_h;
    }
    const int64_t per_batch = d->N_q * d->N_h * d->N_l * d->N_p;  // samples in one batch item
    if (d->loc_layout == MSDA_LAYOUT_BQHLP2) {
        p.l_sB = 2 * per_batch;
        p.l_sJ = 2;
        p.l_sXY = 1;
    } else {
        p.l_sB = 2 * per_batch;
        p.l_sJ = 1;
        p.l_sXY = (int)per_batch;
    }
    for (int64_t l = 0; l < d->N_l; ++l) {
        const int64_t H = d->spatial_shapes[2 * l], W = d->spatial_shapes[2 * l + 1];
        p.H[l] = (int)H;
        p.W[l] = (int)W;
        p.start[l] = (int)d->level_start_index[l];
        // align_corners: [0,1] -> [0, size-1] (True) or [-0.5, size-0.5] (False)
        p.sx[l] = (float)(d->align_corners ? W - 1 : W);
        p.sy[l] = (float)(d->align_corners ? H - 1 : H);
    }
    p.off = d->align_corners ? 0.0f : -0.5f;
    const TileGeom tg = tile_geom(d);
    p.NB = (int)tg.NB;
    for (int l = 0; l < (int)d->N_l; ++l) {
        p.bst[l] = (int)tg.bst[l];
        p.BX[l] = (int)tg.BX[l];
    }
    p.nbins = tg.usable ? (uint32_t)tg.nbins : 0u;
    p.parts = (uint32_t)tg.parts;
    p.part_rows = (uint32_t)tg.part_rows;
    p.span = (int)tg.span;
    p.capacity = (uint32_t)(d->B * d->N_q * d->N_h * d->N_l * d->N_p);
    return p;
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cached[dev] = n;
    return n;
}

// Workspace of the backward, in 256-byte aligned regions:
//   acc      binary32 grad_value accumulator (bfloat16 value with grad_value)
//   offsets  (tile, part) counts, then offsets (nbins * parts + 1 int32)  \
//   chunks   per-tile chunk counts, then chunk offsets (nbins + 1)        |  tile-sorted
//   tiles    tile sums of the scans                                      |  grad_value
//   entries  the samples grouped by tile (samples x 16 bytes)            /
// The tile-sorted grad_value is used when grad_value is the only output, there
// are at least MSDA_SORT_MIN_DENSITY samples per bilinear cell on average
// (below that its partition passes cost more than the atomics they save), the
// vector path applies (C_h a multiple of 4) and the tile geometry is usable;
// its regions are planned whenever grad_value is requested (the workspace size
// depends on the descriptor only).
#ifndef MSDA_SORT_MIN_DENSITY
#define MSDA_SORT_MIN_DENSITY 2
#endif
struct BwdPlan {
    bool sort;
    size_t acc_off, offsets_off, chunks_off, tiles_off, entries_off, total;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

BwdPlan plan_backward(const msda_desc *d, int compute_grad_value, bool allow_sort) {
    BwdPlan w;
    memset(&w, 0, sizeof(w));
    if (!compute_grad_value) return w;
    const int64_t samples = d->B * d->N_q * d->N_h * d->N_l * d->N_p;
    int64_t cells = 0;
    for (int64_t l = 0; l < d->N_l; ++l) cells += (d->spatial_shapes[2 * l] + 1) * (d->spatial_shapes[2 * l + 1] + 1);
    cells *= d->B * d->N_h;
    const TileGeom tg = tile_geom(d);
    w.sort = allow_sort && samples > 0 && samples >= (int64_t)MSDA_SORT_MIN_DENSITY * cells && tg.usable &&
             d->C_h % 4 == 0;
    size_t end = 0;  // end of the regions so far (each region starts 256-byte aligned)
    if (d->value_dtype == MSDA_DTYPE_BF16) {
        w.acc_off = 0;
        end = (size_t)(d->B * d->L * d->N_h * d->C_h) * sizeof(float);
    }
    if (w.sort) {
        const int64_t n = tg.nbins * tg.parts;
        const int64_t tiles = (n + 1 + msda::kScanTile - 1) / msda::kScanTile;
        w.offsets_off = align256(end);
        w.chunks_off = align256(w.offsets_off + (size_t)(n + 1) * sizeof(int));
        w.tiles_off = align256(w.chunks_off + (size_t)(tg.nbins + 1) * sizeof(int));
        w.entries_off = align256(w.tiles_off + (size_t)tiles * sizeof(int));
        end = w.entries_off + (size_t)samples * 16;
    }
    w.total = end;
    return w;
}

// Parts a row's samples are split into (log2; see block_rows): more than one
// only while rows x lanes fill at most half of the GPU's resident threads
// (2048 a multiprocessor), every part keeps at least one batch of G samples
// and a row's parts stay within one warp.
// The warp-aggregated grad_value scatter is on unless the environment
// variable MSDA_BWD_AGGREGATE is "0" (read at every backward call).
int aggregate_enabled() {
    const char *v = getenv("MSDA_BWD_AGGREGATE");
    return (v && v[0] == '0' && v[1] == '\0') ? 0 : 1;
}

int choose_split(const Params &p, int G, bool allowed) {
    if (!allowed || p.rows == 0) return 0;
    const uint64_t capacity = (uint64_t)(p.n_sm > 0 ? p.n_sm : 1) * 2048;
    const uint64_t lanes = (uint64_t)p.rows * (uint64_t)G;
    int s = 0;
    while ((G << (s + 1)) <= 32 && (int64_t)((2 << s) - 1) * G < p.NLP && (lanes << (s + 1)) * 2 <= capacity) ++s;
    return s;
}

// Staged-level forward (msda_forward_staged): the coarsest levels, from the
// last one down, whose pixels of one head fit MSDA_STAGE_BYTES of shared
// memory, each level's region rounded up to whole TMA boxes.  40 KB keeps
// three blocks per SM; a 96 KB budget (two levels of the bfloat16 workloads,
// two blocks per SM) measured slower.
#ifndef MSDA_STAGE_BYTES
#define MSDA_STAGE_BYTES (40 * 1024)
#endif

// false when the staged kernel does not apply (the direct forward runs):
// 16-bit locations, scalar path or wide rows, a pixel row that is not a
// multiple of 16 bytes, value not 16-byte aligned, or no level that fits.
// The levels themselves: from the last one down while their pixels of one
// head (pxb bytes each) fit the budget.
bool plan_levels(const msda_desc *d, int64_t pxb, msda::StagePlan *sp, size_t *smem) {
    memset(sp, 0, sizeof(*sp));
    sp->ls = (int)d->N_l;
    int64_t pix = 0;
    for (int64_t l = d->N_l - 1; l >= 0; --l) {
        const int64_t n = d->spatial_shapes[2 * l] * d->spatial_shapes[2 * l + 1];
        const int64_t region = (n + msda::kStageBox - 1) / msda::kStageBox * msda::kStageBox;
        if ((pix + region) * pxb > MSDA_STAGE_BYTES) break;
        pix += region;
        sp->ls = (int)l;
    }
    if (sp->ls == (int)d->N_l) return false;
    int64_t off = 0;
    for (int64_t l = sp->ls; l < d->N_l; ++l) {
        const int64_t n = d->spatial_shapes[2 * l] * d->spatial_shapes[2 * l + 1];
        const int64_t region = (n + msda::kStageBox - 1) / msda::kStageBox * msda::kStageBox;
        sp->sp[l] = (int)off;
        off += region;
        sp->boxes += (int)(region / msda::kStageBox);
    }
    sp->bytes = (uint32_t)(pix * pxb);
    sp->layout = d->value_layout == MSDA_LAYOUT_BLNC ? 0 : 1;
    *smem = (size_t)(pix * pxb);
    return true;
}

bool plan_stage(const msda_desc *d, const Config &cfg, const void *value, msda::StagePlan *sp, size_t *smem) {
    const int64_t pxb = d->C_h * (int64_t)value_elem_size(d);  // bytes of one pixel of one head
    if (d->loc_dtype != MSDA_DTYPE_F32 || !cfg.vec || !msda::specialised_shape(cfg.G, cfg.NCH) || pxb % 16 != 0 ||
        d->C_h < 4 || d->C_h > 256 || !aligned(value, 16) || d->N_l < 1 || d->L < msda::kStageBox)
        return false;
    if (!plan_levels(d, pxb, sp, smem)) return false;
    *smem += 128;  // slack for the kernel's 128-byte alignment of the TMA destinations
    return true;
}

// msda_backward_staged: the binary32 grad_value accumulator of the staged
// levels (C_h * 4 bytes a pixel), the vector path's specialised shapes.
bool plan_stage_backward(const msda_desc *d, const Config &cfg, msda::StagePlan *sp, size_t *smem) {
    if (!cfg.vec || !msda::specialised_shape(cfg.G, cfg.NCH) || d->C_h < 4 || d->N_l < 1) return false;
    if (!plan_levels(d, d->C_h * 4, sp, smem)) return false;
    const int chunks = (int)(d->C_h / 4);
    sp->rot = (chunks & (chunks - 1)) == 0 ? (chunks < 8 ? chunks : 8) - 1 : 0;
    return true;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); null when the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// value as a 4-D tensor, innermost first: (C_h, N_h, L, B) for (B, L, N_h, C_h)
// or (C_h, L, N_h, B) for (B, N_h, L, C_h); a box is one head's channel rows of
// kStageBox consecutive pixels.
bool encode_value_map(const msda_desc *d, const void *value, CUtensorMap *tm) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t e = value_elem_size(d), C = (cuuint64_t)d->C_h, H = (cuuint64_t)d->N_h,
                     L = (cuuint64_t)d->L, B = (cuuint64_t)d->B;
    const bool blnc = d->value_layout == MSDA_LAYOUT_BLNC;
    const cuuint64_t dims[4] = {C, blnc ? H : L, blnc ? L : H, B};
    const cuuint64_t strides[3] = {C * e, (blnc ? H : L) * C * e, L * H * C * e};
    const cuuint32_t box[4] = {(cuuint32_t)C, blnc ? 1u : (cuuint32_t)msda::kStageBox,
                               blnc ? (cuuint32_t)msda::kStageBox : 1u, 1u};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = enc(tm, d->value_dtype == MSDA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                           4, const_cast<void *>(value), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

namespace msda {

__global__ void msda_zero_f32_kernel(float *__restrict__ p, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (((uintptr_t)p & 15) == 0) {
        const int64_t n4 = n / 4;
        float4 *p4 = reinterpret_cast<float4 *>(p);
        for (int64_t k = i; k < n4; k += stride) p4[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int64_t k = n4 * 4 + i; k < n; k += stride) p[k] = 0.0f;
    } else {
        for (int64_t k = i; k < n; k += stride) p[k] = 0.0f;
    }
}

__global__ void msda_f32_to_bf16_kernel(const float *__restrict__ acc, __nv_bfloat16 *__restrict__ out,
                                        int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if ((((uintptr_t)acc | (uintptr_t)out) & 15) == 0) {
        const int64_t n8 = n / 8;
        for (int64_t k = i; k < n8; k += stride) {
            float x[8];
            const float4 a = reinterpret_cast<const float4 *>(acc)[2 * k];
            const float4 b = reinterpret_cast<const float4 *>(acc)[2 * k + 1];
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
            x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
            VecIO<__nv_bfloat16, 8>::store(out + 8 * k, x);
        }
        for (int64_t k = n8 * 8 + i; k < n; k += stride) out[k] = __float2bfloat16_rn(acc[k]);
    } else {
        for (int64_t k = i; k < n; k += stride) out[k] = __float2bfloat16_rn(acc[k]);
    }
}

__device__ __forceinline__ int block_exclusive_scan(int x, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        warp_sums[lane] = wi - w;  // exclusive
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    return warp_sums[warp] + incl - x;
}

__global__ void __launch_bounds__(kScanThreads)
msda_scan_tiles_kernel(const int *__restrict__ counts, uint32_t n, int *__restrict__ tile_sums) {
    __shared__ int red[kScanThreads / 32];
    const uint64_t base = (uint64_t)blockIdx.x * kScanTile + (uint64_t)threadIdx.x * kScanPer;
    int s = 0;
#pragma unroll
    for (int i = 0; i < kScanPer; ++i)
        if (base + i < n) s += counts[base + i];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x < 32) {
        int t = red[threadIdx.x];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (threadIdx.x == 0) tile_sums[blockIdx.x] = t;
    }
}

__global__ void __launch_bounds__(kScanThreads)
msda_scan_apply_kernel(int *__restrict__ offsets, uint32_t n, const int *__restrict__ tile_sums) {
    __shared__ int warp_sums[32];
    __shared__ int total;
    __shared__ int prefix;
    // sum of the tiles before this one
    int pre = 0;
    for (uint32_t t = threadIdx.x; t < blockIdx.x; t += kScanThreads) pre += tile_sums[t];
    {
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) pre += __shfl_xor_sync(0xffffffffu, pre, o);
        if (lane == 0) warp_sums[threadIdx.x >> 5] = pre;
        __syncthreads();
        if (threadIdx.x < 32) {
            int t = warp_sums[threadIdx.x];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
            if (threadIdx.x == 0) prefix = t;
        }
        __syncthreads();
    }
    const uint64_t base = (uint64_t)blockIdx.x * kScanTile + (uint64_t)threadIdx.x * kScanPer;
    int v[kScanPer];
    int s = 0;
#pragma unroll
    for (int i = 0; i < kScanPer; ++i) {
        v[i] = base + i < n ? offsets[base + i] : 0;
        s += v[i];
    }
    const int ex = block_exclusive_scan(s, warp_sums, &total) + prefix;
    int run = ex;
#pragma unroll
    for (int i = 0; i < kScanPer; ++i) {
        if (base + i < n) offsets[base + i] = run;
        run += v[i];
    }
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) offsets[n] = prefix + total;
}

static unsigned helper_grid(int64_t n, int per_thread) {
    const int64_t threads = (n + per_thread - 1) / per_thread;
    int64_t blocks = (threads + 255) / 256;
    const int64_t cap = 152 * 16;  // a few waves over the SMs; the loops are grid-stride
    if (blocks > cap) blocks = cap;
    return (unsigned)(blocks < 1 ? 1 : blocks);
}

cudaError_t launch_zero_f32(float *p, int64_t n, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    msda_zero_f32_kernel<<<helper_grid(n, 4), 256, 0, stream>>>(p, n);
    return cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float *acc, __nv_bfloat16 *out, int64_t n, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    msda_f32_to_bf16_kernel<<<helper_grid(n, 8), 256, 0, stream>>>(acc, out, n);
    return cudaGetLastError();
}

__global__ void msda_tile_items_kernel(const __grid_constant__ Params p, const int *__restrict__ offsets,
                                       int *__restrict__ chunks) {
    const uint32_t tile = blockIdx.x * blockDim.x + threadIdx.x;
    if (tile >= p.nbins) return;
    const int beg = offsets[(size_t)tile * p.parts], end = offsets[(size_t)(tile + 1) * p.parts];
    chunks[tile] = (end - beg + kChunk - 1) / kChunk;
}

// Exclusive scan of n int32 in place; data[n] = total.
static cudaError_t launch_scan(int *data, uint32_t n, int *tile_sums, cudaStream_t stream) {
    const unsigned tiles = (unsigned)(((uint64_t)n + kScanTile - 1) / kScanTile);
    if (tiles == 0) return cudaSuccess;
    msda_scan_tiles_kernel<<<tiles, kScanThreads, 0, stream>>>(data, n, tile_sums);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    msda_scan_apply_kernel<<<tiles, kScanThreads, 0, stream>>>(data, n, tile_sums);
    return cudaGetLastError();
}

cudaError_t launch_tile_partition(const Params &p, const float *loc, const float *attn, const BwdBuffers &bb,
                                  cudaStream_t stream) {
    if (p.nbins == 0 || p.rows == 0) return cudaSuccess;
    const uint32_t n = p.nbins * p.parts;
    cudaError_t e = launch_zero_f32(reinterpret_cast<float *>(bb.offsets), (int64_t)n + 1, stream);
    if (e != cudaSuccess) return e;
    const size_t hist = (size_t)p.span * p.NB * sizeof(int);
    const unsigned parts = (unsigned)((p.rows + p.part_rows - 1) / p.part_rows);
    if (p.padding == 0)
        msda_tile_count_kernel<0><<<parts, 256, hist, stream>>>(p, loc, bb.offsets);
    else
        msda_tile_count_kernel<1><<<parts, 256, hist, stream>>>(p, loc, bb.offsets);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_scan(bb.offsets, n, bb.tile_sums, stream);
    if (e != cudaSuccess) return e;
    msda_tile_items_kernel<<<(p.nbins + 255) / 256, 256, 0, stream>>>(p, bb.offsets, bb.chunks);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_scan(bb.chunks, p.nbins, bb.tile_sums, stream);
    if (e != cudaSuccess) return e;
    if (p.padding == 0)
        msda_tile_append_kernel<0><<<parts, 256, hist, stream>>>(p, loc, attn, bb.offsets, bb.entries);
    else
        msda_tile_append_kernel<1><<<parts, 256, hist, stream>>>(p, loc, attn, bb.offsets, bb.entries);
    return cudaGetLastError();
}

size_t backward_workspace_bytes(const msda_desc *desc, int compute_grad_value, bool allow_sort) {
    if (validate_desc(desc) != MSDA_OK) return 0;
    return plan_backward(desc, compute_grad_value, allow_sort).total;
}

int backward_entry(const msda_desc *desc, const void *grad_output, const void *value,
                   const void *sampling_locations, const void *attention_weights, int compute_grad_value,
                   int compute_grad_sampling_locations, int compute_grad_attention_weights, void *grad_value,
                   void *grad_sampling_locations, void *grad_attention_weights, void *workspace,
                   size_t workspace_bytes, BwdMode mode, cudaStream_t stream) {
    const bool allow_sort = mode.allow_sort, accumulate = mode.accumulate;
    int rc = validate_desc(desc);
    if (rc) return rc;
    const msda_desc *d = desc;
    const int fv = compute_grad_value, fl = compute_grad_sampling_locations, fa = compute_grad_attention_weights;
    if ((fv != 0 && fv != 1) || (fl != 0 && fl != 1) || (fa != 0 && fa != 1)) return MSDA_ERR_BAD_ENUM;
    if (!fv && !fl && !fa) return MSDA_ERR_NO_OUTPUT;  // backward page: at least one flag must be True
    const int64_t samples = d->B * d->N_q * d->N_h * d->N_l * d->N_p;
    const int64_t value_elems = d->B * d->L * d->N_h * d->C_h;
    const int64_t go_elems = d->B * d->N_q * d->N_h * d->C_h;
    const bool need_v = (fl || fa) && samples > 0 && d->C_h > 0;
    const bool need_a = (fv || fl || (mode.logits && fa)) && samples > 0;
    if (samples > 0 && !sampling_locations) return MSDA_ERR_NULL_POINTER;
    if (samples > 0 && go_elems > 0 && !grad_output) return MSDA_ERR_NULL_POINTER;
    if (need_v && !value) return MSDA_ERR_NULL_POINTER;
    if (need_a && !attention_weights) return MSDA_ERR_NULL_POINTER;
    if (fv && value_elems > 0 && !grad_value) return MSDA_ERR_NULL_POINTER;
    if (fl && samples > 0 && !grad_sampling_locations) return MSDA_ERR_NULL_POINTER;
    if (fa && samples > 0 && !grad_attention_weights) return MSDA_ERR_NULL_POINTER;
    const size_t es = value_elem_size(d);
    if (!aligned(grad_output, es) || !aligned(value, es) || !aligned(grad_value, accumulate ? 4 : es) ||
        !aligned(sampling_locations, loc_elem_size(d)) || !aligned(attention_weights, loc_elem_size(d)) ||
        !aligned(grad_sampling_locations, loc_elem_size(d)) || !aligned(grad_attention_weights, loc_elem_size(d)))
        return MSDA_ERR_MISALIGNED;
    const bool bf16 = d->value_dtype == MSDA_DTYPE_BF16;
    const BwdPlan plan = plan_backward(d, fv, allow_sort);
    if (plan.total > 0) {
        if (workspace_bytes < plan.total) return MSDA_ERR_WORKSPACE;
        if (!workspace) return MSDA_ERR_NULL_POINTER;
        if (!aligned(workspace, 16)) return MSDA_ERR_MISALIGNED;
    }
    unsigned char *ws = (unsigned char *)workspace;
    BwdBuffers bb;
    memset(&bb, 0, sizeof(bb));
    // the binary32 accumulator: the caller's (accumulate), grad_value itself
    // (binary32 value) or the workspace (bfloat16 value)
    bb.gv_acc = fv ? ((bf16 && !accumulate) ? (float *)(ws + plan.acc_off) : (float *)grad_value) : nullptr;
    bb.grad_loc = (float *)grad_sampling_locations;
    bb.grad_attn = (float *)grad_attention_weights;
    if (plan.sort) {
        bb.offsets = (int *)(ws + plan.offsets_off);
        bb.chunks = (int *)(ws + plan.chunks_off);
        bb.tile_sums = (int *)(ws + plan.tiles_off);
        bb.entries = (uint4 *)(ws + plan.entries_off);
    }
    Config cfg;
    const int V = BwdVecWidth<float>::value;
    rc = choose_config(d, V,
                       aligned(grad_output, V * es) && aligned(value, V * es) && (!fv || aligned(bb.gv_acc, 16)),
                       MSDA_BWD_LANES, &cfg);
    if (rc) return rc;
    Params p = make_params(d, cfg, V);
    p.flags = (fv ? kGradValue : 0) | (fl ? kGradLoc : 0) | (fa ? kGradAttn : 0);
    p.logits = mode.logits ? 1 : 0;
    p.n_sm = samples > 0 ? sm_count() : 0;
    p.split_log2 = choose_split(p, cfg.G, !mode.logits);  // the logits' gradient needs whole rows
    p.aggregate = aggregate_enabled();

    cudaError_t e = cudaSuccess;
    if (fv && !accumulate) e = launch_zero_f32(bb.gv_acc, value_elems, stream);
    // staged variant (msda_backward_staged): the per-level shared-memory
    // accumulator kernel in place of the row kernel, where it applies
    StagePlan sp;
    size_t smem = 0;
    const bool staged = mode.staged && fv && !mode.logits && samples > 0 && plan_stage_backward(d, cfg, &sp, &smem);
    if (staged) {
        if (e == cudaSuccess) {
            if (bf16)
                e = launch_backward_staged<__nv_bfloat16>(p, sp, smem, cfg.G, cfg.NCH,
                                                          (const __nv_bfloat16 *)grad_output,
                                                          (const __nv_bfloat16 *)value, (const float *)sampling_locations,
                                                          (const float *)attention_weights, bb.gv_acc, bb.grad_loc,
                                                          bb.grad_attn, stream);
            else
                e = launch_backward_staged<float>(p, sp, smem, cfg.G, cfg.NCH, (const float *)grad_output,
                                                  (const float *)value, (const float *)sampling_locations,
                                                  (const float *)attention_weights, bb.gv_acc, bb.grad_loc,
                                                  bb.grad_attn, stream);
        }
        if (e == cudaSuccess && bf16 && !accumulate)
            e = launch_f32_to_bf16(bb.gv_acc, (__nv_bfloat16 *)grad_value, value_elems, stream);
        return record_cuda(e);
    }
    // tile-sorted grad_value (vector path): partition, the row kernel for the
    // other two gradients only, then the per-tile reduction
    const bool sort = plan.sort && cfg.vec && !fl && !fa;
    if (e == cudaSuccess && samples > 0 && sort)
        e = launch_tile_partition(p, (const float *)sampling_locations, (const float *)attention_weights, bb, stream);
    Params prow = p;
    if (sort) prow.flags &= ~kGradValue;
    if (e == cudaSuccess && samples > 0 && prow.flags) {
        if (bf16)
            e = launch_backward<__nv_bfloat16>(prow, cfg.vec, cfg.G, cfg.NCH, (const __nv_bfloat16 *)grad_output,
                                               (const __nv_bfloat16 *)value, (const float *)sampling_locations,
                                               (const float *)attention_weights, bb, stream);
        else
            e = launch_backward<float>(prow, cfg.vec, cfg.G, cfg.NCH, (const float *)grad_output,
                                       (const float *)value, (const float *)sampling_locations,
                                       (const float *)attention_weights, bb, stream);
    }
    if (e == cudaSuccess && samples > 0 && sort) {
        if (bf16)
            e = launch_tile_reduce<__nv_bfloat16, true>(p, cfg.G, cfg.NCH, (const __nv_bfloat16 *)grad_output, bb,
                                                        stream);
        else
            e = launch_tile_reduce<float, true>(p, cfg.G, cfg.NCH, (const float *)grad_output, bb, stream);
    }
    if (e == cudaSuccess && fv && bf16 && !accumulate) e = launch_f32_to_bf16(bb.gv_acc, (__nv_bfloat16 *)grad_value, value_elems, stream);
    return record_cuda(e);
}

// Blocks of the staged forward that gave up waiting for their copy [0], and
// of those, blocks that exited while the copy was still unfinished [1].
__device__ unsigned int g_stage_timeouts[2] = {0u, 0u};

// The counter's device address on the current device, looked up once per
// device (null when the lookup fails).
unsigned int *stage_timeout_counter() {
    constexpr int kMaxDevices = 64;
    static std::atomic<unsigned int *> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    unsigned int *c = cache[dev].load(std::memory_order_acquire);
    if (!c) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, g_stage_timeouts) != cudaSuccess) return nullptr;
        c = static_cast<unsigned int *>(a);
        cache[dev].store(c, std::memory_order_release);
    }
    return c;
}

int staged_timeouts(unsigned int *count) {
    if (!count) return MSDA_ERR_NULL_POINTER;
    unsigned int c[2] = {0u, 0u};
    const int rc = record_cuda(cudaMemcpyFromSymbol(c, g_stage_timeouts, sizeof(c)));
    if (rc != MSDA_OK) return rc;
    *count = c[0];
    return c[1] ? MSDA_ERR_STAGE_COPY : MSDA_OK;
}

int forward_entry(const msda_desc *desc, const void *value, const void *sampling_locations,
                  const void *attention_weights, void *out, bool logits, bool staged, cudaStream_t stream) {
    int rc = validate_desc(desc);
    if (rc) return rc;
    const msda_desc *d = desc;
    const int64_t samples = d->B * d->N_q * d->N_h * d->N_l * d->N_p;
    const int64_t out_elems = d->B * d->N_q * d->N_h * d->C_h;
    const int64_t value_elems = d->B * d->L * d->N_h * d->C_h;
    const bool reads = out_elems > 0 && samples > 0;
    if ((out_elems > 0 && !out) || (reads && (!sampling_locations || !attention_weights)) ||
        (reads && value_elems > 0 && !value))
        return MSDA_ERR_NULL_POINTER;
    const size_t es = value_elem_size(d);
    if (!aligned(value, es) || !aligned(out, es) || !aligned(sampling_locations, loc_elem_size(d)) ||
        !aligned(attention_weights, loc_elem_size(d)))
        return MSDA_ERR_MISALIGNED;
    Config cfg;
    const int V = d->value_dtype == MSDA_DTYPE_BF16 ? msda::VecWidth<__nv_bfloat16>::value
                                                     : msda::VecWidth<float>::value;
    rc = choose_config(d, V, aligned(value, V * es) && aligned(out, V * es), MSDA_FWD_LANES, &cfg);
    if (rc) return rc;
    if (out_elems == 0) return MSDA_OK;
    Params p = make_params(d, cfg, V);
    p.n_sm = sm_count();
    p.logits = logits ? 1 : 0;
    p.split_log2 = choose_split(p, cfg.G, true);
    cudaError_t e;
    StagePlan sp;
    size_t smem = 0;
    CUtensorMap tm;
    if (staged && !logits && samples > 0 && plan_stage(d, cfg, value, &sp, &smem) &&
        encode_value_map(d, value, &tm)) {
        unsigned int *timeouts = stage_timeout_counter();
        e = timeouts ? cudaSuccess : cudaErrorInvalidSymbol;
        if (e == cudaSuccess) {
            if (d->value_dtype == MSDA_DTYPE_F32)
                e = launch_forward_staged<float>(p, sp, tm, smem, cfg.G, cfg.NCH, (const float *)value,
                                                 (const float *)sampling_locations,
                                                 (const float *)attention_weights, (float *)out, timeouts, stream);
            else
                e = launch_forward_staged<__nv_bfloat16>(p, sp, tm, smem, cfg.G, cfg.NCH,
                                                         (const __nv_bfloat16 *)value,
                                                         (const float *)sampling_locations,
                                                         (const float *)attention_weights, (__nv_bfloat16 *)out,
                                                         timeouts, stream);
        }
        return record_cuda(e);
    }
    if (d->value_dtype == MSDA_DTYPE_F32)
        e = msda::launch_forward<float>(p, cfg.vec, cfg.G, cfg.NCH, (const float *)value,
                                        (const float *)sampling_locations, (const float *)attention_weights,
                                        (float *)out, stream);
    else
        e = msda::launch_forward<__nv_bfloat16>(p, cfg.vec, cfg.G, cfg.NCH, (const __nv_bfloat16 *)value,
                                                (const float *)sampling_locations,
                                                (const float *)attention_weights, (__nv_bfloat16 *)out, stream);
    return record_cuda(e);
}

}  // namespace msda

extern "C" {

int msda_forward(const msda_desc *desc, const void *value, const void *sampling_locations,
                 const void *attention_weights, void *out, cudaStream_t stream) {
    return msda::forward_entry(desc, value, sampling_locations, attention_weights, out, false, false, stream);
}

int msda_forward_staged(const msda_desc *desc, const void *value, const void *sampling_locations,
                        const void *attention_weights, void *out, cudaStream_t stream) {
    return msda::forward_entry(desc, value, sampling_locations, attention_weights, out, false, true, stream);
}

int msda_staged_timeouts(unsigned int *count) { return msda::staged_timeouts(count); }

int msda_backward_staged(const msda_desc *desc, const void *grad_output, const void *value,
                         const void *sampling_locations, const void *attention_weights, int compute_grad_value,
                         int compute_grad_sampling_locations, int compute_grad_attention_weights, void *grad_value,
                         void *grad_sampling_locations, void *grad_attention_weights, void *workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
    msda::BwdMode mode{true, false, false};
    mode.staged = true;
    return msda::backward_entry(desc, grad_output, value, sampling_locations, attention_weights, compute_grad_value,
                                compute_grad_sampling_locations, compute_grad_attention_weights, grad_value,
                                grad_sampling_locations, grad_attention_weights, workspace, workspace_bytes, mode,
                                stream);
}

int msda_backward_staged_levels(const msda_desc *desc, int *first_level) {
    if (!first_level) return MSDA_ERR_NULL_POINTER;
    const int rc = validate_desc(desc);
    if (rc) return rc;
    Config cfg;
    const int rc2 = choose_config(desc, msda::BwdVecWidth<float>::value, true, MSDA_BWD_LANES, &cfg);
    if (rc2) return rc2;
    msda::StagePlan sp;
    size_t smem;
    *first_level = plan_stage_backward(desc, cfg, &sp, &smem) ? sp.ls : (int)desc->N_l;
    return MSDA_OK;
}

int msda_forward_staged_levels(const msda_desc *desc, int *first_level) {
    if (!first_level) return MSDA_ERR_NULL_POINTER;
    const int rc = validate_desc(desc);
    if (rc) return rc;
    Config cfg;
    const int V = msda::VecWidth<float>::value;  // the same for both value dtypes
    const int rc2 = choose_config(desc, V, true, MSDA_FWD_LANES, &cfg);
    if (rc2) return rc2;
    msda::StagePlan sp;
    size_t smem;
    *first_level = plan_stage(desc, cfg, (const void *)16, &sp, &smem) ? sp.ls : (int)desc->N_l;
    return MSDA_OK;
}

size_t msda_backward_workspace_size(const msda_desc *desc, int compute_grad_value) {
    return msda::backward_workspace_bytes(desc, compute_grad_value, true);
}

int msda_backward(const msda_desc *desc, const void *grad_output, const void *value,
                  const void *sampling_locations, const void *attention_weights, int compute_grad_value,
                  int compute_grad_sampling_locations, int compute_grad_attention_weights, void *grad_value,
                  void *grad_sampling_locations, void *grad_attention_weights, void *workspace,
                  size_t workspace_bytes, cudaStream_t stream) {
    return msda::backward_entry(desc, grad_output, value, sampling_locations, attention_weights, compute_grad_value,
                                compute_grad_sampling_locations, compute_grad_attention_weights, grad_value,
                                grad_sampling_locations, grad_attention_weights, workspace, workspace_bytes,
                                msda::BwdMode{true, false, false}, stream);
}

int msda_backward_accumulate(const msda_desc *desc, const void *grad_output, const void *value,
                             const void *sampling_locations, const void *attention_weights, int compute_grad_value,
                             int compute_grad_sampling_locations, int compute_grad_attention_weights,
                             float *grad_value_accum, void *grad_sampling_locations, void *grad_attention_weights,
                             void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return msda::backward_entry(desc, grad_output, value, sampling_locations, attention_weights, compute_grad_value,
                                compute_grad_sampling_locations, compute_grad_attention_weights, grad_value_accum,
                                grad_sampling_locations, grad_attention_weights, workspace, workspace_bytes,
                                msda::BwdMode{true, true, false}, stream);
}

int msda_forward_logits(const msda_desc *desc, const void *value, const void *sampling_locations,
                        const void *attention_logits, void *out, cudaStream_t stream) {
    return msda::forward_entry(desc, value, sampling_locations, attention_logits, out, true, false, stream);
}

int msda_backward_logits(const msda_desc *desc, const void *grad_output, const void *value,
                         const void *sampling_locations, const void *attention_logits, int compute_grad_value,
                         int compute_grad_sampling_locations, int compute_grad_attention_logits,
                         void *grad_value, void *grad_sampling_locations, void *grad_attention_logits,
                         void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return msda::backward_entry(desc, grad_output, value, sampling_locations, attention_logits, compute_grad_value,
                                compute_grad_sampling_locations, compute_grad_attention_logits, grad_value,
                                grad_sampling_locations, grad_attention_logits, workspace, workspace_bytes,
                                msda::BwdMode{true, false, true}, stream);
}

const char *msda_status_string(int status) {
    switch (status) {
    case MSDA_OK: return "success";
    case MSDA_ERR_NULL_POINTER: return "a required pointer is NULL";
    case MSDA_ERR_BAD_ENUM: return "an enum or flag argument is out of range";
    case MSDA_ERR_BAD_DIM: return "a dimension is negative or N_l exceeds MSDA_MAX_LEVELS";
    case MSDA_ERR_NO_OUTPUT: return "all compute_grad_* flags are 0; at least one must be 1";
    case MSDA_ERR_LEVELS: return "spatial_shapes / level_start_index / L are inconsistent";
    case MSDA_ERR_WORKSPACE: return "workspace is smaller than msda_backward_workspace_size()";
    case MSDA_ERR_TOO_LARGE: return "a size exceeds the library's 32-bit index limits";
    case MSDA_ERR_UNSUPPORTED: return "valid but unsupported combination (binary16 value, or C_h > 256 unaligned)";
    case MSDA_ERR_MISALIGNED: return "a pointer is not aligned to its element size";
    case MSDA_ERR_CUDA: return "the CUDA runtime reported an error (see msda_last_cuda_error)";
    case MSDA_ERR_STAGE_COPY:
        return "a staged-forward block exited before its shared-memory copy landed; staged results since "
               "then are suspect";
    default: return "unknown status";
    }
}

int msda_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"
