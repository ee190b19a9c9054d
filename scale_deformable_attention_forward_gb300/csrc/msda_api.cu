// msda_api.cu -- the C ABI declared in include/msda.h: argument validation,
// kernel parameter set-up and dispatch, plus the two small helper kernels
// (accumulator zero-fill and binary32 -> bfloat16 conversion).
#include "msda.h"
#include "msda_kernels.cuh"
#include "msda_shape.cuh"

#include <limits.h>
#include <string.h>

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

// Shape, enum and level checks shared by every entry point ("MS Deformable
// Attention Kernel API Reference", Parameters: spatial_shapes,
// level_start_index; Dimensions: L is the sum of H_i * W_i).
int validate_desc(const msda_desc *d) {
    if (!d) return MSDA_ERR_NULL_POINTER;
    if (d->value_layout != MSDA_LAYOUT_BLNC && d->value_layout != MSDA_LAYOUT_BNLC) return MSDA_ERR_BAD_ENUM;
    if (d->loc_layout != MSDA_LAYOUT_BQHLP2 && d->loc_layout != MSDA_LAYOUT_B2QHLP) return MSDA_ERR_BAD_ENUM;
    if (d->padding_mode != MSDA_PADDING_ZEROS && d->padding_mode != MSDA_PADDING_BORDER) return MSDA_ERR_BAD_ENUM;
    if (d->align_corners != 0 && d->align_corners != 1) return MSDA_ERR_BAD_ENUM;
    if (d->value_dtype != MSDA_DTYPE_F32 && d->value_dtype != MSDA_DTYPE_BF16) return MSDA_ERR_BAD_ENUM;
    if (d->loc_dtype != MSDA_DTYPE_F32 && d->loc_dtype != MSDA_DTYPE_BF16) return MSDA_ERR_BAD_ENUM;
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
    if (d->loc_dtype != MSDA_DTYPE_F32) return MSDA_ERR_UNSUPPORTED;
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
    p.padding = d->padding_mode;
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
    return p;
}

// Shared memory a block may give to privatised grad_value levels.
#ifndef MSDA_PRIV_SMEM_BYTES
#define MSDA_PRIV_SMEM_BYTES (160 * 1024)
#endif

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

// Backward work split: queries per block, and which levels each block
// accumulates in shared memory.  A level is privatised (smallest levels first,
// within MSDA_PRIV_SMEM_BYTES) only if a block adds, on average, at least two
// corner contributions per privatised pixel: below that the flush costs more
// atomics than it saves.  Privatising blocks hold one (b, h) and a long run of
// queries, sized so the blocks fill whole waves of the GPU.
void plan_backward(const msda_desc *d, const Config &cfg, bool want_gv, int n_sm, Params *p, bool *priv) {
    const int groups = msda::kBwdThreads / cfg.G;
    const int64_t BH = d->B * d->N_h;
    *priv = false;
    for (int l = 0; l < msda::kMaxLevels; ++l) p->priv_start[l] = -1;
    p->priv_pixels = 0;
    p->swizzle = (d->C_h % 32 == 0) ? 1 : 0;
    int64_t q_chunk = groups;  // one query row per group
    if (want_gv && cfg.vec && cfg.G <= 8 && d->C_h % 4 == 0 && d->N_l > 0 && n_sm > 0 && BH > 0) {
        // smallest levels first
        int order[msda::kMaxLevels];
        for (int l = 0; l < d->N_l; ++l) order[l] = l;
        for (int a = 1; a < d->N_l; ++a)
            for (int b2 = a; b2 > 0 && p->H[order[b2]] * (int64_t)p->W[order[b2]] <
                                           p->H[order[b2 - 1]] * (int64_t)p->W[order[b2 - 1]]; --b2) {
                const int t = order[b2]; order[b2] = order[b2 - 1]; order[b2 - 1] = t;
            }
        int64_t pixels = 0;
        int nlev = 0;
        int start[msda::kMaxLevels];
        for (int i = 0; i < d->N_l; ++i) {
            const int l = order[i];
            const int64_t hw = (int64_t)p->H[l] * p->W[l];
            if ((pixels + hw) * d->C_h * 4 > MSDA_PRIV_SMEM_BYTES) break;
            start[l] = (int)pixels;
            pixels += hw;
            ++nlev;
        }
        if (nlev > 0) {
            // blocks: one (b, h) and ceil(N_q / chunks) queries each; pick the
            // chunk count that fills whole waves best, with at least two waves
            int64_t best = 1;
            double best_eff = -1.0;
            for (int64_t c = 1; c <= 256; ++c) {
                const int64_t blocks = BH * c;
                if (blocks < 2 * n_sm && c < 256) continue;
                const int64_t waves = (blocks + n_sm - 1) / n_sm;
                const double eff = (double)blocks / (double)(waves * n_sm);
                if (eff > best_eff + 1e-9) {
                    best_eff = eff;
                    best = c;
                }
                if (blocks >= 8 * n_sm) break;
            }
            const int64_t qc = (d->N_q + best - 1) / best;
            const int64_t adds = qc * d->N_p * nlev * 4;
            if (qc >= groups && adds >= 2 * pixels) {
                *priv = true;
                q_chunk = qc;
                p->priv_pixels = (int)pixels;
                for (int i = 0; i < nlev; ++i) p->priv_start[order[i]] = start[order[i]];
            }
        }
    }
    // at most 65535 query chunks per (b, h) (the grid's y extent)
    const int64_t min_chunk = (d->N_q + 65534) / 65535;
    if (q_chunk < min_chunk) q_chunk = ((min_chunk + groups - 1) / groups) * groups;
    p->q_chunk = (int)(q_chunk < 1 ? 1 : q_chunk);
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

}  // namespace msda

extern "C" {

int msda_forward(const msda_desc *desc, const void *value, const void *sampling_locations,
                 const void *attention_weights, void *out, cudaStream_t stream) {
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
    if (!aligned(value, es) || !aligned(out, es) || !aligned(sampling_locations, 4) ||
        !aligned(attention_weights, 4))
        return MSDA_ERR_MISALIGNED;
    Config cfg;
    const int V = d->value_dtype == MSDA_DTYPE_BF16 ? msda::VecWidth<__nv_bfloat16>::value
                                                     : msda::VecWidth<float>::value;
    rc = choose_config(d, V, aligned(value, V * es) && aligned(out, V * es), MSDA_FWD_LANES, &cfg);
    if (rc) return rc;
    if (out_elems == 0) return MSDA_OK;
    Params p = make_params(d, cfg, V);
    p.n_sm = sm_count();
    cudaError_t e;
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

size_t msda_backward_workspace_size(const msda_desc *desc, int compute_grad_value) {
    if (validate_desc(desc) != MSDA_OK) return 0;
    if (!compute_grad_value || desc->value_dtype != MSDA_DTYPE_BF16) return 0;
    return (size_t)(desc->B * desc->L * desc->N_h * desc->C_h) * sizeof(float);
}

int msda_backward(const msda_desc *desc, const void *grad_output, const void *value,
                  const void *sampling_locations, const void *attention_weights, int compute_grad_value,
                  int compute_grad_sampling_locations, int compute_grad_attention_weights, void *grad_value,
                  void *grad_sampling_locations, void *grad_attention_weights, void *workspace,
                  size_t workspace_bytes, cudaStream_t stream) {
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
    const bool need_a = (fv || fl) && samples > 0;
    if (samples > 0 && !sampling_locations) return MSDA_ERR_NULL_POINTER;
    if (samples > 0 && go_elems > 0 && !grad_output) return MSDA_ERR_NULL_POINTER;
    if (need_v && !value) return MSDA_ERR_NULL_POINTER;
    if (need_a && !attention_weights) return MSDA_ERR_NULL_POINTER;
    if (fv && value_elems > 0 && !grad_value) return MSDA_ERR_NULL_POINTER;
    if (fl && samples > 0 && !grad_sampling_locations) return MSDA_ERR_NULL_POINTER;
    if (fa && samples > 0 && !grad_attention_weights) return MSDA_ERR_NULL_POINTER;
    const size_t es = value_elem_size(d);
    if (!aligned(grad_output, es) || !aligned(value, es) || !aligned(grad_value, es) ||
        !aligned(sampling_locations, 4) || !aligned(attention_weights, 4) ||
        !aligned(grad_sampling_locations, 4) || !aligned(grad_attention_weights, 4))
        return MSDA_ERR_MISALIGNED;
    const bool bf16 = d->value_dtype == MSDA_DTYPE_BF16;
    const size_t ws_need = msda_backward_workspace_size(d, fv);
    if (ws_need > 0) {
        if (workspace_bytes < ws_need) return MSDA_ERR_WORKSPACE;
        if (!workspace) return MSDA_ERR_NULL_POINTER;
        if (!aligned(workspace, 16)) return MSDA_ERR_MISALIGNED;
    }
    float *acc = fv ? (bf16 ? (float *)workspace : (float *)grad_value) : nullptr;
    Config cfg;
    const int V = d->value_dtype == MSDA_DTYPE_BF16 ? msda::BwdVecWidth<__nv_bfloat16>::value
                                                     : msda::BwdVecWidth<float>::value;
    rc = choose_config(d, V,
                       aligned(grad_output, V * es) && aligned(value, V * es) && (!fv || aligned(acc, 16)),
                       MSDA_BWD_LANES, &cfg);
    if (rc) return rc;
    Params p = make_params(d, cfg, V);
    p.flags = (fv ? msda::kGradValue : 0) | (fl ? msda::kGradLoc : 0) | (fa ? msda::kGradAttn : 0);
    bool priv = false;
    p.n_sm = samples > 0 ? sm_count() : 0;
    plan_backward(d, cfg, fv != 0, p.n_sm, &p, &priv);

    cudaError_t e = cudaSuccess;
    if (fv) e = msda::launch_zero_f32(acc, value_elems, stream);
    if (e == cudaSuccess && samples > 0) {
        if (bf16)
            e = msda::launch_backward<__nv_bfloat16>(
                p, cfg.vec, cfg.G, cfg.NCH, priv, (const __nv_bfloat16 *)grad_output, (const __nv_bfloat16 *)value,
                (const float *)sampling_locations, (const float *)attention_weights, acc,
                (float *)grad_sampling_locations, (float *)grad_attention_weights, stream);
        else
            e = msda::launch_backward<float>(p, cfg.vec, cfg.G, cfg.NCH, priv, (const float *)grad_output,
                                             (const float *)value, (const float *)sampling_locations,
                                             (const float *)attention_weights, acc,
                                             (float *)grad_sampling_locations, (float *)grad_attention_weights,
                                             stream);
    }
    if (e == cudaSuccess && fv && bf16)
        e = msda::launch_f32_to_bf16(acc, (__nv_bfloat16 *)grad_value, value_elems, stream);
    return record_cuda(e);
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
    case MSDA_ERR_UNSUPPORTED: return "valid but unsupported combination (bf16 locations, or C_h > 256 unaligned)";
    case MSDA_ERR_MISALIGNED: return "a pointer is not aligned to its element size";
    case MSDA_ERR_CUDA: return "the CUDA runtime reported an error (see msda_last_cuda_error)";
    default: return "unknown status";
    }
}

int msda_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"
