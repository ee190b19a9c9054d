/*
 * msda.h -- C ABI of libmsda: multi-scale deformable attention (MSDA),
 * forward and backward, on an NVIDIA GB300 (sm_103a).
 *
 * The operations follow two pages of the AWS Neuron NKI library:
 *   "MS Deformable Attention Kernel API Reference" (the forward:
 *    Background, Parameters, Returns) and
 *   "MS Deformable Attention Backward Kernel API Reference" (the backward:
 *    Background, Parameters, Returns, Notes).
 *
 * Definitions used by every entry point.  A sample s = (b, q, h, l, p) has a
 * normalised location (x, y) and an attention weight A_s.  Its pixel
 * coordinate on level l (H_l rows, W_l columns) is
 *     align_corners = 0:  px = x * W_l - 0.5,   py = y * H_l - 0.5
 *     align_corners = 1:  px = x * (W_l - 1),   py = y * (H_l - 1)
 * (forward page, Parameters: align_corners).  The sample S_s is the bilinear
 * interpolation of the head-h value map of level l at (px, py), over the four
 * corners of the cell floor(px), floor(py).  With padding "zeros" a corner
 * outside the map reads 0; with "border" each corner index is clamped into
 * the map (Parameters: padding_mode; backward page, Notes).  Pixel (y, x) of
 * level l is row level_start_index[l] + y * W_l + x of the flattened L axis.
 *     out[b, q, h*C_h + c] = sum_l sum_p A_s * S_s[c]      (forward, Returns)
 * The backward returns the derivatives of <grad_output, out> with respect to
 * value, sampling_locations and attention_weights (backward page, Background
 * and Returns).
 *
 * Memory and threading rules for every call:
 *   - All tensor pointers are DEVICE pointers, C-contiguous in the layout the
 *     descriptor names, owned by the caller.  The library allocates nothing,
 *     keeps no pointer after the call returns and never synchronises.
 *   - spatial_shapes and level_start_index are HOST arrays read during the
 *     call only.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) on the current device.  Results are ready
 *     when the stream reaches that point.
 *   - Every argument is validated before anything is enqueued: a call that
 *     returns an error has not touched any output.
 *   - Functions are thread-safe; concurrent calls on different streams may
 *     not share output buffers.
 */
#ifndef MSDA_H
#define MSDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's stream handle (same declaration as in driver_types.h). */
typedef struct CUstream_st *cudaStream_t;

/* Layout of `value` and of `grad_value` (forward page, Parameters: value,
 * value_layout).  Default BLNC. */
enum msda_value_layout {
    MSDA_LAYOUT_BLNC = 0, /* (B, L, N_h, C_h) */
    MSDA_LAYOUT_BNLC = 1  /* (B, N_h, L, C_h) */
};

/* Layout of `sampling_locations` and its gradient (forward page, Parameters:
 * sampling_locations, sampling_locations_layout).  The "2" axis holds (x, y):
 * x runs along the width W_l, y along the height H_l.  Default BQHLP2. */
enum msda_loc_layout {
    MSDA_LAYOUT_BQHLP2 = 0, /* (B, N_q, N_h, N_l, N_p, 2) */
    MSDA_LAYOUT_B2QHLP = 1  /* (B, 2, N_q, N_h, N_l, N_p) */
};

/* padding_mode (forward page, Parameters; backward page, Notes). */
enum msda_padding {
    MSDA_PADDING_ZEROS = 0, /* a bilinear corner outside the map reads 0 */
    MSDA_PADDING_BORDER = 1 /* a bilinear corner is clamped onto the edge */
};

/* Element types. */
enum msda_dtype {
    MSDA_DTYPE_F32 = 0,  /* IEEE binary32 */
    MSDA_DTYPE_BF16 = 1, /* bfloat16; arithmetic is binary32, stores round to nearest even */
    MSDA_DTYPE_F16 = 2   /* IEEE binary16 (loc_dtype only); arithmetic is binary32, stores round
                            to nearest even */
};

/* Status codes: 0 on success, negative on failure. */
enum msda_status {
    MSDA_OK = 0,
    MSDA_ERR_NULL_POINTER = -1, /* a tensor with elements, the descriptor or a level array is NULL */
    MSDA_ERR_BAD_ENUM = -2,     /* layout / padding / dtype / flag value out of range */
    MSDA_ERR_BAD_DIM = -3,      /* a dimension is negative, or N_l > MSDA_MAX_LEVELS */
    MSDA_ERR_NO_OUTPUT = -4,    /* backward with all three compute_grad_* flags 0 */
    MSDA_ERR_LEVELS = -5,       /* H_l or W_l < 1, level_start_index[0] != 0,
                                   start[l+1] != start[l] + H_l*W_l, or L != sum H_l*W_l */
    MSDA_ERR_WORKSPACE = -6,    /* workspace smaller than msda_backward_workspace_size() */
    MSDA_ERR_TOO_LARGE = -7,    /* a size exceeds the 32-bit index limits stated below */
    MSDA_ERR_UNSUPPORTED = -8,  /* a valid but unimplemented combination (value_dtype F16,
                                   C_h > 256 with unaligned pointers) */
    MSDA_ERR_MISALIGNED = -9,   /* a pointer not aligned to its element size */
    MSDA_ERR_CUDA = -10,        /* the CUDA runtime reported an error (msda_last_cuda_error) */
    MSDA_ERR_STAGE_COPY = -11   /* msda_staged_timeouts: a staged-forward block exited while its
                                   shared-memory copy was still in flight (see there) */
};

/* Levels the descriptor may describe. */
#define MSDA_MAX_LEVELS 16

/* Problem descriptor.  Dimensions follow the pages' Dimensions list:
 *   B batch, N_q queries, N_h heads, C_h channels per head, N_l levels,
 *   N_p points per query, head and level, L = sum_l H_l * W_l.
 * Zero-sized dimensions are allowed (empty tensors).  Index limits (the
 * kernels form element offsets in 32-bit arithmetic): (L + 2*max_l W_l + 4)
 * * N_h * C_h, N_q * N_h * N_l * N_p * 2 and B * N_q * N_h must each be at
 * most 2^31 - 1 (MSDA_ERR_TOO_LARGE otherwise; whole-quotient checks, so a
 * size a few elements short of the bound may be refused too). */
typedef struct msda_desc {
    int64_t B, N_q, N_h, C_h, N_l, N_p, L;
    const int64_t *spatial_shapes;    /* host, N_l pairs (H_l, W_l) */
    const int64_t *level_start_index; /* host, N_l entries; start of level l in L */
    int32_t value_layout;             /* enum msda_value_layout */
    int32_t loc_layout;               /* enum msda_loc_layout */
    int32_t align_corners;            /* 0 or 1 (default 0) */
    int32_t padding_mode;             /* enum msda_padding */
    int32_t value_dtype;              /* enum msda_dtype of value, out, grad_output, grad_value */
    int32_t loc_dtype;                /* enum msda_dtype of sampling_locations,
                                         attention_weights (or logits) and their
                                         gradients: F32, BF16 or F16.  The pages
                                         leave it open; 16-bit locations quantise
                                         a 167-pixel level to ~0.3-1 pixel */
} msda_desc;

/* Forward ("MS Deformable Attention Kernel API Reference", Parameters and
 * Returns).
 *   value               (B,L,N_h,C_h) or (B,N_h,L,C_h), value_dtype
 *   sampling_locations  (B,N_q,N_h,N_l,N_p,2) or (B,2,N_q,N_h,N_l,N_p), loc_dtype
 *   attention_weights   (B,N_q,N_h,N_l,N_p), loc_dtype
 *   out                 (B,N_q,N_h*C_h), value_dtype, column h*C_h + c;
 *                       fully overwritten.
 * Returns MSDA_OK or a negative msda_status. */
int msda_forward(const msda_desc *desc, const void *value, const void *sampling_locations,
                 const void *attention_weights, void *out, cudaStream_t stream);

/* The forward with a staged gather (the same operation as msda_forward:
 * "MS Deformable Attention Kernel API Reference", Parameters and Returns;
 * the page's gather_method chooses how the kernel fetches value rows, and
 * this is the GPU counterpart of choosing).  Each thread block serves a run of
 * queries of one (b, h) and first copies the coarsest levels of that head
 * whose pixels fit 40 KB of shared memory, as TMA tensor copies, into shared
 * memory; samples on those levels read their corners from there, samples on
 * finer levels from global memory.  out is bit-identical to msda_forward's.
 * Arguments, layouts, ownership and errors are msda_forward's.  The staged
 * kernel applies to binary32 locations and weights, C_h * sizeof(value
 * element) a multiple of 16 bytes, C_h <= 64, value 16-byte aligned and
 * L >= 32; otherwise, and when no level
 * fits, the call runs msda_forward's kernel.  A block whose copy has not
 * completed after a bounded wait gathers every level from global memory and
 * is counted (msda_staged_timeouts).  The first call on a device looks up
 * that counter's device address: make it before any stream capture. */
int msda_forward_staged(const msda_desc *desc, const void *value, const void *sampling_locations,
                        const void *attention_weights, void *out, cudaStream_t stream);

/* The number of staged-forward blocks, since the library was loaded, that
 * gave up waiting for their shared-memory copy (expected 0), in *count.  Such
 * a block gathers from global memory instead (same results) and waits for the
 * copy once more, bounded, before it exits; if that wait runs out too, the
 * copy may still write into shared memory that a later block on the same
 * multiprocessor owns, and this call returns MSDA_ERR_STAGE_COPY (the staged
 * outputs produced since are suspect; *count is still written).  Synchronises
 * with the device.  Returns MSDA_OK, MSDA_ERR_STAGE_COPY,
 * MSDA_ERR_NULL_POINTER or MSDA_ERR_CUDA. */
int msda_staged_timeouts(unsigned int *count);

/* The first level msda_forward_staged stages for this descriptor (levels
 * first_level..N_l-1 go to shared memory), N_l when it would run
 * msda_forward's kernel; assumes a 16-byte aligned value.  Host only.
 * Returns MSDA_OK or the descriptor's validation status. */
int msda_forward_staged_levels(const msda_desc *desc, int *first_level);

/* The backward with a per-level shared-memory grad_value accumulator (the
 * same operation as msda_backward: "MS Deformable Attention Backward Kernel
 * API Reference", Parameters and Returns; the page scatters grad_value into
 * several HBM buffers, and a per-block accumulator is the GPU counterpart).
 * Each thread block serves a run of queries of one (b, h) and keeps a
 * binary32 accumulator for the coarsest levels of that head whose pixels fit
 * 40 KB of shared memory; samples on those levels add their corner
 * contributions there, samples on finer levels straight into grad_value's
 * accumulator, and the block adds its shared rows in at its end.
 * grad_sampling_locations and grad_attention_weights are bit-identical to
 * msda_backward's; grad_value equals it up to summation order.  Arguments,
 * workspace size, ownership and errors are msda_backward's.  Applies when
 * grad_value is requested with C_h a multiple of 4 and at most 64 and
 * 16-byte aligned tensors; otherwise msda_backward's kernels run. */
int msda_backward_staged(const msda_desc *desc, const void *grad_output, const void *value,
                         const void *sampling_locations, const void *attention_weights,
                         int compute_grad_value, int compute_grad_sampling_locations,
                         int compute_grad_attention_weights, void *grad_value,
                         void *grad_sampling_locations, void *grad_attention_weights, void *workspace,
                         size_t workspace_bytes, cudaStream_t stream);

/* The first level msda_backward_staged accumulates in shared memory for this
 * descriptor (N_l when it runs msda_backward's kernels), assuming aligned
 * tensors and grad_value requested.  Host only.  Returns MSDA_OK or the
 * descriptor's validation status. */
int msda_backward_staged_levels(const msda_desc *desc, int *first_level);

/* Bytes of device workspace msda_backward needs, 0 when compute_grad_value is
 * 0.  With compute_grad_value set it is the sum of (each part starting at a
 * 256-byte boundary of the workspace):
 *   - B*L*N_h*C_h*4, a binary32 grad_value accumulator, when value_dtype is
 *     BF16;
 *   - when the problem has at least two samples per bilinear cell on average
 *     (S = B*N_q*N_h*N_l*N_p >= 2*B*N_h*sum_l (H_l+1)*(W_l+1), C_h a multiple
 *     of 4, S < 2^31 and B*N_h*N_q < 2^24): the buffers of the tile-sorted
 *     grad_value, which calls with grad_value as the only output use --
 *     4*(T*P + 1) bytes of per-tile and per-block counts (T tiles of 16x16
 *     cells over all levels and (b, h), P = min(1024, ceil(B*N_h*N_q/512))
 *     partition blocks), 4*(T + 1) bytes of chunk counts, the scans' partial
 *     sums and 16*S bytes of sample entries.
 * The size depends on the descriptor and the flag only.  Returns 0 for an
 * invalid descriptor. */
size_t msda_backward_workspace_size(const msda_desc *desc, int compute_grad_value);

/* Backward ("MS Deformable Attention Backward Kernel API Reference",
 * Parameters and Returns; gradients are the bilinear-interpolation
 * derivatives, Notes).
 *   grad_output         (B,N_q,N_h*C_h), value_dtype
 *   value               as in msda_forward; may be NULL when only
 *                       compute_grad_value is set (it is not read then)
 *   sampling_locations  as in msda_forward
 *   attention_weights   as in msda_forward; may be NULL when only
 *                       compute_grad_attention_weights is set
 *   compute_grad_*      0 or 1 each, at least one 1 (Parameters:
 *                       compute_grad_value / _sampling_locations /
 *                       _attention_weights)
 *   grad_value          value's shape, layout and dtype; overwritten
 *   grad_sampling_locations  sampling_locations' shape and layout, binary32
 *   grad_attention_weights   (B,N_q,N_h,N_l,N_p), binary32
 *   A disabled output is neither read nor written and may be NULL.
 *   workspace           device scratch of at least
 *                       msda_backward_workspace_size(desc, compute_grad_value)
 *                       bytes (NULL when that is 0), 16-byte aligned; its
 *                       contents on entry do not matter.
 * grad_value is accumulated in binary32 with atomic adds (per corner and
 * sample, or per cell of samples grouped by cell), so its summation order
 * (and last-bit rounding) varies from run to run.
 * Returns MSDA_OK or a negative msda_status. */
int msda_backward(const msda_desc *desc, const void *grad_output, const void *value,
                  const void *sampling_locations, const void *attention_weights,
                  int compute_grad_value, int compute_grad_sampling_locations,
                  int compute_grad_attention_weights, void *grad_value,
                  void *grad_sampling_locations, void *grad_attention_weights, void *workspace,
                  size_t workspace_bytes, cudaStream_t stream);

/* Accumulating backward ("MS Deformable Attention Backward Kernel API
 * Reference", Parameters: grad_value_buffers_in, prev_reduced_grad_value,
 * dump_reduced_grad_value).  The pages let a call add into persistent
 * grad_value buffers instead of zeroing them, so that calls over query chunks
 * or over several micro-batches build one total.  Here that state is one
 * caller-owned binary32 buffer:
 *   grad_value_accum    binary32, value's shape and layout, 4-byte aligned
 *                       (16-byte for the vector path); this call's grad_value
 *                       is ADDED to it (read-modify-write, never zeroed, never
 *                       rounded to value_dtype, also for BF16 value).
 * Every other argument is as in msda_backward (the workspace size is
 * msda_backward_workspace_size's; the accumulator part of it is not used).
 * grad_sampling_locations and grad_attention_weights are overwritten as in
 * msda_backward.  After the call grad_value_accum = its previous contents +
 * this call's grad_value, up to binary32 rounding in an unspecified order
 * (atomic adds).  Calls that overlap on the GPU may add into the same
 * accumulator.  Returns MSDA_OK or a negative msda_status; a failed call
 * leaves the accumulator untouched. */
int msda_backward_accumulate(const msda_desc *desc, const void *grad_output, const void *value,
                             const void *sampling_locations, const void *attention_weights,
                             int compute_grad_value, int compute_grad_sampling_locations,
                             int compute_grad_attention_weights, float *grad_value_accum,
                             void *grad_sampling_locations, void *grad_attention_weights, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/* Forward and backward with attention LOGITS.  The pages take attention
 * weights as an input ("MS Deformable Attention Kernel API Reference",
 * Parameters: attention_weights); models produce them as a softmax over the
 * N_l*N_p (level, point) slots of each (b, q, h) (the workloads here are built
 * that way).  These entry points fuse that producer: attention_logits has
 * attention_weights' shape and dtype, and for every (b, q, h)
 *     A[l, p] = exp(z[l, p] - m) / sum_{l', p'} exp(z[l', p'] - m),
 *     m = max z over the row,
 * then the operation is msda_forward / msda_backward with those weights.
 * msda_backward_logits returns in grad_attention_logits the gradient with
 * respect to the logits,
 *     dz[l, p] = A[l, p] * (gA[l, p] - sum_{l', p'} A[l', p'] gA[l', p']),
 * gA being the attention-weight gradient; attention_logits is read for every
 * output flag.  All other arguments, results, ownership and errors are those
 * of msda_forward / msda_backward (same workspace size). */
int msda_forward_logits(const msda_desc *desc, const void *value, const void *sampling_locations,
                        const void *attention_logits, void *out, cudaStream_t stream);
int msda_backward_logits(const msda_desc *desc, const void *grad_output, const void *value,
                         const void *sampling_locations, const void *attention_logits,
                         int compute_grad_value, int compute_grad_sampling_locations,
                         int compute_grad_attention_logits, void *grad_value, void *grad_sampling_locations,
                         void *grad_attention_logits, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/* Size of the library-owned scratch array used by msda_backward_noalloc:
 * 32 MiB, i.e. room for a binary32 accumulator of B*L*N_h*C_h <= 8,388,608
 * elements (one 4-level Deformable-DETR pyramid image with 8 heads of 32
 * channels needs 5,689,088). */
#define MSDA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* msda_backward for callers that cannot allocate device memory.  The pages
 * have no counterpart: it exists for hosts that may not call cudaMalloc (a
 * plug-in living inside another application's memory pool, a loop where
 * allocation is forbidden after start-up, a caller that can only hand over
 * the tensors it already owns).
 *
 * Arguments and results are those of msda_backward without the workspace:
 * the binary32 grad_value accumulator that bfloat16 value needs lives in a
 * fixed array inside the library (MSDA_NOALLOC_SCRATCH_BYTES, held on every
 * GPU that loads the library until the process exits).  A problem whose
 * accumulator would not fit (bfloat16 value, compute_grad_value set and
 * B*L*N_h*C_h*4 > MSDA_NOALLOC_SCRATCH_BYTES) is refused with
 * MSDA_ERR_WORKSPACE before anything is enqueued; binary32 value needs no
 * scratch and has no such limit.  Nothing is allocated.
 *
 * The first call on a device looks up the array's device address on that
 * (current) device; make that first call before any stream capture.  All
 * calls share the one array, which keeps the last call's contents (each call
 * clears what it uses): calls whose GPU work overlaps -- different streams,
 * or unordered host threads -- race on it and corrupt grad_value.  Returns
 * MSDA_OK or a negative msda_status (MSDA_ERR_CUDA also when the address
 * lookup fails). */
int msda_backward_noalloc(const msda_desc *desc, const void *grad_output, const void *value,
                          const void *sampling_locations, const void *attention_weights,
                          int compute_grad_value, int compute_grad_sampling_locations,
                          int compute_grad_attention_weights, void *grad_value,
                          void *grad_sampling_locations, void *grad_attention_weights,
                          cudaStream_t stream);

/* A static, human-readable description of a status code. */
const char *msda_status_string(int status);

/* The cudaError_t behind the calling thread's last MSDA_ERR_CUDA (0 if none). */
int msda_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MSDA_H */
