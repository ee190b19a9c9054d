// msda_noalloc.cu -- msda_backward_noalloc: the backward for callers that
// cannot allocate device memory.
//
// Some callers have no way to obtain a device buffer of their own: code that
// runs inside another framework's allocator regime (a plug-in that must not
// call cudaMalloc behind the host application's memory pool), real-time or
// safety-certified loops where every allocation is forbidden after start-up,
// and hosts that can only pass the tensors they already own.  The bfloat16
// backward needs a binary32 grad_value accumulator that msda_backward takes
// as caller-owned workspace; this entry point uses a fixed array that lives
// in the library instead.
//
// The array is a file-scope __device__ variable of MSDA_NOALLOC_SCRATCH_BYTES
// bytes.  Every GPU that loads the library holds it until the process exits.
// Host code cannot use the array's name as a device address (it is a
// host-side stand-in); the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// it.  That first call on each device should therefore happen before any
// stream capture.
//
// All calls share the one array and it keeps the last call's contents; the
// backward clears the part it uses before accumulating.  Calls whose work
// overlaps on the GPU (different streams, or different host threads without
// ordering) race on the array and give wrong grad_value.
#include "msda.h"
#include "msda_entry.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

constexpr size_t kScratchBytes = (size_t)MSDA_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// The device address of the scratch array on the current device.
int scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return MSDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MSDA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return MSDA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MSDA_OK;
}

}  // namespace

extern "C" int msda_backward_noalloc(const msda_desc *desc, const void *grad_output, const void *value,
                                     const void *sampling_locations, const void *attention_weights,
                                     int compute_grad_value, int compute_grad_sampling_locations,
                                     int compute_grad_attention_weights, void *grad_value,
                                     void *grad_sampling_locations, void *grad_attention_weights,
                                     cudaStream_t stream) {
    if (!desc) return MSDA_ERR_NULL_POINTER;
    // Refuse, before anything else, a problem whose accumulator does not fit.
    // The size is computed here from the descriptor alone, in 64-bit
    // arithmetic that cannot overflow for dimensions the library accepts.
    const int64_t dims[4] = {desc->B, desc->L, desc->N_h, desc->C_h};
    bool needs_scratch = compute_grad_value == 1 && desc->value_dtype == MSDA_DTYPE_BF16;
    if (needs_scratch) {
        uint64_t elems = 1;
        for (int i = 0; i < 4; ++i) {
            if (dims[i] < 0) return MSDA_ERR_BAD_DIM;
            if (dims[i] == 0) {
                elems = 0;
                break;
            }
            if (elems > (uint64_t)kScratchBytes / (uint64_t)dims[i]) return MSDA_ERR_WORKSPACE;
            elems *= (uint64_t)dims[i];
        }
        if (elems * sizeof(float) > kScratchBytes) return MSDA_ERR_WORKSPACE;
    }
    // grad_value goes straight into the accumulator with atomics here: the
    // tile-sorted path's buffers grow with the number of samples.
    const size_t need = msda::backward_workspace_bytes(desc, compute_grad_value, false);
    if (need > kScratchBytes) return MSDA_ERR_WORKSPACE;
    void *ws = nullptr;
    if (need > 0) {
        const int rc = scratch_address(&ws);
        if (rc != MSDA_OK) return rc;
    }
    // The backward validates every argument, zeroes the part of the
    // accumulator it uses and enqueues the kernels on `stream`.
    return msda::backward_entry(desc, grad_output, value, sampling_locations, attention_weights,
                                compute_grad_value, compute_grad_sampling_locations,
                                compute_grad_attention_weights, grad_value, grad_sampling_locations,
                                grad_attention_weights, ws, need, msda::BwdMode{false, false, false}, stream);
}
