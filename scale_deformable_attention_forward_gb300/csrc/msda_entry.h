// msda_entry.h -- the backward behind msda_backward and msda_backward_noalloc.
#pragma once

#include "msda.h"

namespace msda {

// Workspace bytes of the backward.  allow_sort = false plans the direct
// atomic grad_value (workspace: the binary32 accumulator for bfloat16 value
// only); true lets the library choose the cell-sorted grad_value.
size_t backward_workspace_bytes(const msda_desc *desc, int compute_grad_value, bool allow_sort);

// msda_backward's argument checks and work, with the same allow_sort choice.
int backward_entry(const msda_desc *desc, const void *grad_output, const void *value,
                   const void *sampling_locations, const void *attention_weights, int compute_grad_value,
                   int compute_grad_sampling_locations, int compute_grad_attention_weights, void *grad_value,
                   void *grad_sampling_locations, void *grad_attention_weights, void *workspace,
                   size_t workspace_bytes, bool allow_sort, cudaStream_t stream);

}  // namespace msda
