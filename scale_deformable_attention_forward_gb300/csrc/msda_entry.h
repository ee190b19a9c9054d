// msda_entry.h -- the backward behind msda_backward and msda_backward_noalloc.
#pragma once

#include "msda.h"

namespace msda {

// Workspace bytes of the backward.  allow_sort = false plans the direct
// atomic grad_value (workspace: the binary32 accumulator for bfloat16 value
// only); true lets the library choose the cell-sorted grad_value.
size_t backward_workspace_bytes(const msda_desc *desc, int compute_grad_value, bool allow_sort);

// How a backward entry point differs from msda_backward:
//   allow_sort  as for backward_workspace_bytes;
//   accumulate  grad_value is a caller-owned binary32 accumulator (value's
//               shape and layout) that this call's grad_value is added to,
//               without zeroing and without conversion;
//   logits      attention_weights holds logits (softmax over each row's
//               N_l*N_p slots gives the weights) and grad_attention_weights
//               receives the logits' gradient;
//   staged      grad_value of the coarse levels accumulated per block in
//               shared memory where that kernel applies (msda_backward_staged).
struct BwdMode {
    bool allow_sort, accumulate, logits;
    bool staged = false;
};

// msda_backward's argument checks and work, in the given mode.
int backward_entry(const msda_desc *desc, const void *grad_output, const void *value,
                   const void *sampling_locations, const void *attention_weights, int compute_grad_value,
                   int compute_grad_sampling_locations, int compute_grad_attention_weights, void *grad_value,
                   void *grad_sampling_locations, void *grad_attention_weights, void *workspace,
                   size_t workspace_bytes, BwdMode mode, cudaStream_t stream);

// msda_forward's argument checks and work; logits as in BwdMode; staged:
// the staged-level kernel where it applies (msda_forward_staged).
int forward_entry(const msda_desc *desc, const void *value, const void *sampling_locations,
                  const void *attention_weights, void *out, bool logits, bool staged, cudaStream_t stream);

}  // namespace msda
