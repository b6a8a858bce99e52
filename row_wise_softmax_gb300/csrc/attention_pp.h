// Launcher of the ping-pong tcgen05 attention kernel: each CTA owns two
// 128-query tiles and overlaps one tile's softmax with the other tile's
// products on the tensor cores; Q, K and V tiles arrive by tensor-memory-
// accelerator copies.  Returns cudaErrorNotSupported, launching nothing, when
// the driver offers no tensor-map encoder, a size does not fit the 32-bit
// copy coordinates or the grid would exceed 2^31 - 1 CTAs.
#pragma once

#include "kernels.h"

namespace rwsm {

cudaError_t launch_attention_pp(const AttentionProblem& p, cudaStream_t s);

}  // namespace rwsm
