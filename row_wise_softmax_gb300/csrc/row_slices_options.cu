// CTA and CLUSTER paths with softmax_options_t (scale, causal mask): the
// kernel of row_slices.cu instantiated with OPTS = true.  A translation unit
// of its own so that the two sets of instantiations compile in parallel.
#define RWSM_ROW_SLICES_OPTIONS 1
#include "row_slices.cu"
