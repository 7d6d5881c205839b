// prefix_early.cu -- the early-start variants of the prefix pass kernel (the
// plan and the first committed-prefix K/V loads issued before the dependency
// wait on the previous kernel; see tree_attn_set_early_prefix_loads in
// tree_attn.h).  They are the same kernel template as kernels.cu's, compiled
// in a translation unit of their own so that the two build in parallel.
#define TREE_ATTN_EARLY_TU 1
#include "kernels.cu"
