// kernels.cuh -- launch interface between the C-ABI layer (tree_attn.cu) and
// the device code (kernels.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace treeattn {

struct VerifyArgs {
    const uint16_t* q;
    const uint16_t* k_pages;
    const uint16_t* v_pages;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const uint16_t* tree_k;
    const uint16_t* tree_v;
    const uint64_t* mask;
    uint16_t* out;
    float* lse;
    float* ws;
    int32_t* status;
    int B, Hq, Hkv, d, T, P, max_pages, num_pages;
    int n_ctas;
    float scale_log2;
    int mask_stride;    // 0: mask[T] shared by the batch; T: mask[B][T]
    int tree_in_cache;  // tree K/V at positions seq_lens[b] .. +T of the paged cache
    // One pass under an explicit mask (uint8 [B][T][dense_cols]); seq_lens
    // then counts every key in the cache and the merge has no suffix
    // (mask == nullptr).  nullptr: the split form.
    const uint8_t* dense;
    int dense_cols;
    // Masks built by the merge kernel from parent arrays ([T] or [B][T],
    // parents_stride 0 or T) instead of read from `mask`; written to
    // mask_out when it is not null.
    const int32_t* parents;
    int parents_stride;
    uint64_t* mask_out;
    // Where the prefix pass finds the tree tokens (TreeMode in layout.h):
    // kTreeNone leaves them to the merge kernel (two-pass form).
    int tmode;
    int ovh;  // overhead slots per unit on the work line (the kernel selector's)
    unsigned long long wait_ns;  // limit of a pipeline wait in the prefix pass
    int early;  // plan and first committed-prefix loads before the dependency wait
};

// Enqueue the explicit-mask builder: dense[b][t][p] for p < dense_cols and
// key_lens[b] = seq_lens[b] + T.
cudaError_t launch_dense_mask_build(const uint64_t* mask, int mask_stride,
                                    const int32_t* seq_lens, int B, int T, int dense_cols,
                                    uint8_t* dense, int32_t* key_lens, int32_t* status,
                                    cudaStream_t stream);

// Enqueue the mask builder (one warp per tree, n_trees trees of T nodes).
cudaError_t launch_mask_build(const int32_t* parents, int T, int n_trees, uint64_t* mask,
                              int32_t* status, cudaStream_t stream);

// Enqueue the prefix pass (partials into a.ws).  `tmap_k`/`tmap_v` point at
// encoded CUtensorMap objects of the paged cache, `tmap_tk`/`tmap_tv` at
// those of the tree K/V buffers (kTreeChunk; otherwise any valid maps).
// All are host memory, copied into the launch.
cudaError_t launch_prefix(const VerifyArgs& a, const void* tmap_k, const void* tmap_v,
                          const void* tmap_tk, const void* tmap_tv, cudaStream_t stream);
// The same for a.early (in prefix_early.cu): the plan and the first committed
// prefix loads go out before the dependency wait.
cudaError_t launch_prefix_early(const VerifyArgs& a, const void* tmap_k, const void* tmap_v,
                                const void* tmap_tk, const void* tmap_tv, cudaStream_t stream);

// Enqueue the suffix pass + merge (reads the partials in a.ws).
cudaError_t launch_merge(const VerifyArgs& a, cudaStream_t stream);

}  // namespace treeattn
