// tree_attn.cu -- the C ABI (include/tree_attn.h): argument checks, workspace
// sizing, TMA tensor-map encoding and kernel launches.  No allocation, no
// synchronisation: every call only enqueues work on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/tree_attn.h"
#include "kernels.cuh"
#include "layout.h"

using namespace treeattn;

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Limit of the prefix pass's pipeline waits, read when a call is enqueued.
std::atomic<unsigned long long> g_wait_ns{TREE_ATTN_DEFAULT_WAIT_NS};
std::atomic<int> g_early{0};

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

bool shape_ok(int B, int Hq, int Hkv, int d, int T, int P) {
    if (B < 0 || T < 1 || T > TREE_ATTN_MAX_T || Hkv < 1 || Hq < Hkv || Hq % Hkv != 0) return false;
    if (d != 64 && d != 128) return false;
    if (P != 16 && P != 32 && P != 64 && P != 128) return false;
    return true;
}

size_t ws_bytes(int B, int Hq, int Hkv, int d, int T, int n_ctas) {
    const long long G = Hq / Hkv;
    const long long M = static_cast<long long>(T) * G;
    const long long RB = (M + kRows - 1) / kRows;
    const long long units = static_cast<long long>(B) * Hkv * RB;
    const long long slots = units + n_ctas;
    const size_t bytes = static_cast<size_t>(slots) * slot_floats(d) * sizeof(float);
    return (bytes + 255) & ~static_cast<size_t>(255);
}

// Row-major [rows][d] bf16 view of a paged cache, boxes of `box_rows` x 64.
bool encode_pages(CUtensorMap* map, const void* base, long long rows, int d, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [B*T][Hkv][d] bf16 view of the tree K or V buffer, boxes of 64 tree
// tokens x one head x 64 columns (the tree chunk of one unit).
bool encode_tree(CUtensorMap* map, const void* base, int B, int T, int Hkv, int d) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hkv),
                                static_cast<cuuint64_t>(B) * T};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                   static_cast<cuuint64_t>(Hkv) * d * 2};
    const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kChunk)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Checks shared by the verify, prefix-pass and merge entry points.
int check_common(int B, int Hq, int Hkv, int d, int T, int page_size, int max_pages_per_seq,
                 float softmax_scale) {
    if (!shape_ok(B, Hq, Hkv, d, T, page_size) || max_pages_per_seq < 1 ||
        !std::isfinite(softmax_scale))
        return TREE_ATTN_ERR_SHAPE;
    return TREE_ATTN_OK;
}

// The kernel selector's plan for a call (n_ctas > 0: the caller's count).
// Returns false when the device cannot be queried.
bool plan_call(int n_ctas, int B, int Hq, int Hkv, int T, int P, int max_pages, int tree_layout,
               Plan& plan) {
    const int sms = n_ctas > 0 ? n_ctas : sm_count();
    if (sms <= 0) return false;
    plan = make_plan(B, Hq, Hkv, T, P, max_pages, sms, n_ctas, tree_layout);
    return true;
}

// Overhead slots per unit for these shapes (the kernel selector's choice).
int ovh_for(int Hq, int Hkv, int T) {
    const int M = T * (Hq / Hkv);
    const int F = M <= kRows ? replicas_of(M) : 1;
    return overhead_slots(F, M);
}

// CTAs of the prefix pass: the caller's count, else the kernel selector's.
int resolve_ctas(int n_ctas, int B, int Hq, int Hkv, int T, int P, int max_pages) {
    Plan plan;
    return plan_call(n_ctas, B, Hq, Hkv, T, P, max_pages, kTreeNone, plan) ? plan.n_ctas : 0;
}

float to_log2(float softmax_scale) {
    return static_cast<float>(static_cast<double>(softmax_scale) * 1.4426950408889634);
}

int prefix_impl(VerifyArgs& a, const uint16_t* k_pages, const uint16_t* v_pages,
                cudaStream_t stream) {
    const long long rows = static_cast<long long>(a.num_pages) * a.Hkv * a.P;
    const int box_rows = a.P < kChunk ? a.P : kChunk;
    CUtensorMap tk, tv, ttk, ttv;
    if (!encode_pages(&tk, k_pages, rows, a.d, box_rows) ||
        !encode_pages(&tv, v_pages, rows, a.d, box_rows))
        return TREE_ATTN_ERR_CUDA;
    if (a.tmode == kTreeChunk) {
        if (!encode_tree(&ttk, a.tree_k, a.B, a.T, a.Hkv, a.d) ||
            !encode_tree(&ttv, a.tree_v, a.B, a.T, a.Hkv, a.d))
            return TREE_ATTN_ERR_CUDA;
    } else {
        ttk = tk;  // unused by the kernel in this mode
        ttv = tv;
    }
    return launch_prefix(a, &tk, &tv, &ttk, &ttv, stream) == cudaSuccess ? TREE_ATTN_OK
                                                                        : TREE_ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

int tree_attn_version(void) { return 10200; }

unsigned long long tree_attn_set_wait_limit_ns(unsigned long long ns) {
    return g_wait_ns.exchange(ns == 0 ? TREE_ATTN_DEFAULT_WAIT_NS : ns);
}

int tree_attn_set_early_prefix_loads(int enable) {
    return g_early.exchange(enable != 0 ? 1 : 0);
}

int tree_mask_build_batched(const int32_t* parents, int T, int n_trees, uint64_t* mask_out,
                            int32_t* status, void* stream) {
    if (T < 1 || T > TREE_ATTN_MAX_T || n_trees < 0) return TREE_ATTN_ERR_SHAPE;
    if (n_trees == 0) return TREE_ATTN_OK;
    if (parents == nullptr || mask_out == nullptr) return TREE_ATTN_ERR_NULL;
    if (!aligned(parents, 4) || !aligned(mask_out, 8) || !aligned(status, 4))
        return TREE_ATTN_ERR_ALIGN;
    const cudaError_t e = launch_mask_build(parents, T, n_trees, mask_out, status,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
}

int tree_mask_build(const int32_t* parents, int T, uint64_t* mask_out, int32_t* status,
                    void* stream) {
    if (parents == nullptr || mask_out == nullptr) return TREE_ATTN_ERR_NULL;
    return tree_mask_build_batched(parents, T, 1, mask_out, status, stream);
}

size_t tree_attn_workspace_size_ctas(int B, int Hq, int Hkv, int d, int T, int page_size,
                                     int n_ctas) {
    if (!shape_ok(B, Hq, Hkv, d, T, page_size)) return 0;
    if (n_ctas <= 0) n_ctas = sm_count();
    if (n_ctas <= 0) return 0;
    return ws_bytes(B, Hq, Hkv, d, T, n_ctas);
}

int tree_attn_plan(int B, int Hq, int Hkv, int d, int T, int page_size, int max_pages_per_seq,
                   int sm_count_hint, tree_attn_plan_info* out) {
    if (out == nullptr) return TREE_ATTN_ERR_NULL;
    if (!shape_ok(B, Hq, Hkv, d, T, page_size) || max_pages_per_seq < 1)
        return TREE_ATTN_ERR_SHAPE;
    const int sms = sm_count_hint > 0 ? sm_count_hint : sm_count();
    if (sms <= 0) return TREE_ATTN_ERR_CUDA;
    const Plan p = make_plan(B, Hq, Hkv, T, page_size, max_pages_per_seq, sms, 0, kTreeChunk);
    out->tree_in_prefix = p.tmode != kTreeNone ? 1 : 0;
    out->units = p.units;
    out->row_blocks = p.RB;
    out->replicas = p.F;
    out->n_ctas = p.n_ctas;
    out->merge_warps_per_row = p.merge_wpr;
    out->merge_rows_per_warp = p.merge_rpw;
    out->max_steps = p.max_steps;
    out->workspace_bytes = ws_bytes(B, Hq, Hkv, d, T, p.n_ctas);
    return TREE_ATTN_OK;
}

size_t tree_attn_workspace_size(int B, int Hq, int Hkv, int d, int T, int max_seq_len,
                                int page_size) {
    (void)max_seq_len;
    return tree_attn_workspace_size_ctas(B, Hq, Hkv, d, T, page_size, 0);
}

int tree_attn_prefix_pass(const uint16_t* q, const uint16_t* k_pages, const uint16_t* v_pages,
                          const int32_t* block_table, int max_pages_per_seq,
                          const int32_t* seq_lens, int B, int Hq, int Hkv, int d, int T,
                          int page_size, int num_pages, float softmax_scale, void* workspace,
                          size_t workspace_bytes, int n_ctas, int32_t* status, void* stream) {
    int rc = check_common(B, Hq, Hkv, d, T, page_size, max_pages_per_seq, softmax_scale);
    if (rc != TREE_ATTN_OK) return rc;
    if (num_pages < 1 || static_cast<long long>(num_pages) * Hkv * page_size >= (1LL << 31))
        return TREE_ATTN_ERR_SHAPE;
    if (B == 0) return TREE_ATTN_OK;
    if (!q || !k_pages || !v_pages || !block_table || !seq_lens) return TREE_ATTN_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) ||
        !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(status, 4))
        return TREE_ATTN_ERR_ALIGN;
    n_ctas = resolve_ctas(n_ctas, B, Hq, Hkv, T, page_size, max_pages_per_seq);
    if (n_ctas <= 0) return TREE_ATTN_ERR_CUDA;
    if (workspace == nullptr || !aligned(workspace, 256) ||
        workspace_bytes < ws_bytes(B, Hq, Hkv, d, T, n_ctas))
        return TREE_ATTN_ERR_WORKSPACE;
    VerifyArgs a = {};
    a.q = q;
    a.k_pages = k_pages;
    a.v_pages = v_pages;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.ws = static_cast<float*>(workspace);
    a.status = status;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.T = T;
    a.P = page_size;
    a.max_pages = max_pages_per_seq;
    a.num_pages = num_pages;
    a.n_ctas = n_ctas;
    a.ovh = ovh_for(Hq, Hkv, T);
    a.scale_log2 = to_log2(softmax_scale);
    a.wait_ns = g_wait_ns.load();
    a.early = g_early.load();
    return prefix_impl(a, k_pages, v_pages, static_cast<cudaStream_t>(stream));
}

int tree_attn_suffix_merge(const uint16_t* q, const int32_t* seq_lens, int max_pages_per_seq,
                           const uint16_t* tree_k, const uint16_t* tree_v, const uint64_t* mask,
                           uint16_t* out, float* lse, int B, int Hq, int Hkv, int d, int T,
                           int page_size, float softmax_scale, const void* workspace,
                           size_t workspace_bytes, int n_ctas, void* stream) {
    int rc = check_common(B, Hq, Hkv, d, T, page_size, max_pages_per_seq, softmax_scale);
    if (rc != TREE_ATTN_OK) return rc;
    if (B == 0) return TREE_ATTN_OK;
    if (!q || !seq_lens || !tree_k || !tree_v || !mask || !out || !lse) return TREE_ATTN_ERR_NULL;
    if (!aligned(q, 16) || !aligned(tree_k, 16) || !aligned(tree_v, 16) || !aligned(out, 16) ||
        !aligned(seq_lens, 4) || !aligned(lse, 4) || !aligned(mask, 8))
        return TREE_ATTN_ERR_ALIGN;
    n_ctas = resolve_ctas(n_ctas, B, Hq, Hkv, T, page_size, max_pages_per_seq);
    if (n_ctas <= 0) return TREE_ATTN_ERR_CUDA;
    if (workspace == nullptr || !aligned(workspace, 256) ||
        workspace_bytes < ws_bytes(B, Hq, Hkv, d, T, n_ctas))
        return TREE_ATTN_ERR_WORKSPACE;
    VerifyArgs a = {};
    a.q = q;
    a.seq_lens = seq_lens;
    a.tree_k = tree_k;
    a.tree_v = tree_v;
    a.mask = mask;
    a.out = out;
    a.lse = lse;
    a.ws = static_cast<float*>(const_cast<void*>(workspace));
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.T = T;
    a.P = page_size;
    a.max_pages = max_pages_per_seq;
    a.n_ctas = n_ctas;
    a.ovh = ovh_for(Hq, Hkv, T);
    a.scale_log2 = to_log2(softmax_scale);
    return launch_merge(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? TREE_ATTN_OK
                                                                           : TREE_ATTN_ERR_CUDA;
}

}  // extern "C"

namespace {

// Shared body of the verify entry points.  mask_stride: 0 (one tree) or T
// (tree b at mask[b * T]); tree_in_cache: tree K/V live in the paged cache at
// positions seq_lens[b] .. seq_lens[b] + T - 1 (tree_k / tree_v unused).
int verify_common(const uint16_t* q, const uint16_t* k_pages, const uint16_t* v_pages,
                  const int32_t* block_table, int max_pages_per_seq, const int32_t* seq_lens,
                  const uint16_t* tree_k, const uint16_t* tree_v, const uint64_t* mask,
                  int mask_stride, bool tree_in_cache, uint16_t* out, float* lse, int B, int Hq,
                  int Hkv, int d, int T, int page_size, int num_pages, float softmax_scale,
                  void* workspace, size_t workspace_bytes, int32_t* status, void* stream,
                  int n_ctas, const uint8_t* dense = nullptr, int dense_cols = 0,
                  const int32_t* parents = nullptr, int parents_stride = 0,
                  uint64_t* mask_out = nullptr) {
    if (mask_stride != 0 && mask_stride != T) return TREE_ATTN_ERR_SHAPE;
    if (tree_in_cache) {
        tree_k = k_pages;  // unused: keep the null checks below meaningful
        tree_v = v_pages;
    }
    if (parents != nullptr) {
        // Masks built inside the merge kernel from the parent arrays.
        if (parents_stride != 0 && parents_stride != T) return TREE_ATTN_ERR_SHAPE;
        if (!aligned(parents, 4) || !aligned(mask_out, 8)) return TREE_ATTN_ERR_ALIGN;
        mask = reinterpret_cast<const uint64_t*>(parents);  // non-null for the checks below
    }
    if (dense != nullptr) {
        // One pass under the explicit mask: no tree mask, no suffix.
        if (dense_cols < 16 || dense_cols % 16 != 0) return TREE_ATTN_ERR_SHAPE;
        if (!aligned(dense, 16)) return TREE_ATTN_ERR_ALIGN;
        mask = reinterpret_cast<const uint64_t*>(dense);  // non-null for the checks below
    }
    int rc = check_common(B, Hq, Hkv, d, T, page_size, max_pages_per_seq, softmax_scale);
    if (rc != TREE_ATTN_OK) return rc;
    if (num_pages < 1 || static_cast<long long>(num_pages) * Hkv * page_size >= (1LL << 31))
        return TREE_ATTN_ERR_SHAPE;
    if (B == 0) return TREE_ATTN_OK;
    if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !tree_k || !tree_v || !mask ||
        !out || !lse)
        return TREE_ATTN_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(tree_k, 16) ||
        !aligned(tree_v, 16) || !aligned(out, 16) || !aligned(block_table, 4) ||
        !aligned(seq_lens, 4) || !aligned(lse, 4) || !aligned(mask, 8) || !aligned(status, 4))
        return TREE_ATTN_ERR_ALIGN;
    // The tree tokens ride on the prefix pass's work line: one extra chunk
    // per unit from the tree buffers, or the positions after the prefix when
    // they are padded into the cache.  The explicit-mask form has no tree.
    // The kernel selector decides which (see make_plan).
    Plan plan;
    if (!plan_call(n_ctas, B, Hq, Hkv, T, page_size, max_pages_per_seq,
                   dense != nullptr ? kTreeNone : (tree_in_cache ? kTreeInCache : kTreeChunk),
                   plan))
        return TREE_ATTN_ERR_CUDA;
    const int tmode = plan.tmode;
    n_ctas = plan.n_ctas;
    const int ovh = plan.ovh;
    if (workspace == nullptr || !aligned(workspace, 256) ||
        workspace_bytes < ws_bytes(B, Hq, Hkv, d, T, n_ctas))
        return TREE_ATTN_ERR_WORKSPACE;

    VerifyArgs a = {};
    a.tmode = tmode;
    a.ovh = ovh;
    a.wait_ns = g_wait_ns.load();
    a.early = g_early.load();
    a.q = q;
    a.k_pages = k_pages;
    a.v_pages = v_pages;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.tree_k = tree_k;
    a.tree_v = tree_v;
    a.mask = mask;
    a.out = out;
    a.lse = lse;
    a.ws = static_cast<float*>(workspace);
    a.status = status;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.T = T;
    a.P = page_size;
    a.max_pages = max_pages_per_seq;
    a.num_pages = num_pages;
    a.n_ctas = n_ctas;
    a.scale_log2 = to_log2(softmax_scale);
    a.mask_stride = mask_stride;
    a.tree_in_cache = tree_in_cache ? 1 : 0;
    a.dense = dense;
    a.dense_cols = dense_cols;
    if (dense != nullptr) a.mask = nullptr;
    a.parents = parents;
    a.parents_stride = parents_stride;
    a.mask_out = mask_out;
    if (parents != nullptr) a.mask = nullptr;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    rc = prefix_impl(a, k_pages, v_pages, st);
    if (rc != TREE_ATTN_OK) return rc;
    return launch_merge(a, st) == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

int tree_attn_verify_ctas(const uint16_t* q, const uint16_t* k_pages, const uint16_t* v_pages,
                          const int32_t* block_table, int max_pages_per_seq,
                          const int32_t* seq_lens, const uint16_t* tree_k,
                          const uint16_t* tree_v, const uint64_t* mask, uint16_t* out,
                          float* lse, int B, int Hq, int Hkv, int d, int T, int page_size,
                          int num_pages, float softmax_scale, void* workspace,
                          size_t workspace_bytes, int32_t* status, void* stream, int n_ctas) {
    return verify_common(q, k_pages, v_pages, block_table, max_pages_per_seq, seq_lens, tree_k,
                         tree_v, mask, 0, false, out, lse, B, Hq, Hkv, d, T, page_size,
                         num_pages, softmax_scale, workspace, workspace_bytes, status, stream,
                         n_ctas);
}

int tree_attn_verify_batched(const uint16_t* q, const uint16_t* k_pages,
                             const uint16_t* v_pages, const int32_t* block_table,
                             int max_pages_per_seq, const int32_t* seq_lens,
                             const uint16_t* tree_k, const uint16_t* tree_v,
                             const uint64_t* masks, uint16_t* out, float* lse, int B, int Hq,
                             int Hkv, int d, int T, int page_size, int num_pages,
                             float softmax_scale, void* workspace, size_t workspace_bytes,
                             int32_t* status, void* stream) {
    return verify_common(q, k_pages, v_pages, block_table, max_pages_per_seq, seq_lens, tree_k,
                         tree_v, masks, T, false, out, lse, B, Hq, Hkv, d, T, page_size,
                         num_pages, softmax_scale, workspace, workspace_bytes, status, stream, 0);
}

int tree_attn_verify_paged_tree(const uint16_t* q, const uint16_t* k_pages,
                                const uint16_t* v_pages, const int32_t* block_table,
                                int max_pages_per_seq, const int32_t* seq_lens,
                                const uint64_t* mask, int mask_stride, uint16_t* out, float* lse,
                                int B, int Hq, int Hkv, int d, int T, int page_size,
                                int num_pages, float softmax_scale, void* workspace,
                                size_t workspace_bytes, int32_t* status, void* stream) {
    return verify_common(q, k_pages, v_pages, block_table, max_pages_per_seq, seq_lens, nullptr,
                         nullptr, mask, mask_stride, true, out, lse, B, Hq, Hkv, d, T,
                         page_size, num_pages, softmax_scale, workspace, workspace_bytes, status,
                         stream, 0);
}

int tree_attn_verify_tree(const uint16_t* q, const uint16_t* k_pages, const uint16_t* v_pages,
                          const int32_t* block_table, int max_pages_per_seq,
                          const int32_t* seq_lens, const uint16_t* tree_k,
                          const uint16_t* tree_v, const int32_t* parents, int parents_stride,
                          uint64_t* mask_out, uint16_t* out, float* lse, int B, int Hq, int Hkv,
                          int d, int T, int page_size, int num_pages, float softmax_scale,
                          void* workspace, size_t workspace_bytes, int32_t* status,
                          void* stream) {
    if (parents == nullptr) return TREE_ATTN_ERR_NULL;
    return verify_common(q, k_pages, v_pages, block_table, max_pages_per_seq, seq_lens, tree_k,
                         tree_v, nullptr, 0, false, out, lse, B, Hq, Hkv, d, T, page_size,
                         num_pages, softmax_scale, workspace, workspace_bytes, status, stream, 0,
                         nullptr, 0, parents, parents_stride, mask_out);
}

int tree_dense_mask_build(const uint64_t* mask, int mask_stride, const int32_t* seq_lens, int B,
                          int T, int dense_cols, uint8_t* dense_mask, int32_t* key_lens,
                          int32_t* status, void* stream) {
    if (B < 0 || T < 1 || T > TREE_ATTN_MAX_T || (mask_stride != 0 && mask_stride != T) ||
        dense_cols < 16 || dense_cols % 16 != 0 || dense_cols / (256 * 16) >= 65535)
        return TREE_ATTN_ERR_SHAPE;
    if (B == 0) return TREE_ATTN_OK;
    if (!mask || !seq_lens || !dense_mask || !key_lens) return TREE_ATTN_ERR_NULL;
    if (!aligned(mask, 8) || !aligned(seq_lens, 4) || !aligned(dense_mask, 16) ||
        !aligned(key_lens, 4) || !aligned(status, 4))
        return TREE_ATTN_ERR_ALIGN;
    return launch_dense_mask_build(mask, mask_stride, seq_lens, B, T, dense_cols, dense_mask,
                                   key_lens, status, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? TREE_ATTN_OK
               : TREE_ATTN_ERR_CUDA;
}

int tree_attn_verify_dense(const uint16_t* q, const uint16_t* k_pages, const uint16_t* v_pages,
                           const int32_t* block_table, int max_pages_per_seq,
                           const int32_t* key_lens, const uint8_t* dense_mask, int dense_cols,
                           uint16_t* out, float* lse, int B, int Hq, int Hkv, int d, int T,
                           int page_size, int num_pages, float softmax_scale, void* workspace,
                           size_t workspace_bytes, int32_t* status, void* stream) {
    if (dense_mask == nullptr) return TREE_ATTN_ERR_NULL;
    return verify_common(q, k_pages, v_pages, block_table, max_pages_per_seq, key_lens, nullptr,
                         nullptr, nullptr, 0, true, out, lse, B, Hq, Hkv, d, T, page_size,
                         num_pages, softmax_scale, workspace, workspace_bytes, status, stream, 0,
                         dense_mask, dense_cols);
}

int tree_attn_verify(const uint16_t* q, const uint16_t* k_pages, const uint16_t* v_pages,
                     const int32_t* block_table, int max_pages_per_seq, const int32_t* seq_lens,
                     const uint16_t* tree_k, const uint16_t* tree_v, const uint64_t* mask,
                     uint16_t* out, float* lse, int B, int Hq, int Hkv, int d, int T,
                     int page_size, int num_pages, float softmax_scale, void* workspace,
                     size_t workspace_bytes, int32_t* status, void* stream) {
    return tree_attn_verify_ctas(q, k_pages, v_pages, block_table, max_pages_per_seq, seq_lens,
                                 tree_k, tree_v, mask, out, lse, B, Hq, Hkv, d, T, page_size,
                                 num_pages, softmax_scale, workspace, workspace_bytes, status,
                                 stream, 0);
}

}  // extern "C"
