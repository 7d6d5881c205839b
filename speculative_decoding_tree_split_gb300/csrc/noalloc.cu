// noalloc.cu -- tree_attn_verify_noalloc: tree_attn_verify for callers that
// may not allocate device memory (fixed-budget memory pools, engines that
// forbid allocation after start-up).  The prefix pass's partial results go
// to a scratch array compiled into the library instead of a caller workspace.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/tree_attn.h"

// The scratch array: TREE_ATTN_NOALLOC_SCRATCH_BYTES on every GPU that loads
// the library, held until the process exits.  In host code this name is only
// a stand-in for the symbol, never a device address: the address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TREE_ATTN_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
// Unique id of the CUDA context the cached address belongs to (0: unknown).
// A device reset destroys the context and with it the array's address; the
// next context gets a new id, so the address is then looked up again.
unsigned long long g_scratch_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Id of the calling thread's current context, or 0 when it cannot be had.
unsigned long long current_ctx_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    if (get_current == nullptr || get_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the scratch array on the current device.  Looked up on
// the first call with a device current, and again only when that device's
// context has changed since (after a cudaDeviceReset); neither call may be
// inside a stream capture.
cudaError_t scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const unsigned long long ctx = current_ctx_id();
    std::lock_guard<std::mutex> lock(g_mu);
    const bool stale = ctx != 0 && g_scratch_ctx[dev] != 0 && ctx != g_scratch_ctx[dev];
    if (g_scratch_ptr[dev] == nullptr || stale) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
        // the lookup made the runtime's context current if it was not yet
        g_scratch_ctx[dev] = ctx != 0 ? ctx : current_ctx_id();
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int tree_attn_verify_noalloc(const uint16_t* q, const uint16_t* k_pages,
                                        const uint16_t* v_pages, const int32_t* block_table,
                                        int max_pages_per_seq, const int32_t* seq_lens,
                                        const uint16_t* tree_k, const uint16_t* tree_v,
                                        const uint64_t* mask, uint16_t* out, float* lse, int B,
                                        int Hq, int Hkv, int d, int T, int page_size,
                                        int num_pages, float softmax_scale, int32_t* status,
                                        void* stream) {
    const size_t need = tree_attn_workspace_size(B, Hq, Hkv, d, T, 0, page_size);
    if (B > 0 && need > TREE_ATTN_NOALLOC_SCRATCH_BYTES) return TREE_ATTN_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    if (B > 0 && need > 0) {
        if (scratch_for_current_device(&scratch) != cudaSuccess) return TREE_ATTN_ERR_CUDA;
    }
    // Same kernels as tree_attn_verify; only the workspace is the built-in array.
    return tree_attn_verify_ctas(q, k_pages, v_pages, block_table, max_pages_per_seq, seq_lens,
                                 tree_k, tree_v, mask, out, lse, B, Hq, Hkv, d, T, page_size,
                                 num_pages, softmax_scale, scratch,
                                 TREE_ATTN_NOALLOC_SCRATCH_BYTES, status, stream, 0);
}
