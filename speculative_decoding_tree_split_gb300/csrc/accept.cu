// accept.cu -- the step after verification: greedy acceptance of the draft
// tree and the commit of the accepted path's K/V into the paged cache.
//
// "Efficient Speculative Decoding for Llama at Scale" (fdeinterviews.com
// summary, opening paragraph): the target verifies the drafted candidates
// and the service commits one accepted path; drafting and verification are
// greedy (mlsanity.com referee report on arXiv 2508.08192, Summary).  After a
// branch is rejected the target cache must hold the committed history only
// (the same summary, paragraph on hidden correctness obligations; the
// report's minor comment on Section 3.3, KV bookkeeping).
//
// Both kernels are latency-bound (a few KB per sequence); they take part in
// programmatic dependent launch so that they overlap the previous kernel's
// tail.  Each lets the next kernel start only after its own wait for the
// kernel before, so no successor runs beside a kernel older than this one.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/tree_attn.h"
#include "layout.h"
#include "ptx.cuh"

namespace treeattn {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kAcceptWarps = 4;
constexpr int kCommitThreads = 128;
// 16-byte vectors one thread moves per tensor: 64 rows x 16 vectors (d = 128)
// over 128 threads.
constexpr int kCommitVecs = TREE_ATTN_MAX_T * 16 / kCommitThreads;

__device__ __forceinline__ void report(int32_t* status, int code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// Greedy acceptance, one warp per sequence; lane l owns nodes l and l + 32.
//
// With the ancestor-or-self masks at hand, node i is accepted exactly when
// every node on its root path passes its own edge test (a root passes; a
// child passes when its token equals the target's token at its parent), so
// acceptance is one ballot and one AND per node.  The parent of i is the
// highest ancestor bit below i: ancestors carry smaller indices and lie on
// one chain, so the deepest of them has the largest index.  The committed
// path is the deepest accepted node's mask; a tie on depth goes to the lower
// index (the reduction key puts 255 - i under the depth).
// ---------------------------------------------------------------------------
struct Accepted {
    int best;     // last node of the committed path, -1 if none
    int n;        // nodes on the path
    uint64_t mb;  // the path's nodes (the mask of `best`)
};

// One warp: the committed path of one sequence (m, dr, tg: its mask row,
// draft and target tokens).
__device__ __forceinline__ Accepted warp_greedy_accept(const uint64_t* m, const int32_t* dr,
                                                       const int32_t* tg, int T, int lane) {
    const uint64_t live = T >= 64 ? ~0ull : (1ull << T) - 1ull;
    uint64_t mi[2];
    bool ok[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        mi[h] = 0;
        ok[h] = false;
        if (i < T) {
            mi[h] = m[i] & live;
            const uint64_t anc = mi[h] & ~(1ull << i);
            if (anc == 0) {
                ok[h] = true;
            } else {
                const int p = 63 - __clzll(static_cast<long long>(anc));
                ok[h] = dr[i] == tg[p];
            }
        }
    }
    const uint64_t okbits = static_cast<uint64_t>(__ballot_sync(kFull, ok[0])) |
                            (static_cast<uint64_t>(__ballot_sync(kFull, ok[1])) << 32);
    unsigned key = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        if (i < T && (mi[h] & ~okbits) == 0) {
            const unsigned k = (static_cast<unsigned>(__popcll(mi[h])) << 8) | (255u - i);
            key = key > k ? key : k;
        }
    }
    key = __reduce_max_sync(kFull, key);
    Accepted r;
    r.best = key != 0 ? 255 - static_cast<int>(key & 255u) : -1;
    const int src_lane = r.best >= 0 ? (r.best & 31) : 0;
    const uint64_t lo = __shfl_sync(kFull, mi[0], src_lane);
    const uint64_t hi = __shfl_sync(kFull, mi[1], src_lane);
    r.mb = r.best < 0 ? 0ull : (r.best < 32 ? lo : hi);
    r.n = __popcll(r.mb);
    return r;
}

// The path's nodes root first, then -1 (one warp).
__device__ __forceinline__ void write_path(int32_t* path, const Accepted& acc, int T, int lane) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        if (i < T) {
            if ((acc.mb >> i) & 1ull) path[__popcll(acc.mb & ((1ull << i) - 1ull))] = i;
            if (i >= acc.n) path[i] = -1;
        }
    }
}

__global__ void __launch_bounds__(32 * kAcceptWarps)
    greedy_accept_kernel(const uint64_t* __restrict__ mask, int mask_stride,
                         const int32_t* __restrict__ draft, const int32_t* __restrict__ target,
                         int B, int T, int32_t* __restrict__ accept_len,
                         int32_t* __restrict__ accept_path, int32_t* __restrict__ bonus) {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kAcceptWarps + (threadIdx.x >> 5);
    if (b >= B) return;
    const int32_t* tg = target + static_cast<size_t>(b) * T;
    const Accepted acc = warp_greedy_accept(mask + static_cast<size_t>(b) * mask_stride,
                                            draft + static_cast<size_t>(b) * T, tg, T, lane);
    write_path(accept_path + static_cast<size_t>(b) * T, acc, T, lane);
    if (lane == 0) {
        accept_len[b] = acc.n;
        bonus[b] = acc.best >= 0 ? tg[acc.best] : -1;
    }
}

// ---------------------------------------------------------------------------
// KV commit: CTA (b, hk) copies the accepted path's K/V rows of KV head hk to
// logical positions L_b + k, k < n_b.  Every row is loaded before any is
// stored, so compacting tree tokens that already sit in the cache (at
// L_b + j) is safe in place; different CTAs touch disjoint (page, head)
// rows.
// ---------------------------------------------------------------------------
struct CommitArgs {
    uint16_t* k_pages;
    uint16_t* v_pages;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const uint16_t* tree_k;  // null: tree tokens live in the cache at L_b + j
    const uint16_t* tree_v;
    const int32_t* accept_path;
    const int32_t* accept_len;
    int32_t* seq_lens_out;
    int32_t* status;
    int Hkv, d, T, P, max_pages, num_pages;
};

// Element offset of (logical position pos, head hk, vector c) of sequence b,
// or -1 (with the status set) when the position has no valid page.
__device__ __forceinline__ long long cache_offset(const CommitArgs& a, int b, int hk, int pos,
                                                  int c) {
    const int slot = pos / a.P;
    if (slot >= a.max_pages) {
        report(a.status, TREE_ATTN_STATUS_BAD_SEQ_LEN);
        return -1;
    }
    const int page = a.block_table[static_cast<size_t>(b) * a.max_pages + slot];
    if (page < 0 || page >= a.num_pages) {
        report(a.status, TREE_ATTN_STATUS_BAD_PAGE);
        return -1;
    }
    return ((static_cast<long long>(page) * a.Hkv + hk) * a.P + pos % a.P) * a.d + c * 8;
}

// CTA (b, hk) of the commit: path node k (path[k], k < n) to position L_b + k.
__device__ __forceinline__ void commit_rows(const CommitArgs& a, int b, int hk, int n,
                                            const int32_t* path) {
    const int tid = threadIdx.x;
    if (n < 0 || n > a.T) {
        if (tid == 0 && hk == 0) report(a.status, TREE_ATTN_STATUS_BAD_PATH);
        n = 0;
    }
    bool bad_len;
    const int32_t L_in = a.seq_lens[b];
    const int L = clamp_seq_len(L_in, a.P, a.max_pages, bad_len);
    if (bad_len) {
        if (tid == 0 && hk == 0) report(a.status, TREE_ATTN_STATUS_BAD_SEQ_LEN);
        n = 0;
    }
    const int vpr = a.d / 8;
    const int nvec = n * vpr;

    uint4 kr[kCommitVecs], vr[kCommitVecs];
    bool have[kCommitVecs];
#pragma unroll
    for (int it = 0; it < kCommitVecs; ++it) {
        const int v = tid + it * kCommitThreads;
        have[it] = false;
        if (v >= nvec) continue;
        const int k = v / vpr, c = v % vpr;
        const int j = path[k];
        if (j < 0 || j >= a.T) {
            report(a.status, TREE_ATTN_STATUS_BAD_PATH);
            continue;
        }
        long long off;
        const uint16_t *sk, *sv;
        if (a.tree_k != nullptr) {
            off = ((static_cast<long long>(b) * a.T + j) * a.Hkv + hk) * a.d + c * 8;
            sk = a.tree_k;
            sv = a.tree_v;
        } else {
            off = cache_offset(a, b, hk, L + j, c);
            sk = a.k_pages;
            sv = a.v_pages;
        }
        if (off < 0) continue;
        kr[it] = *reinterpret_cast<const uint4*>(sk + off);
        vr[it] = *reinterpret_cast<const uint4*>(sv + off);
        have[it] = true;
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < kCommitVecs; ++it) {
        if (!have[it]) continue;
        const int v = tid + it * kCommitThreads;
        const int k = v / vpr, c = v % vpr;
        const long long off = cache_offset(a, b, hk, L + k, c);
        if (off < 0) continue;
        *reinterpret_cast<uint4*>(a.k_pages + off) = kr[it];
        *reinterpret_cast<uint4*>(a.v_pages + off) = vr[it];
    }
    if (hk == 0 && tid == 0 && a.seq_lens_out != nullptr)
        a.seq_lens_out[b] = bad_len ? L_in : L + n;
}

__global__ void __launch_bounds__(kCommitThreads) kv_commit_kernel(CommitArgs a) {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    const int b = blockIdx.x;
    commit_rows(a, b, blockIdx.y, a.accept_len[b], a.accept_path + static_cast<size_t>(b) * a.T);
}

// Acceptance and commit in one launch: warp 0 of every CTA (b, hk) finds
// sequence b's path (a few hundred cycles, so each CTA repeats it rather
// than waiting for another kernel); CTA (b, 0) writes the acceptance out.
struct AcceptArgs {
    const uint64_t* mask;
    int mask_stride;
    const int32_t* draft;
    const int32_t* target;
    int32_t* accept_len;   // nullable
    int32_t* accept_path;  // nullable
    int32_t* bonus;        // nullable
};

__global__ void __launch_bounds__(kCommitThreads)
    accept_commit_kernel(CommitArgs a, AcceptArgs g) {
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    __shared__ int32_t path[TREE_ATTN_MAX_T];
    __shared__ int n_s;
    const int b = blockIdx.x, hk = blockIdx.y;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int32_t* tg = g.target + static_cast<size_t>(b) * a.T;
        const Accepted acc =
            warp_greedy_accept(g.mask + static_cast<size_t>(b) * g.mask_stride,
                               g.draft + static_cast<size_t>(b) * a.T, tg, a.T, lane);
        write_path(path, acc, a.T, lane);
        if (lane == 0) n_s = acc.n;
        if (hk == 0) {
            if (g.accept_path != nullptr)
                write_path(g.accept_path + static_cast<size_t>(b) * a.T, acc, a.T, lane);
            if (lane == 0 && g.accept_len != nullptr) g.accept_len[b] = acc.n;
            if (lane == 0 && g.bonus != nullptr) g.bonus[b] = acc.best >= 0 ? tg[acc.best] : -1;
        }
    }
    __syncthreads();
    commit_rows(a, b, hk, n_s, path);
}

template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace treeattn

using namespace treeattn;

extern "C" {

int tree_greedy_accept(const uint64_t* mask, int mask_stride, const int32_t* draft_tokens,
                       const int32_t* target_tokens, int B, int T, int32_t* accept_len,
                       int32_t* accept_path, int32_t* bonus_token, void* stream) {
    if (B < 0 || T < 1 || T > TREE_ATTN_MAX_T || (mask_stride != 0 && mask_stride != T))
        return TREE_ATTN_ERR_SHAPE;
    if (B == 0) return TREE_ATTN_OK;
    if (!mask || !draft_tokens || !target_tokens || !accept_len || !accept_path || !bonus_token)
        return TREE_ATTN_ERR_NULL;
    if (!aligned(mask, 8) || !aligned(draft_tokens, 4) || !aligned(target_tokens, 4) ||
        !aligned(accept_len, 4) || !aligned(accept_path, 4) || !aligned(bonus_token, 4))
        return TREE_ATTN_ERR_ALIGN;
    const dim3 grid((B + kAcceptWarps - 1) / kAcceptWarps);
    const cudaError_t e =
        launch_pdl(greedy_accept_kernel, grid, dim3(32 * kAcceptWarps),
                   static_cast<cudaStream_t>(stream), mask, mask_stride, draft_tokens,
                   target_tokens, B, T, accept_len, accept_path, bonus_token);
    return e == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
}

int tree_kv_commit(uint16_t* k_pages, uint16_t* v_pages, const int32_t* block_table,
                   int max_pages_per_seq, const int32_t* seq_lens, const uint16_t* tree_k,
                   const uint16_t* tree_v, const int32_t* accept_path, const int32_t* accept_len,
                   int32_t* seq_lens_out, int B, int Hkv, int d, int T, int page_size,
                   int num_pages, int32_t* status, void* stream) {
    if (B < 0 || Hkv < 1 || Hkv > 65535 || (d != 64 && d != 128) || T < 1 ||
        T > TREE_ATTN_MAX_T || max_pages_per_seq < 1 || num_pages < 1 ||
        (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128))
        return TREE_ATTN_ERR_SHAPE;
    if (static_cast<long long>(num_pages) * Hkv * page_size * d >= (1LL << 62))
        return TREE_ATTN_ERR_SHAPE;
    if (seq_lens_out != nullptr && seq_lens_out == seq_lens) return TREE_ATTN_ERR_SHAPE;
    if (B == 0) return TREE_ATTN_OK;
    if (!k_pages || !v_pages || !block_table || !seq_lens || !accept_path || !accept_len ||
        ((tree_k == nullptr) != (tree_v == nullptr)))
        return TREE_ATTN_ERR_NULL;
    if (!aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(tree_k, 16) ||
        !aligned(tree_v, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
        !aligned(accept_path, 4) || !aligned(accept_len, 4) || !aligned(seq_lens_out, 4) ||
        !aligned(status, 4))
        return TREE_ATTN_ERR_ALIGN;
    CommitArgs a;
    a.k_pages = k_pages;
    a.v_pages = v_pages;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.tree_k = tree_k;
    a.tree_v = tree_v;
    a.accept_path = accept_path;
    a.accept_len = accept_len;
    a.seq_lens_out = seq_lens_out;
    a.status = status;
    a.Hkv = Hkv;
    a.d = d;
    a.T = T;
    a.P = page_size;
    a.max_pages = max_pages_per_seq;
    a.num_pages = num_pages;
    const cudaError_t e = launch_pdl(kv_commit_kernel, dim3(B, Hkv), dim3(kCommitThreads),
                                     static_cast<cudaStream_t>(stream), a);
    return e == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
}

int tree_accept_commit(const uint64_t* mask, int mask_stride, const int32_t* draft_tokens,
                       const int32_t* target_tokens, uint16_t* k_pages, uint16_t* v_pages,
                       const int32_t* block_table, int max_pages_per_seq, const int32_t* seq_lens,
                       const uint16_t* tree_k, const uint16_t* tree_v, int32_t* accept_len,
                       int32_t* accept_path, int32_t* bonus_token, int32_t* seq_lens_out, int B,
                       int Hkv, int d, int T, int page_size, int num_pages, int32_t* status,
                       void* stream) {
    if (B < 0 || Hkv < 1 || Hkv > 65535 || (d != 64 && d != 128) || T < 1 ||
        T > TREE_ATTN_MAX_T || max_pages_per_seq < 1 || num_pages < 1 ||
        (mask_stride != 0 && mask_stride != T) ||
        (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128))
        return TREE_ATTN_ERR_SHAPE;
    if (seq_lens_out != nullptr && seq_lens_out == seq_lens) return TREE_ATTN_ERR_SHAPE;
    if (B == 0) return TREE_ATTN_OK;
    if (!mask || !draft_tokens || !target_tokens || !k_pages || !v_pages || !block_table ||
        !seq_lens || ((tree_k == nullptr) != (tree_v == nullptr)))
        return TREE_ATTN_ERR_NULL;
    if (!aligned(mask, 8) || !aligned(draft_tokens, 4) || !aligned(target_tokens, 4) ||
        !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(tree_k, 16) ||
        !aligned(tree_v, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
        !aligned(accept_len, 4) || !aligned(accept_path, 4) || !aligned(bonus_token, 4) ||
        !aligned(seq_lens_out, 4) || !aligned(status, 4))
        return TREE_ATTN_ERR_ALIGN;
    CommitArgs a;
    a.k_pages = k_pages;
    a.v_pages = v_pages;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.tree_k = tree_k;
    a.tree_v = tree_v;
    a.accept_path = nullptr;
    a.accept_len = nullptr;
    a.seq_lens_out = seq_lens_out;
    a.status = status;
    a.Hkv = Hkv;
    a.d = d;
    a.T = T;
    a.P = page_size;
    a.max_pages = max_pages_per_seq;
    a.num_pages = num_pages;
    AcceptArgs g;
    g.mask = mask;
    g.mask_stride = mask_stride;
    g.draft = draft_tokens;
    g.target = target_tokens;
    g.accept_len = accept_len;
    g.accept_path = accept_path;
    g.bonus = bonus_token;
    const cudaError_t e = launch_pdl(accept_commit_kernel, dim3(B, Hkv), dim3(kCommitThreads),
                                     static_cast<cudaStream_t>(stream), a, g);
    return e == cudaSuccess ? TREE_ATTN_OK : TREE_ATTN_ERR_CUDA;
}

}  // extern "C"
