// kernels.cu -- sm_103a device code of split tree attention.
//
//   tree_mask_kernel     ancestor bitmask per tree node (pointer jumping).
//   prefix_pass_kernel   persistent, warp-specialised flash-decoding prefix
//                        pass over the paged KV cache: TMA -> shared memory
//                        ring, S = Q.K^T and O += P.V on tcgen05 tensor cores
//                        with fp32 accumulators in TMEM, online softmax in
//                        registers; writes one (m, l, acc) partial per
//                        segment of its share of the work line.
//   suffix_merge_kernel  tree-masked suffix pass (T <= 64 keys, SIMT) and
//                        log-sum-exp merge of every partial into out / lse.
//
// Method: split tree attention ("Efficient Speculative Decoding for Llama at
// Scale", pith.science review, "What carries the argument"): prefix attention
// needs no mask, tree attention needs the tree mask, and merge_attentions
// joins the two (verdict record, supporting_citations: attention over
// disjoint KV chunks, Hydragen).  The prefix pass is split over the KV length
// as in flash-decoding (Dao, Haziza, Massa, Sizov; review reference list).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/tree_attn.h"
#include "kernels.cuh"
#include "layout.h"
#include "ptx.cuh"

namespace treeattn {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ void report(int32_t* status, int code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

// ===========================================================================
// Tree mask: node i sees itself and its ancestors.  One warp; lane l owns
// nodes l and l + 32.  Pointer jumping: after round k, anc[i] holds every
// node at distance < 2^k above i and jump[i] is the 2^k-th ancestor.  Six
// rounds cover any depth <= 64.
// ===========================================================================
__device__ __forceinline__ uint64_t pick64(uint64_t lo, uint64_t hi, int node) {
    const uint64_t a = __shfl_sync(kFull, lo, node & 31);
    const uint64_t b = __shfl_sync(kFull, hi, node & 31);
    return node < 32 ? a : b;
}

__device__ __forceinline__ int pick32(int lo, int hi, int node) {
    const int a = __shfl_sync(kFull, lo, node & 31);
    const int b = __shfl_sync(kFull, hi, node & 31);
    return node < 32 ? a : b;
}

// Ancestor-or-self masks of one tree (T <= 64 nodes, parents[i] in [-1, i)),
// computed by one warp: lane l returns the masks of nodes l and l + 32.
// Returns true if a parent was invalid (that node is then taken as a root).
__device__ __forceinline__ bool warp_tree_mask(const int32_t* parents, int T, int lane,
                                               uint64_t anc[2]) {
    int jump[2];
    bool bad = false;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        int p = -1;
        if (i < T) {
            p = parents[i];
            if (p < -1 || p >= i) {
                bad = true;
                p = -1;  // treat as a root so the rest stays well defined
            }
        }
        jump[h] = p;
        anc[h] = (i < T) ? (1ull << i) : 0ull;
    }
#pragma unroll
    for (int round = 0; round < 6; ++round) {
        uint64_t na[2];
        int nj[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = jump[h] < 0 ? 0 : jump[h];
            const uint64_t aj = pick64(anc[0], anc[1], j);
            const int jj = pick32(jump[0], jump[1], j);
            na[h] = jump[h] < 0 ? anc[h] : (anc[h] | aj);
            nj[h] = jump[h] < 0 ? -1 : jj;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            anc[h] = na[h];
            jump[h] = nj[h];
        }
    }
    return __any_sync(kFull, bad);
}

#ifndef TREE_ATTN_EARLY_TU
__global__ void __launch_bounds__(32) tree_mask_kernel(const int32_t* __restrict__ parents, int T,
                                                       uint64_t* __restrict__ mask,
                                                       int32_t* status) {
    // CTA b builds the mask of tree b (a batch of trees is [B][T]).
    parents += static_cast<size_t>(blockIdx.x) * T;
    mask += static_cast<size_t>(blockIdx.x) * T;
    // Wait for the kernel before; only then may the next kernel start (it
    // waits for this grid before reading anything this grid writes), so no
    // successor ever runs beside a kernel older than this one.
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    const int lane = threadIdx.x;
    uint64_t anc[2];
    if (warp_tree_mask(parents, T, lane, anc) && lane == 0)
        report(status, TREE_ATTN_STATUS_BAD_PARENT);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        if (i < T) mask[i] = anc[h];
    }
}
#endif  // !TREE_ATTN_EARLY_TU

// ===========================================================================
// Prefix pass
//
// Keys are processed in blocks of up to 128 (two 64-token steps of the work
// line).  Every tcgen05.mma instruction costs about the same issue time
// whatever its N, so S = Q.K^T uses N = 128 keys per instruction and P is
// kept in TMEM as the A operand of O += P.V; per 128 keys the tensor pipe
// sees 2*d/16 instructions.
// ===========================================================================
constexpr int kBlock = 2 * kChunk;  // keys per MMA block
// Block tables of at most this many entries (B * max_pages) are staged in
// shared memory by the plan, in the same round trip as the sequence lengths.
constexpr int kSmallBt = 128;
// Threads of a prefix-pass CTA: the four softmax warps, the copy warp, the
// MMA warp and a seventh warp that has no role and waits at the final
// barrier.  Measured on GB300 against the same kernel with six warps: the
// one-row-copy (Maverick-shaped) pass 92.5 -> 91.0 us, the Llama-3.1-70B
// pass 57.2 -> 57.0 us, the others unchanged; compiling for 224 threads
// but launching 192 gave nothing, so the gain comes from the extra warp's
// presence, by a mechanism these measurements do not identify.
constexpr int kPrefixThreads = 224;
// Early start: K/V blocks a CTA loads before its dependency wait.  The plan
// and the first block's page lookups always go first; each block loaded
// early also takes memory bandwidth from the tail of the kernel before.
constexpr int kEarlyBlocks = 3;
static_assert(kEarlyBlocks <= 3, "early blocks go to ring stages that need no release");

template <int D>
struct PrefixShape {
    static constexpr int DH = D / 64;                       // 128-byte column blocks of d
    static constexpr int Q_BYTES = kRows * D * 2;           // Q tile, DH atom columns
    static constexpr int QATOM_BYTES = kRows * 128;         // one atom column of Q
    static constexpr int HALF_BYTES = kBlock * 128;         // 128 keys x 64 d of K or V
    static constexpr int TILE_BYTES = DH * HALF_BYTES;      // K (or V) of one block
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int NS = (D == 128) ? 3 : 6;           // ring depth
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_STAGE = OFF_Q + Q_BYTES;
    static constexpr int OFF_BAR = OFF_STAGE + NS * STAGE_BYTES;
    // barrier indices
    static constexpr int KV_FULL = 0;
    static constexpr int KV_EMPTY = NS;
    static constexpr int S_FULL = 2 * NS;
    static constexpr int S_FREE = 2 * NS + 2;
    static constexpr int P_FULL = 2 * NS + 4;
    static constexpr int P_FREE = 2 * NS + 6;
    static constexpr int O_FULL = 2 * NS + 8;
    static constexpr int O_FREE = 2 * NS + 9;
    static constexpr int Q_FULL = 2 * NS + 10;
    static constexpr int DRAIN = 2 * NS + 11;
    static constexpr int FOLD = 2 * NS + 12;  // softmax warps meet before the fold
    static constexpr int NBAR = 2 * NS + 13;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int OFF_SBT = OFF_MISC + 64;  // a small block table (kSmallBt entries)
    static constexpr int SMEM_BYTES = OFF_SBT + kSmallBt * 4 + 1024;  // + alignment slack
    // TMEM columns: O at [0, D); S[2] (fp32, 128 keys each) after it; P[2]
    // (bf16 pairs, 64 columns each) after S.
    static constexpr int TM_O = 0;
    static constexpr int TM_S = D;
    static constexpr int TM_P = D + 2 * kBlock;
    static constexpr int TMEM_COLS = 512;
    static_assert(TM_P + 2 * (kBlock / 2) <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(SMEM_BYTES > 114 * 1024, "one CTA per SM keeps TMEM allocation uncontended");
    static_assert(kRows * (D + 4 + 2) * 4 <= NS * STAGE_BYTES,
                  "the last segment's epilogue stages every row copy in the K/V ring");
};

struct PrefixMisc {
    uint32_t tmem_base;
    int abort;
};

// This CTA's share of the work line: total length W, its range [x0, x1), the
// sequence b0 holding x0, that sequence's base position and seq_lens[b0].
struct CtaPlan {
    long long W, x0, x1, base0;
    int b0;
    int32_t lraw0;
};
static_assert(sizeof(PrefixMisc) <= 64, "PrefixMisc fits its shared-memory slot");

struct PrefixArgs {
    const int32_t* block_table;
    const int32_t* seq_lens;
    const uint16_t* q;
    float* ws;
    int32_t* status;
    int B, Hq, Hkv, G, T, M, RB, P, max_pages, num_pages, n_ctas;
    float scale_log2;
    // One-pass form under an explicit mask (DENSE kernels only): key p of
    // query token t of sequence b is visible when dense[(b*T + t)*dense_cols + p]
    // is non-zero; seq_lens then counts every key in the cache, tree included.
    const uint8_t* dense;
    int dense_cols;
    // Tree tokens on the work line (TreeMode; kTreeNone for DENSE kernels):
    // their mask bits come from `mask` ([T] or [B][T] by mask_stride) or are
    // built from `parents` (stride 0 or T), and are then also written to
    // mask_out when it is not null.
    int tmode;
    const uint64_t* mask;
    int mask_stride;
    const int32_t* parents;
    int parents_stride;
    uint64_t* mask_out;
    int ovh;  // overhead slots per unit on the work line
    // Limit of every wait on another role of the CTA (ns of %globaltimer);
    // past it the kernel reports TREE_ATTN_STATUS_TIMEOUT and winds down.
    unsigned long long wait_ns;
};

// Kernel variants of the prefix pass: the tree modes of layout.h, plus the
// one-pass form under an explicit byte mask.
constexpr int kModeDense = 3;

__device__ __forceinline__ long long warp_incl_scan(long long v, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long n = __shfl_up_sync(kFull, v, off);
        if (lane >= off) v += n;
    }
    return v;
}

constexpr int kL1Line = 128;  // bytes per L1 cache line

// Sequences whose work-line lengths the plan keeps in registers (32 per
// entry): their seq_lens are read in one round trip, all loads in flight.
constexpr int kPlanRegs = 4;

// Total work W and this CTA's range and starting sequence (one warp, every
// lane gets the result).  Every warp of the CTA computes it for itself, so no
// role waits for a hand-over: the loads of all warps go out together and
// share their L1 lines.  When `sbt` is not null a block table of at most
// kSmallBt entries is also copied there (shared memory), its loads issued
// together with the sequence lengths'.
__device__ CtaPlan compute_plan(const PrefixArgs& a, int lane, int32_t* sbt) {
    const int upb = a.Hkv * a.RB;
    auto len_of = [&](int32_t L_raw, bool report_bad) -> int {
        bool bad;
        const int n = unit_len(unit_chunks(L_raw, a.P, a.max_pages, a.tmode, a.T, bad), a.ovh);
        if (report_bad && bad && blockIdx.x == 0) report(a.status, TREE_ATTN_STATUS_BAD_SEQ_LEN);
        return n;
    };
    // All loads first, so that they are in flight together.
    int32_t lraw[kPlanRegs];
#pragma unroll
    for (int i = 0; i < kPlanRegs; ++i) {
        const int b = 32 * i + lane;
        lraw[i] = b < a.B ? a.seq_lens[b] : 0;
    }
    const int nbt = a.B * a.max_pages;
    if (sbt != nullptr && nbt <= kSmallBt) {
        int32_t e[kSmallBt / 32];
#pragma unroll
        for (int i = 0; i < kSmallBt / 32; ++i)
            e[i] = 32 * i + lane < nbt ? a.block_table[32 * i + lane] : -1;
#pragma unroll
        for (int i = 0; i < kSmallBt / 32; ++i)
            if (32 * i + lane < nbt) sbt[32 * i + lane] = e[i];
    }
    int nreg[kPlanRegs];
#pragma unroll
    for (int i = 0; i < kPlanRegs; ++i) nreg[i] = 32 * i + lane < a.B ? len_of(lraw[i], true) : 0;
    long long tot = 0;
#pragma unroll
    for (int i = 0; i < kPlanRegs; ++i)
        if (32 * i < a.B) tot += __reduce_add_sync(kFull, nreg[i]);
    for (int b0 = 32 * kPlanRegs; b0 < a.B; b0 += 32) {
        const int b = b0 + lane;
        tot += __reduce_add_sync(kFull, b < a.B ? len_of(a.seq_lens[b], true) : 0);
    }
    const long long W = tot * upb;
    const long long x0 = cta_start(blockIdx.x, W, a.n_ctas);
    const long long x1 = cta_start(blockIdx.x + 1, W, a.n_ctas);
    int b_start = 0;
    long long base0 = 0;
    int32_t lraw0 = 0;
    if (x0 < x1) {
        long long run = 0;
        for (int b0 = 0; b0 < a.B; b0 += 32) {
            const int b = b0 + lane;
            int nb = 0;
#pragma unroll
            for (int i = 0; i < kPlanRegs; ++i)
                if (b0 == 32 * i) nb = nreg[i];
            if (b0 >= 32 * kPlanRegs && b < a.B) nb = len_of(a.seq_lens[b], false);
            const long long n = static_cast<long long>(upb) * nb;
            const long long incl = warp_incl_scan(n, lane);
            const long long excl = incl - n;
            const bool hit = (b < a.B) && (run + excl <= x0) && (x0 < run + incl);
            const unsigned m = __ballot_sync(kFull, hit);
            if (m != 0) {
                const int src = __ffs(m) - 1;
                b_start = b0 + src;
                base0 = run + __shfl_sync(kFull, excl, src);
                int32_t lr = 0;
#pragma unroll
                for (int i = 0; i < kPlanRegs; ++i)
                    if (b0 == 32 * i) lr = __shfl_sync(kFull, lraw[i], src);
                lraw0 = b0 >= 32 * kPlanRegs ? a.seq_lens[b_start] : lr;
                break;
            }
            run += __shfl_sync(kFull, incl, 31);
        }
    }
    CtaPlan pl;
    pl.W = W;
    pl.x0 = x0;
    pl.x1 = x1;
    pl.b0 = b_start;
    pl.base0 = base0;
    pl.lraw0 = lraw0;
    return pl;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Blocks of one segment: block i covers work-line steps
// [chunk_begin + 2i, min(chunk_begin + 2i + 2, chunk_end)).
__device__ __forceinline__ int blocks_of(const Segment& sg) {
    return (sg.chunk_end - sg.chunk_begin + 1) / 2;
}

// EARLY: seq_lens, block_table and the committed prefix K/V are not written
// by the kernel before this one in the stream, so the plan and the first ring
// stages' loads of committed-prefix blocks go out before the dependency wait
// (q, the tree K/V and the masks are read after it).  The explicit-mask form
// has no early variant.
template <int D, int F, int MODE, bool EARLY>
__global__ void __launch_bounds__(kPrefixThreads, 1)
    prefix_pass_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_tk,
                       const __grid_constant__ CUtensorMap tm_tv, const PrefixArgs a) {
    using S = PrefixShape<D>;
    constexpr bool DENSE = MODE == kModeDense;
    constexpr int TM = DENSE ? kTreeNone : MODE;  // tree mode of the work line
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t sb = raw_addr + pad;  // 1024-aligned shared address of the layout
    PrefixMisc* misc = reinterpret_cast<PrefixMisc*>(smem + S::OFF_MISC);
    volatile int* abort_flag = &misc->abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) -> uint32_t { return sb + S::OFF_BAR + 8u * i; };

    // ---------------- prologue (overlaps the previous kernel under PDL)
    if (warp == 4 && lane == 0) {
        for (int s = 0; s < S::NS; ++s) {
            ptx::mbar_init(bar(S::KV_FULL + s), 1);
            ptx::mbar_init(bar(S::KV_EMPTY + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(bar(S::S_FULL + i), 1);
            ptx::mbar_init(bar(S::S_FREE + i), 4);
            ptx::mbar_init(bar(S::P_FULL + i), 4);
            ptx::mbar_init(bar(S::P_FREE + i), 1);
        }
        ptx::mbar_init(bar(S::O_FULL), 1);
        ptx::mbar_init(bar(S::O_FREE), 4);
        ptx::mbar_init(bar(S::Q_FULL), 4);
        ptx::mbar_init(bar(S::DRAIN), 1);
        ptx::mbar_init(bar(S::FOLD), 4);
        misc->abort = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
    }
    if (warp == 5) {
        ptx::tmem_alloc(ptx::smem_u32(&misc->tmem_base), S::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    // L2 policy of the K/V loads (reads no input, so it is made before the wait).
    const uint64_t pol = (warp == 4 && lane == 0) ? ptx::policy_evict_first() : 0ull;
    // The barriers and the TMEM base are in place before any role starts.
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const int upb = a.Hkv * a.RB;
    const bool small_bt = static_cast<long long>(a.B) * a.max_pages <= kSmallBt;
    int32_t* sbt = reinterpret_cast<int32_t*>(smem + S::OFF_SBT);

    auto fail = [&]() {
        *abort_flag = 1;
        report(a.status, TREE_ATTN_STATUS_TIMEOUT);
    };

    // Physical pages of block jj -- work-line steps ch and ch + 1 of segment
    // sg: the block-table loads are only issued here (all at once), and used
    // by issue_block, so the caller can wait for the ring in between.
    struct BlockPages {
        int pids[8];
        bool use[8];
    };
    auto block_pages = [&](const Segment& sg, int ch, BlockPages& bp) {
        bool bad;
        const int L = clamp_seq_len(sg.len_raw, a.P, a.max_pages, bad);
        // Pages holding this unit's keys: the prefix, and for kTreeInCache
        // the tree tokens padded after it.
        int npages = (L + a.P - 1) / a.P;
        if (TM == kTreeInCache) npages = min(a.max_pages, (L + a.T + a.P - 1) / a.P);
        const int tree_ch = chunks_of(L);
        const int Pb = a.P < kChunk ? a.P : kChunk;
        const int nsub = kChunk / Pb;
        const int pshift = __ffs(a.P) - 1;
        const size_t row = static_cast<size_t>(sg.b) * a.max_pages;
        const int nh = min(2, sg.chunk_end - ch);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int k = hh * 4 + i;
                const int tok = (ch + hh) * kChunk + i * Pb;
                const int lp = tok >> pshift;
                bp.use[k] = hh < nh && i < nsub && lp < npages &&
                            !(TM == kTreeChunk && ch + hh == tree_ch);
                bp.pids[k] = bp.use[k] ? (small_bt ? sbt[row + lp] : a.block_table[row + lp]) : -1;
            }
        }
    };
    // Whether block (sg, ch) holds committed-prefix keys only, i.e. reads no
    // tree K/V (kTreeChunk: the tree chunk; kTreeInCache: the pages past the
    // prefix, where the tree tokens are written).
    auto committed_block = [&](const Segment& sg, int ch) -> bool {
        bool bad;
        const int L = clamp_seq_len(sg.len_raw, a.P, a.max_pages, bad);
        const int nh = min(2, sg.chunk_end - ch);
        if (TM == kTreeInCache) return static_cast<long long>(ch + nh) * kChunk <= L;
        if (TM == kTreeChunk) return ch + nh <= chunks_of(L);
        return true;
    };
    // Issues the K/V loads of block jj (pages from block_pages) into ring
    // stage jj % NS, which the caller has found free.
    auto issue_block = [&](const Segment& sg, int ch, uint32_t jj, const BlockPages& bp) {
        bool bad;
        const int L = clamp_seq_len(sg.len_raw, a.P, a.max_pages, bad);
        const int tree_ch = chunks_of(L);            // the tree chunk (kTreeChunk)
        const int Pb = a.P < kChunk ? a.P : kChunk;  // rows per TMA box
        const int nh = min(2, sg.chunk_end - ch);    // 64-token steps in this block
        const int s = jj % S::NS;
        int ys[8];
        int rows[8];
        int nl = 0;
        int tree_half = -1;  // half of the block holding the tree chunk
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            if (TM == kTreeChunk && hh < nh && ch + hh == tree_ch) tree_half = hh;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int k = hh * 4 + i;
                if (!bp.use[k]) continue;
                const int pid = bp.pids[k];
                if (pid < 0 || pid >= a.num_pages) {
                    report(a.status, TREE_ATTN_STATUS_BAD_PAGE);
                    continue;
                }
                const int tok = (ch + hh) * kChunk + i * Pb;
                ys[nl] = (pid * a.Hkv + sg.hk) * a.P + (tok & (a.P - 1));
                rows[nl] = hh * kChunk + i * Pb;
                ++nl;
            }
        }
        const uint32_t fb = bar(S::KV_FULL + s);
        // a tree chunk is one 64-row box per 64 columns of K and of V
        const uint32_t bytes =
            static_cast<uint32_t>((nl * Pb + (tree_half >= 0 ? kChunk : 0)) * 128 * S::DH * 2);
        if (bytes != 0) {
            ptx::mbar_arrive_expect_tx(fb, bytes);
        } else {
            ptx::mbar_arrive(fb);
        }
        const uint32_t kst = sb + S::OFF_STAGE + s * S::STAGE_BYTES;
        const uint32_t vst = kst + S::TILE_BYTES;
#pragma unroll 1
        for (int l = 0; l < nl; ++l) {
#pragma unroll
            for (int h = 0; h < S::DH; ++h) {
                ptx::tma_load_2d(kst + h * S::HALF_BYTES + rows[l] * 128, &tm_k, h * 64, ys[l], fb,
                                 pol);
                ptx::tma_load_2d(vst + h * S::HALF_BYTES + rows[l] * 128, &tm_v, h * 64, ys[l], fb,
                                 pol);
            }
        }
        if (TM == kTreeChunk && tree_half >= 0) {
            // Tree tokens 0..63 of (b, hk): rows b*T + j of the [B*T][Hkv][d]
            // buffers (rows past the tree are other sequences' tokens or zero
            // fill; they are masked and their V rows zeroed).
#pragma unroll
            for (int h = 0; h < S::DH; ++h) {
                const uint32_t off = h * S::HALF_BYTES + tree_half * kChunk * 128;
                ptx::tma_load_3d(kst + off, &tm_tk, h * 64, sg.hk, sg.b * a.T, fb, pol);
                ptx::tma_load_3d(vst + off, &tm_tv, h * 64, sg.hk, sg.b * a.T, fb, pol);
            }
        }
    };

    // Inputs may come from the kernel before us in the stream.  Under EARLY
    // the plan's inputs do not, and each role waits where it first reads one
    // that may (the producer before its first block that is not committed
    // prefix or does not fit the ring; the softmax warps before Q).
    constexpr bool early = EARLY && !DENSE;
    if (!early) ptx::grid_dep_wait();
    const CtaPlan pl = compute_plan(a, lane, warp == 4 && small_bt ? sbt : nullptr);
    if (warp == 4 && small_bt) __syncwarp();  // the staged table is visible to lane 0
    if (warp == 4 && !small_bt) {
        // A block table of a few lines is pulled into L1 while the producer
        // starts, so its first page lookups do not each wait for L2.
        const long long lines =
            (static_cast<long long>(a.B) * a.max_pages * 4 + kL1Line - 1) / kL1Line;
        if (lines <= 2 * 32) {
            const char* bt = reinterpret_cast<const char*>(a.block_table);
            if (lane < lines) ptx::prefetch_l1(bt + static_cast<size_t>(lane) * kL1Line);
            if (lane + 32 < lines) ptx::prefetch_l1(bt + static_cast<size_t>(lane + 32) * kL1Line);
        }
    }
    // The next kernel may start once every CTA has passed here; it reads, before
    // its own dependency wait, inputs of the kernel before us (the merge reads
    // q, the tree K/V and the parents), so under EARLY the signal is given
    // only after this CTA has waited for that kernel (softmax warps, below).
    if (!early) ptx::grid_dep_launch();
    const uint32_t tmem = misc->tmem_base;
    auto init_walker = [&](Walker& w) {
        w.init_known(a.seq_lens, a.B, a.P, a.max_pages, upb, a.RB, pl.b0, pl.base0, pl.x0, pl.x1,
                     TM, a.T, a.ovh, pl.lraw0);
    };

    if (warp == 4) {
        // ================= TMA producer (one thread)
        if (lane == 0) {
            Walker w;
            init_walker(w);
            uint32_t jj = 0;
            bool ok = true;
            bool dep_done = !early;  // the dependency wait is behind this thread
            Segment sg;
            while (ok && w.next(sg)) {
#pragma unroll 1
                for (int ch = sg.chunk_begin; ch < sg.chunk_end; ch += 2, ++jj) {
                    // The block's page lookups go out before the wait for its
                    // ring stage, so their round trip overlaps that wait.
                    BlockPages bp;
                    block_pages(sg, ch, bp);
                    if (!dep_done && (jj >= kEarlyBlocks || !committed_block(sg, ch))) {
                        ptx::grid_dep_wait();
                        dep_done = true;
                    }
                    const int s = jj % S::NS;
                    if (jj >= S::NS &&
                        !ptx::mbar_wait(bar(S::KV_EMPTY + s), ((jj / S::NS) - 1) & 1, a.wait_ns)) {
                        fail();
                        ok = false;
                        break;
                    }
                    if (*abort_flag) {
                        ok = false;
                        break;
                    }
                    issue_block(sg, ch, jj, bp);
                }
            }
            if (!ok) {
                // Let every copy still in flight land before the CTA exits
                // (they complete on their own: no other role is waited for).
                const uint32_t first = jj > S::NS ? jj - S::NS : 0;
                for (uint32_t j = first; j < jj; ++j)
                    (void)ptx::mbar_wait(bar(S::KV_FULL + j % S::NS), (j / S::NS) & 1,
                                         ptx::kDrainLimitNs);
            }
        }
    } else if (warp == 5) {
        // ================= MMA issuer (one thread)
        // Issues S = Q.K^T for the next block as soon as its K/V has landed
        // and P.V for the oldest block as soon as its P is ready, whichever
        // comes first, so neither waits behind the other.
        if (lane == 0) {
            Walker w;
            init_walker(w);
            const uint32_t idesc_qk = idesc_bf16_f32(kRows, kBlock, false, false);
            const uint32_t idesc_pv = idesc_bf16_f32(kRows, D, false, true);
            uint32_t jj = 0, kk = 0;  // blocks of earlier segments, segments done
            bool ok = true;
            Segment sg;
            while (ok && w.next(sg)) {
                if (!ptx::mbar_wait(bar(S::Q_FULL), kk & 1, a.wait_ns)) {
                    fail();
                    break;
                }
                ptx::tc_fence_after();
                const int n = blocks_of(sg);
                int nq = 0, np = 0;  // S MMAs / P.V MMAs issued in this segment
                uint64_t t0 = 0;
                while (np < n) {
                    bool progress = false;
                    // P.V for block np once P is ready (and, for the first
                    // block, once the previous epilogue has read O).
                    if (np < nq) {
                        const uint32_t j = jj + np;
                        if (ptx::mbar_try_wait(bar(S::P_FULL + (j & 1)), (j >> 1) & 1) &&
                            (np > 0 || kk == 0 ||
                             ptx::mbar_try_wait(bar(S::O_FREE), (kk - 1) & 1))) {
                            ptx::tc_fence_after();
                            const uint32_t vst =
                                sb + S::OFF_STAGE + (j % S::NS) * S::STAGE_BYTES + S::TILE_BYTES;
                            const uint32_t pt = tmem + S::TM_P + (j & 1) * (kBlock / 2);
                            // A block of one 64-token step has no keys in its
                            // second half (P is zero there): half the MMAs.
                            const int nk = sg.chunk_end - sg.chunk_begin - 2 * np >= 2
                                               ? kBlock / 16
                                               : kChunk / 16;
#pragma unroll
                            for (int k = 0; k < kBlock / 16; ++k) {
                                if (k >= nk) break;
                                const uint64_t bd =
                                    smem_desc_sw128(vst + k * 16 * 128, S::HALF_BYTES, 1024);
                                ptx::mma_bf16_ts(tmem + S::TM_O, pt + k * 8, bd, idesc_pv,
                                                 (np == 0 && k == 0) ? 0u : 1u);
                            }
                            ptx::mma_commit(bar(S::KV_EMPTY + j % S::NS));
                            ptx::mma_commit(bar(S::P_FREE + (j & 1)));
                            ++np;
                            progress = true;
                        }
                    }
                    // S for block nq once its K/V has landed and its S buffer
                    // has been read by the softmax (block nq - 2).
                    if (nq < n) {
                        const uint32_t j = jj + nq;
                        const int s = j % S::NS;
                        if (ptx::mbar_try_wait(bar(S::KV_FULL + s), (j / S::NS) & 1) &&
                            (j < 2 ||
                             ptx::mbar_try_wait(bar(S::S_FREE + (j & 1)), ((j >> 1) - 1) & 1))) {
                            ptx::tc_fence_after();
                            const uint32_t kst = sb + S::OFF_STAGE + s * S::STAGE_BYTES;
                            const uint32_t d_s = tmem + S::TM_S + (j & 1) * kBlock;
#pragma unroll
                            for (int k = 0; k < D / 16; ++k) {
                                const uint64_t ad = smem_desc_sw128(
                                    sb + S::OFF_Q + (k >> 2) * S::QATOM_BYTES + (k & 3) * 32, 16,
                                    1024);
                                const uint64_t bd = smem_desc_sw128(
                                    kst + (k >> 2) * S::HALF_BYTES + (k & 3) * 32, 16, 1024);
                                ptx::mma_bf16(d_s, ad, bd, idesc_qk, k > 0 ? 1u : 0u);
                            }
                            ptx::mma_commit(bar(S::S_FULL + (j & 1)));
                            ++nq;
                            progress = true;
                        }
                    }
                    if (progress) {
                        t0 = 0;
                    } else {
                        const uint64_t now = ptx::globaltimer();
                        if (t0 == 0) t0 = now;
                        if (now - t0 > a.wait_ns || *abort_flag) {
                            ok = false;
                            break;
                        }
                    }
                }
                if (!ok) {
                    fail();
                    break;
                }
                ptx::mma_commit(bar(S::O_FULL));
                jj += n;
                ++kk;
            }
            // Every MMA issued above must finish before TMEM is released
            // (they read only landed tiles and written P: they complete).
            ptx::mma_commit(bar(S::DRAIN));
            (void)ptx::mbar_wait(bar(S::DRAIN), 0, ptx::kDrainLimitNs);
        }
    } else if (warp == 6) {
        // ================= idle (see kPrefixThreads)
    } else {
        // ================= softmax + epilogue warpgroup (warps 0-3)
        constexpr int R = kRows / F;    // tile rows per replica
        constexpr int KF = kBlock / F;  // keys of each block one replica handles
        const int r = threadIdx.x;      // tile row == TMEM lane
        const int g = r / R;            // replica of this row (warp-uniform)
        const int lt = r % R;           // tile row within the replica
        const int k0 = g * KF;          // first key of this replica in a block
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        // Query row of tile row lt when the row block holds Mrb query rows
        // (R when none).  A warp reaches only its own 32 TMEM lanes, and the
        // four warps run on the SM's four sub-partitions, so the rows are
        // spread evenly over the replica's 32-lane groups: with 80 rows and
        // one replica each group takes 20 and every sub-partition computes
        // 20 rows' exponentials, instead of 32, 32, 16 and 0.
        auto query_row = [&](int Mrb) -> int {
            constexpr int groups = R / 32;
            const int per = (Mrb + groups - 1) / groups;
            const int within = lt & 31;
            const int q = (lt >> 5) * per + within;
            return (within < per && q < Mrb) ? q : R;
        };
        if constexpr (early) {
            ptx::grid_dep_wait();  // Q and the tree inputs may be the previous kernel's
            ptx::grid_dep_launch();
        }
        Walker w;
        init_walker(w);
        auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
            const bool ok = ptx::mbar_wait(b, parity, a.wait_ns);
            const bool all = __all_sync(kFull, ok && !*abort_flag);
            if (!ok) fail();
            return all;
        };
        // P columns outside this replica's keys must read as zero: clear both
        // P buffers once; afterwards only the replica's own columns are written.
        {
            float z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll
            for (int c = 0; c < kBlock; c += 32) ptx::tmem_st32(lane_base + S::TM_P + c, z);
            ptx::tmem_wait_st();
        }
        // Stage Q rows of a segment into the swizzled K-major A tile (every
        // replica gets a copy).
        auto load_q = [&](const Segment& sg) {
            const int Mrb = min(R, a.M - sg.rb * kRows);
            const int lq = query_row(Mrb);
            uint8_t* qs = smem + S::OFF_Q;
            if (lq < Mrb) {
                const int rr = sg.rb * kRows + lq;
                const int t = rr / a.G, gg = rr % a.G;
                const int h = sg.hk * a.G + gg;
                const uint4* src = reinterpret_cast<const uint4*>(
                    a.q + ((static_cast<size_t>(sg.b) * a.T + t) * a.Hq + h) * D);
#pragma unroll
                for (int c = 0; c < D / 8; ++c) {
                    const uint4 v = __ldg(src + c);
                    *reinterpret_cast<uint4*>(qs + (c >> 3) * S::QATOM_BYTES +
                                              sw128_offset(r, c & 7)) = v;
                }
            } else {
#pragma unroll
                for (int c = 0; c < D / 8; ++c)
                    *reinterpret_cast<uint4*>(qs + (c >> 3) * S::QATOM_BYTES +
                                              sw128_offset(r, c & 7)) = make_uint4(0, 0, 0, 0);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(S::Q_FULL));
        };

        uint32_t jj = 0, kk = 0;
        Segment cur;
        bool have = w.next(cur);
        bool ok = true;
        if (have) load_q(cur);
        while (ok && have) {
            const int Mrb = min(R, a.M - cur.rb * kRows);
            const int lr = query_row(Mrb);  // query row within the row block
            const bool row_ok = lr < Mrb;
            const bool warp_any = __any_sync(kFull, row_ok);
            const int prow = g * R + lr;    // row of this copy's partial in a slot
            bool bad;
            const int L = clamp_seq_len(cur.len_raw, a.P, a.max_pages, bad);
            const int tree_ch = chunks_of(L);  // the tree chunk (kTreeChunk)
            // Ancestor bits of this row's tree node (tree modes): given, or
            // built here from the parent array by this warp (pointer
            // jumping, as in tree_mask_kernel).
            uint64_t tbits = 0;
            if constexpr (TM != kTreeNone) {
                const int t = row_ok ? (cur.rb * kRows + lr) / a.G : 0;
                if (a.parents != nullptr) {
                    uint64_t anc[2];
                    const bool bad_tree = warp_tree_mask(
                        a.parents + static_cast<size_t>(cur.b) * a.parents_stride, a.T, lane, anc);
                    tbits = pick64(anc[0], anc[1], t);
                    // One warp per tree reports and writes the masks out: the
                    // one holding the tree of the sequence's first unit.
                    bool bad_l;
                    const bool writer =
                        warp == 0 && cur.unit == cur.b * upb &&
                        cur.chunk_end ==
                            unit_chunks(cur.len_raw, a.P, a.max_pages, TM, a.T, bad_l) &&
                        (a.parents_stride != 0 || cur.b == 0);
                    if (writer && bad_tree && lane == 0)
                        report(a.status, TREE_ATTN_STATUS_BAD_PARENT);
                    if (writer && a.mask_out != nullptr) {
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int i = lane + 32 * hh;
                            if (i < a.T)
                                a.mask_out[static_cast<size_t>(cur.b) * a.parents_stride + i] =
                                    anc[hh];
                        }
                    }
                } else if (row_ok) {
                    tbits = a.mask[static_cast<size_t>(cur.b) * a.mask_stride + t];
                }
                if (a.T < 64) tbits &= (1ull << a.T) - 1ull;
            }
            // Keys of chunk c that this row may attend (bit i = key i): the
            // committed prefix unmasked, the tree tokens by the ancestor bits,
            // nothing past the data or outside this segment.
            auto chunk_vis = [&](int c) -> uint64_t {
                if (c >= cur.chunk_end) return 0ull;
                if (TM == kTreeChunk && c == tree_ch) return tbits;
                const long long rem =
                    static_cast<long long>(L) - static_cast<long long>(c) * kChunk;
                uint64_t v = rem >= kChunk ? ~0ull : (rem <= 0 ? 0ull : ((1ull << rem) - 1ull));
                if (TM == kTreeInCache) {
                    if (rem >= 0)
                        v |= rem < 64 ? (tbits << rem) : 0ull;
                    else
                        v |= -rem < 64 ? (tbits >> -rem) : 0ull;
                }
                return v;
            };
            // Rows of chunk c that hold keys (the rest is stale or foreign data
            // whose V rows are zeroed before P.V).
            auto chunk_rows = [&](int c) -> int {
                if (c >= cur.chunk_end) return 0;
                if (TM == kTreeChunk && c == tree_ch) return a.T;
                const long long e = static_cast<long long>(L) + (TM == kTreeInCache ? a.T : 0) -
                                    static_cast<long long>(c) * kChunk;
                return e >= kChunk ? kChunk : (e <= 0 ? 0 : static_cast<int>(e));
            };
            float m_ref = kNegInf;  // base-2 reference; -inf until a key is seen
            float l_sum = 0.f;
            // The probabilities enter P.V as bf16.  In blocks holding tree
            // keys (and everywhere under an explicit mask) a row may see just
            // a few keys -- tree tokens after a short prefix -- where that
            // rounding does not average out, so l_err sums bf16(p) - p there;
            // the epilogue rescales the row's accumulator by
            // l_sum / (l_sum + l_err): out keeps a consistent numerator and
            // denominator, while lse keeps the exact sum.
            float l_err = 0.f;
            for (int ch = cur.chunk_begin; ch < cur.chunk_end; ch += 2, ++jj) {
                const bool first = ch == cur.chunk_begin;
                const int nh = min(2, cur.chunk_end - ch);
                // Two whole chunks of committed prefix: every key is there and
                // visible to every row (the common case, decided per block).
                const bool plain = nh == 2 && static_cast<long long>(ch + 2) * kChunk <= L;
                // Otherwise: visibility of this thread's KF keys (k0 .. k0 + KF - 1).
                uint64_t vis0 = ~0ull, vis1 = ~0ull;
                int rows0 = kChunk, rows1 = kChunk;
                if (!plain) {
                    if constexpr (KF == 128) {
                        vis0 = chunk_vis(ch);
                        vis1 = chunk_vis(ch + 1);
                    } else if constexpr (KF == 64) {
                        vis0 = chunk_vis(ch + g) | 0ull;
                    } else {
                        vis0 = (chunk_vis(ch + (g >> 1)) >> ((g & 1) * 32)) | 0xffffffff00000000ull;
                    }
                    rows0 = chunk_rows(ch);
                    rows1 = chunk_rows(ch + 1);
                }
                const bool all_vis = vis0 == ~0ull && (KF < 128 || vis1 == ~0ull);
                // Explicit mask bytes of this row's keys, fetched before the
                // scores are waited for (16 keys per vector).
                uint4 mbits[DENSE ? KF / 16 : 1];
                if constexpr (DENSE) {
                    const int p0 = ch * kChunk + k0;
                    const int lim = min(L, a.dense_cols);
                    const uint8_t* mrow = a.dense;
                    if (row_ok)
                        mrow += (static_cast<size_t>(cur.b) * a.T + (cur.rb * kRows + lr) / a.G) *
                                a.dense_cols;
#pragma unroll
                    for (int j = 0; j < KF / 16; ++j) {
                        mbits[j] = make_uint4(0, 0, 0, 0);
                        if (row_ok && p0 + 16 * j < lim)
                            mbits[j] = __ldg(reinterpret_cast<const uint4*>(mrow + p0 + 16 * j));
                    }
                }
                if (!wait_all(bar(S::S_FULL + (jj & 1)), (jj >> 1) & 1)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                float s[KF];
                if (warp_any) {
                    const uint32_t ta = lane_base + S::TM_S + (jj & 1) * kBlock + k0;
#pragma unroll
                    for (int c = 0; c < KF; c += 32) ptx::tmem_ld32(ta + c, s + c);
                    ptx::tmem_wait_ld();
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(S::S_FREE + (jj & 1)));

                // Softmax in the base-2 domain: x = s * scale * log2(e)
                // (scale > 0, so the max of the raw scores gives the max of x).
                float alpha = 1.f;
                bool rescale = false;
                if (!all_vis) {
                    // Keys this row may not see score -inf: they add nothing
                    // to the max or the sum, and their probabilities are 0.
#pragma unroll
                    for (int i = 0; i < KF; ++i) {
                        const uint64_t bit = i < 64 ? (vis0 >> i) : (vis1 >> (i - 64));
                        if ((bit & 1ull) == 0) s[i] = kNegInf;
                    }
                }
                if constexpr (DENSE) {
                    // Hidden keys score -inf: they add nothing to the max or
                    // the sum, and their probabilities are exactly 0.
#pragma unroll
                    for (int i = 0; i < KF; ++i) {
                        const uint4 w4 = mbits[i / 16];
                        const uint32_t w = ((i % 16) / 4 == 0)   ? w4.x
                                           : ((i % 16) / 4 == 1) ? w4.y
                                           : ((i % 16) / 4 == 2) ? w4.z
                                                                 : w4.w;
                        if (((w >> (8 * (i % 4))) & 0xffu) == 0) s[i] = kNegInf;
                    }
                }
                // Blocks whose rounding of P to bf16 is tracked (see the epilogue).
                const bool track = DENSE || (TM != kTreeNone && !plain &&
                                             ((TM == kTreeChunk && ch + nh > tree_ch) ||
                                              (TM == kTreeInCache && (ch + nh) * kChunk > L)));
                if (row_ok) {
                    // Eight independent partial maxima / sums keep the
                    // dependency chains short.
                    float mp[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) mp[u] = kNegInf;
#pragma unroll
                    for (int i = 0; i < KF; i += 2)
                        mp[(i >> 1) & 7] = ptx::fmax3(mp[(i >> 1) & 7], s[i], s[i + 1]);
                    float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                                     fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
                    mx *= a.scale_log2;
                    if (first) {
                        m_ref = mx;
                    } else if (mx > m_ref + 8.f) {
                        // Keep 2^(x - m_ref) <= 2^8: move the reference and
                        // rescale the running sums (alpha = 0 if there were none).
                        alpha = ptx::ex2(m_ref - mx);
                        m_ref = mx;
                        l_sum *= alpha;
                        l_err *= alpha;
                        rescale = true;
                    }
                    const float neg_m = (m_ref == kNegInf) ? 0.f : -m_ref;
                    // Keys in pairs: one f32x2 fma forms both exponents and one
                    // f32x2 add folds both probabilities into the running sums
                    // (key i into sum i & 7, as eight scalar sums would), so
                    // the issue slots go to the exponentials.
                    const uint64_t sc2 = ptx::f2_pack(a.scale_log2, a.scale_log2);
                    const uint64_t nm2 = ptx::f2_pack(neg_m, neg_m);
                    uint64_t sp2[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) sp2[u] = ptx::f2_pack(0.f, 0.f);
#pragma unroll
                    for (int i = 0; i < KF; i += 2) {
                        float x0, x1;
                        ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(s[i], s[i + 1]), sc2, nm2), x0, x1);
                        s[i] = ptx::ex2(x0);
                        s[i + 1] = ptx::ex2(x1);
                        sp2[(i >> 1) & 3] = ptx::f2_add(sp2[(i >> 1) & 3], ptx::f2_pack(s[i], s[i + 1]));
                    }
                    float sp[8];
#pragma unroll
                    for (int u = 0; u < 4; ++u) ptx::f2_unpack(sp2[u], sp[2 * u], sp[2 * u + 1]);
                    l_sum += ((sp[0] + sp[1]) + (sp[2] + sp[3])) +
                             ((sp[4] + sp[5]) + (sp[6] + sp[7]));
                }
                // P buffer (jj & 1) is free once PV(jj - 2) has completed.
                if (jj >= 2 && !wait_all(bar(S::P_FREE + (jj & 1)), ((jj >> 1) - 1) & 1)) {
                    ok = false;
                    break;
                }
                if (warp_any) {
                    const uint32_t tp = lane_base + S::TM_P + (jj & 1) * (kBlock / 2) + k0 / 2;
                    uint32_t pk[KF / 2];
                    // With tracking, sum the rounding errors of the bf16 values
                    // P.V will use, while the pairs are packed (bf16(p) - p).
                    // A lane without a query row packs whatever its registers
                    // hold: its P row only reaches its own O row, which is
                    // never stored.
                    float sr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int i = 0; i < KF / 2; ++i) {
                        pk[i] = pack_bf16(s[2 * i], s[2 * i + 1]);
                        if (track && row_ok) {
                            sr[(2 * i) & 3] += __uint_as_float(pk[i] << 16) - s[2 * i];
                            sr[(2 * i + 1) & 3] +=
                                __uint_as_float(pk[i] & 0xffff0000u) - s[2 * i + 1];
                        }
                    }
                    if (track && row_ok) l_err += (sr[0] + sr[1]) + (sr[2] + sr[3]);
                    if constexpr (KF / 2 >= 32) {
#pragma unroll
                        for (int c = 0; c < KF / 2; c += 32)
                            ptx::tmem_st32(tp + c, reinterpret_cast<const float*>(pk + c));
                    } else {
                        ptx::tmem_st16(tp, pk);
                    }
                    ptx::tmem_wait_st();
                }
                if (__any_sync(kFull, rescale)) {
                    // O must hold PV(jj - 1) before it is rescaled in place.
                    if (!wait_all(bar(S::P_FREE + ((jj - 1) & 1)), ((jj - 1) >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t to = lane_base + S::TM_O;
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        float o[32];
                        ptx::tmem_ld32(to + c, o);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        ptx::tmem_st32(to + c, o);
                    }
                    ptx::tmem_wait_st();
                }
                if (rows0 < kChunk || rows1 < kChunk) {
                    // Rows past the keys of each chunk hold stale or foreign
                    // data; zero their V rows so 0 * garbage cannot reach O.
                    if (!wait_all(bar(S::KV_FULL + jj % S::NS), (jj / S::NS) & 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t vst =
                        sb + S::OFF_STAGE + (jj % S::NS) * S::STAGE_BYTES + S::TILE_BYTES;
                    const int n0 = kChunk - rows0;
                    const int items = (n0 + kChunk - rows1) * S::DH * 8;
                    for (int it = r; it < items; it += 128) {
                        const int idx = it / (S::DH * 8);
                        const int row = idx < n0 ? rows0 + idx : kChunk + rows1 + (idx - n0);
                        const int rem = it % (S::DH * 8);
                        st_shared_v4(vst + (rem >> 3) * S::HALF_BYTES + row * 128 + (rem & 7) * 16,
                                     0u, 0u, 0u, 0u);
                    }
                    ptx::fence_proxy_async_smem();
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(S::P_FULL + (jj & 1)));
            }
            if (!ok) break;
            // Stage the next segment's Q first so its S MMA overlaps this
            // epilogue (every S MMA of this segment has completed).
            Segment nxt;
            const bool have_next = w.next(nxt);
            if (have_next) load_q(nxt);
            if (!wait_all(bar(S::O_FULL), kk & 1)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            float* slot = a.ws + static_cast<size_t>(cur.unit + blockIdx.x) * slot_floats(D);
            const uint32_t to = lane_base + S::TM_O;
            const float acc_scale =
                (l_err != 0.f && l_sum + l_err > 0.f) ? __fdividef(l_sum, l_sum + l_err) : 1.f;
            if (!have_next) {
                // Last segment of this CTA: every MMA and copy has completed,
                // so the K/V ring is free.  Each row copy stages its O (scaled
                // by its own rounding correction) and (m, l) there, rows
                // padded to D + 4 floats (conflict-free).  Then the four warps
                // fold the F copies of each query row into one partial, so the
                // merge reads one partial per CTA instead of F, and store it a
                // whole row per warp instruction: stored straight from TMEM,
                // one row per thread, each instruction would touch 32 rows.
                constexpr int RS = D + 4;
                constexpr int VE = D / 32;                                    // floats per lane
                float* stg = reinterpret_cast<float*>(smem + S::OFF_STAGE);  // [F][R][RS]
                float* stg_ml = stg + F * R * RS;                             // [F][R][2]
                if (warp_any) {
                    float* dst = stg + static_cast<size_t>(g * R + lr) * RS;
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        float o[32];
                        ptx::tmem_ld32(to + c, o);
                        ptx::tmem_wait_ld();
                        if (row_ok) {
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                *reinterpret_cast<float4*>(dst + c + 4 * i) =
                                    make_float4(o[4 * i] * acc_scale, o[4 * i + 1] * acc_scale,
                                                o[4 * i + 2] * acc_scale, o[4 * i + 3] * acc_scale);
                        }
                    }
                    if (row_ok) {
                        stg_ml[(g * R + lr) * 2] = m_ref;
                        stg_ml[(g * R + lr) * 2 + 1] = l_sum;
                    }
                }
                // The four warps meet on an mbarrier rather than bar.sync: a
                // warp that gave up on an earlier wait never arrives, and
                // this wait is bounded.  Used once per launch (phase 0).
                if (lane == 0) ptx::mbar_arrive(bar(S::FOLD));
                if (!wait_all(bar(S::FOLD), 0)) {
                    ok = false;
                    break;
                }
                // RU rows per warp at a time: their shared-memory reads are
                // all issued before any is used.
                constexpr int RU = 4 / F;
                for (int q0 = warp; q0 < Mrb; q0 += 4 * RU) {
                    float mg[RU][F], lg[RU][F], x[RU][F][VE];
#pragma unroll
                    for (int u = 0; u < RU; ++u) {
                        const int q = q0 + 4 * u;
#pragma unroll
                        for (int k = 0; k < F; ++k) {
                            mg[u][k] = kNegInf;
                            lg[u][k] = 0.f;
#pragma unroll
                            for (int e = 0; e < VE; ++e) x[u][k][e] = 0.f;
                            if (q < Mrb) {
                                mg[u][k] = stg_ml[(k * R + q) * 2];
                                lg[u][k] = stg_ml[(k * R + q) * 2 + 1];
                                const float* src =
                                    stg + static_cast<size_t>(k * R + q) * RS + lane * VE;
                                if constexpr (VE == 4) {
                                    const float4 v4 = *reinterpret_cast<const float4*>(src);
                                    x[u][k][0] = v4.x;
                                    x[u][k][1] = v4.y;
                                    x[u][k][2] = v4.z;
                                    x[u][k][3] = v4.w;
                                } else {
                                    const float2 v2 = *reinterpret_cast<const float2*>(src);
                                    x[u][k][0] = v2.x;
                                    x[u][k][1] = v2.y;
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < RU; ++u) {
                        const int q = q0 + 4 * u;
                        if (q >= Mrb) break;
                        float mx = kNegInf;
#pragma unroll
                        for (int k = 0; k < F; ++k) mx = fmaxf(mx, mg[u][k]);
                        float lc = 0.f;
                        float o[VE];
#pragma unroll
                        for (int e = 0; e < VE; ++e) o[e] = 0.f;
#pragma unroll
                        for (int k = 0; k < F; ++k) {
                            const float wk =
                                (mg[u][k] == kNegInf) ? 0.f : ptx::ex2(mg[u][k] - mx);
                            lc = fmaf(wk, lg[u][k], lc);
#pragma unroll
                            for (int e = 0; e < VE; ++e) o[e] = fmaf(wk, x[u][k][e], o[e]);
                        }
                        float* acc = slot + 2 * kRows + static_cast<size_t>(q) * D + lane * VE;
                        if constexpr (VE == 4) {
                            *reinterpret_cast<float4*>(acc) = make_float4(o[0], o[1], o[2], o[3]);
                        } else {
                            *reinterpret_cast<float2*>(acc) = make_float2(o[0], o[1]);
                        }
                        if (lane == 0) {
                            slot[q] = mx;
                            slot[kRows + q] = lc;
                        }
                    }
                }
            } else if (warp_any) {
                // A later segment follows: the ring holds its K/V, so each row
                // stores its own partial (hidden behind the next segment's
                // loads, which are already in flight).
                float4* acc =
                    reinterpret_cast<float4*>(slot + 2 * kRows + static_cast<size_t>(prow) * D);
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    float o[32];
                    ptx::tmem_ld32(to + c, o);
                    ptx::tmem_wait_ld();
                    if (row_ok) {
                        if (acc_scale != 1.f) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] *= acc_scale;
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            acc[c / 4 + i] =
                                make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                    }
                }
                if (row_ok) {
                    slot[prow] = m_ref;
                    slot[kRows + prow] = l_sum;
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(S::O_FREE));
            ++kk;
            cur = nxt;
            have = have_next;
        }
    }

    // ---------------- teardown
    __syncwarp();  // lanes 1-31 of the producer / MMA warps wait for lane 0
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, S::TMEM_COLS);
    }
}

#ifndef TREE_ATTN_EARLY_TU
// ===========================================================================
// Suffix pass + merge.  One warp per query row; lane l holds elements
// [l*E, l*E + E) of the head dimension.
// ===========================================================================
struct MergeArgs {
    const uint16_t* q;
    const uint16_t* tree_k;
    const uint16_t* tree_v;
    const uint64_t* mask;
    const int32_t* seq_lens;
    const float* ws;
    uint16_t* out;
    float* lse;
    int B, Hq, Hkv, G, T, M, RB, P, max_pages, n_ctas;
    int wpr;  // warps per query row in the merge (1, 2, 4 or 8)
    int rpw;  // rows per warp (taken in turn; merge without the tree pass only)
    float scale_log2;
    int mask_stride;  // 0: one tree for the batch; T: tree b at mask[b * T]
    // Tree tokens padded inside the paged cache (tree_k / tree_v unused):
    // tree token j of sequence b sits at logical position seq_lens[b] + j.
    int tree_in_cache;
    const uint16_t* k_pages;
    const uint16_t* v_pages;
    const int32_t* block_table;
    int num_pages;
    int32_t* status;
    // Tree masks built here from parent arrays (mask == nullptr then):
    // parents [T] (parents_stride 0) or [B][T] (parents_stride T); the masks
    // are also written to mask_out when it is not null.
    const int32_t* parents;
    int parents_stride;
    uint64_t* mask_out;
    // TreeMode of the prefix pass: with the tree on its work line there is
    // no suffix pass here.
    int tmode;
    int ovh;  // overhead slots per unit on the work line
};

template <int E>
__device__ __forceinline__ void load_bf16(const uint16_t* p, float* v) {
    if constexpr (E == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        v[0] = __uint_as_float(u.x << 16);
        v[1] = __uint_as_float(u.x & 0xffff0000u);
        v[2] = __uint_as_float(u.y << 16);
        v[3] = __uint_as_float(u.y & 0xffff0000u);
    } else {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
        v[0] = __uint_as_float(u << 16);
        v[1] = __uint_as_float(u & 0xffff0000u);
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
    return v;
}

// E consecutive fp32 accumulator values through L2 only, or zeros.
template <int E>
__device__ __forceinline__ void load_acc(const float* p, bool use, float* v) {
    if (use) {
        if constexpr (E == 4) {
            const float4 x = __ldcg(reinterpret_cast<const float4*>(p));
            v[0] = x.x;
            v[1] = x.y;
            v[2] = x.z;
            v[3] = x.w;
        } else {
            const float2 x = __ldcg(reinterpret_cast<const float2*>(p));
            v[0] = x.x;
            v[1] = x.y;
        }
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = 0.f;
    }
}


// One CTA = 4 warps = 4 / wpr query rows; the wpr warps of a row split its
// partials (virtual slot v goes to warp v % wpr) and combine through shared
// memory.  Every independent load of a phase is issued before any of its
// results is used, so each phase costs about one memory round trip.
// SUFFIX: the two-pass form (the tree keys are attended here); otherwise the
// tree rode on the prefix pass's work line and this is the merge alone.
// MULTI: each warp takes a.rpw rows in turn (merge alone only).
template <int D, int F, bool SUFFIX, bool MULTI>
__global__ void __launch_bounds__(32 * kMergeWarps, kMergeResident)
    suffix_merge_kernel(const MergeArgs a) {
    constexpr int E = D / 32;
    // Accumulator rows each warp loads in the first round trip, together
    // with the (m, l) of its partials (the later round trips reuse the same
    // registers for four rows at a time, so NF is at least 4).
    constexpr int NF = 4;
    constexpr int R = kRows / F;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int wpr = a.wpr;
    const int rows_per_cta = kMergeWarps / wpr;
    const int wr = warp / wpr;   // row slot of this warp in the CTA
    const int sub = warp % wpr;  // this warp's share of the row's partials
    const int unit = blockIdx.x;
    const int rb = unit % a.RB;
    const int hk = (unit / a.RB) % a.Hkv;
    const int b = unit / (a.RB * a.Hkv);
    // The next kernel may start its prologue once every CTA of this grid is
    // running; it waits for this grid before reading anything it writes.
    ptx::grid_dep_launch();

    __shared__ float red_m[kMergeWarps];
    __shared__ float red_l[kMergeWarps];
    __shared__ float red_o[kMergeWarps][D];

    // Parent array of this row's tree (masks built here): lane l holds the
    // parents of nodes l and l + 32.  Loaded now, used after the plan.
    constexpr bool suffix_here = SUFFIX;
    int par0 = -1, par1 = -1;
    if (suffix_here && a.parents != nullptr && sub == 0) {
        const int32_t* pr = a.parents + static_cast<size_t>(b) * a.parents_stride;
        if (lane < a.T) par0 = pr[lane];
        if (lane + 32 < a.T) par1 = pr[lane + 32];
    }

    // ---- work-line plan of this unit (inputs only): sequence lengths of
    // the whole batch, the first 32 * kPlanRegs and this unit's own loaded in
    // one round trip.
    const int upb = a.Hkv * a.RB;
    int32_t lraw[kPlanRegs];
#pragma unroll
    for (int i = 0; i < kPlanRegs; ++i) {
        const int bi = 32 * i + lane;
        lraw[i] = bi < a.B ? a.seq_lens[bi] : 0;
    }
    const int32_t l_own = a.seq_lens[b];
    long long W = 0, base_b = 0;
    auto add_len = [&](int bi, int32_t L_raw) {
        bool bad_i;
        const int n =
            bi < a.B ? unit_len(unit_chunks(L_raw, a.P, a.max_pages, a.tmode, a.T, bad_i), a.ovh)
                     : 0;
        W += __reduce_add_sync(kFull, n);
        base_b += __reduce_add_sync(kFull, bi < b ? n : 0);
    };
#pragma unroll
    for (int i = 0; i < kPlanRegs; ++i)
        if (32 * i < a.B) add_len(32 * i + lane, lraw[i]);
#pragma unroll 1
    for (int b0 = 32 * kPlanRegs; b0 < a.B; b0 += 32) {
        const int bi = b0 + lane;
        add_len(bi, bi < a.B ? a.seq_lens[bi] : 0);
    }
    W *= upb;
    base_b *= upb;
    bool bad;
    const int nch = unit_chunks(l_own, a.P, a.max_pages, a.tmode, a.T, bad);
    int c_first = 0, c_last = -1;
    // A prefix CTA folds its F row copies into one partial in its last
    // segment.  Every CTA before c_last ends inside this unit; c_last does
    // only if its range stops at the unit's end.
    bool last_folded = F == 1;
    if (nch > 0) {
        // The unit's chunks, then its overhead slots (no chunks there).
        const int len = unit_len(nch, a.ovh);
        const long long ustart = base_b + static_cast<long long>(unit - b * upb) * len;
        c_first = cta_of(ustart, W, a.n_ctas);
        c_last = cta_of(ustart + nch - 1, W, a.n_ctas);
        if (F > 1) last_folded = cta_start(c_last + 1, W, a.n_ctas) <= ustart + len;
    }

    // Each warp takes rpw rows in turn (more than one only for the merge
    // alone, when one row per warp would need more CTAs than fit at once).
    static_assert(!(SUFFIX && MULTI), "the tree pass runs one row per warp");
    const int rpw = MULTI ? a.rpw : 1;
#pragma unroll 1
    for (int rep = 0; rep < rpw; ++rep) {
        const int r = (blockIdx.y * rpw + rep) * rows_per_cta + wr;
        const int rr = rb * kRows + r;
        const bool active = r < kRows && rr < a.M;
        int t = 0, h = 0;
        if (active) {
            t = rr / a.G;
            h = hk * a.G + rr % a.G;
        }

        // ---- suffix (sub-warp 0 of each row): softmax over the tree keys
        // mask[t] allows, four keys per round trip.  Reads only inputs of this
        // call, so it runs before waiting for the prefix pass.
        float m_s = kNegInf, l_s = 0.f;
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
        // Tree mask of this row's node: given, or built here from the parent
        // array -- by walking the parent links up from node t (the row's warp
        // holds the array in registers: one shuffle per ancestor).  A link that
        // does not point to an earlier node ends the walk (that node is then a
        // root, as in tree_mask_kernel, which reports it).
        uint64_t bits = 0;
        if (suffix_here && a.parents != nullptr && sub == 0) {
            for (int node = t, steps = 0; node >= 0 && steps < 64; ++steps) {
                bits |= 1ull << node;
                const int n0 = __shfl_sync(kFull, par0, node & 31);
                const int n1 = __shfl_sync(kFull, par1, node & 31);
                const int nxt = node < 32 ? n0 : n1;
                node = (nxt >= -1 && nxt < node) ? nxt : -1;
            }
            // One warp per tree validates the array and writes the masks out:
            // the first unit's of the sequence (per-sequence trees) or of the
            // batch (pointer jumping over all nodes, as in tree_mask_kernel).
            const bool writer = unit == b * upb && blockIdx.y == 0 && warp == 0 &&
                                (a.parents_stride != 0 || b == 0);
            uint64_t anc[2] = {0ull, 0ull};
            bool bad_tree = false;
            if (writer)
                bad_tree = warp_tree_mask(a.parents + static_cast<size_t>(b) * a.parents_stride,
                                          a.T, lane, anc);
            if (writer && bad_tree && lane == 0) report(a.status, TREE_ATTN_STATUS_BAD_PARENT);
            if (writer && a.mask_out != nullptr) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int i = lane + 32 * hh;
                    if (i < a.T)
                        a.mask_out[static_cast<size_t>(b) * a.parents_stride + i] = anc[hh];
                }
            }
        } else if (suffix_here && a.mask != nullptr && active && sub == 0) {
            bits = a.mask[static_cast<size_t>(b) * a.mask_stride + t];
        }
        if (a.T < 64) bits &= (1ull << a.T) - 1ull;
        if (suffix_here && active && sub == 0 && (a.mask != nullptr || a.parents != nullptr)) {
            float qv[E];
            load_bf16<E>(a.q + ((static_cast<size_t>(b) * a.T + t) * a.Hq + h) * D + lane * E, qv);
            int L_b = 0;
            if (a.tree_in_cache) {
                bool bad_len;
                L_b = clamp_seq_len(l_own, a.P, a.max_pages, bad_len);
            }
            while (bits != 0) {
                int js[4];
                int n = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    js[i] = 0;
                    if (bits != 0) {
                        js[i] = __ffsll(static_cast<long long>(bits)) - 1;
                        bits &= bits - 1;
                        n = i + 1;
                    }
                }
                float kv[4][E], vv[4][E];
                if (a.tree_in_cache) {
                    // Position L_b + j of the paged cache (the tree padding).
                    int page[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        page[i] = -1;
                        const int pos = L_b + js[i];
                        if (i < n && pos / a.P < a.max_pages)
                            page[i] =
                                a.block_table[static_cast<size_t>(b) * a.max_pages + pos / a.P];
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (i >= n) continue;
                        const int pos = L_b + js[i];
                        if (page[i] < 0 || page[i] >= a.num_pages) {
                            if (lane == 0)
                                report(a.status, pos / a.P < a.max_pages
                                                     ? TREE_ATTN_STATUS_BAD_PAGE
                                                     : TREE_ATTN_STATUS_BAD_SEQ_LEN);
#pragma unroll
                            for (int e = 0; e < E; ++e) kv[i][e] = vv[i][e] = 0.f;
                            continue;
                        }
                        const size_t off =
                            ((static_cast<size_t>(page[i]) * a.Hkv + hk) * a.P + pos % a.P) * D +
                            lane * E;
                        load_bf16<E>(a.k_pages + off, kv[i]);
                        load_bf16<E>(a.v_pages + off, vv[i]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (i < n) {
                            const size_t off =
                                ((static_cast<size_t>(b) * a.T + js[i]) * a.Hkv + hk) * D +
                                lane * E;
                            load_bf16<E>(a.tree_k + off, kv[i]);
                            load_bf16<E>(a.tree_v + off, vv[i]);
                        }
                    }
                }
                float x[4];
                float mx = m_s;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float dot = 0.f;
                    if (i < n) {
#pragma unroll
                        for (int e = 0; e < E; ++e) dot = fmaf(qv[e], kv[i][e], dot);
                    }
                    x[i] = warp_sum(dot) * a.scale_log2;
                    if (i < n) mx = fmaxf(mx, x[i]);
                }
                const float al = ptx::ex2(m_s - mx);
                l_s *= al;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] *= al;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (i < n) {
                        const float p = ptx::ex2(x[i] - mx);
                        l_s += p;
#pragma unroll
                        for (int e = 0; e < E; ++e) acc[e] = fmaf(p, vv[i][e], acc[e]);
                    }
                }
                m_s = mx;
            }
        }

        // ---- merge with the partials of the prefix pass
        ptx::grid_dep_wait();
        const size_t sf = static_cast<size_t>(slot_floats(D));
        // Partials are indexed by "virtual slot" v: v < n1 is the folded partial
        // of prefix CTA c_first + v (copy 0, tile rows r); the rest are those of
        // c_last: one if it folded, else its F copies (tile rows g * R + r).  This
        // warp takes v = sub, sub + wpr, ...; its k-th one is v = sub + k * wpr.
        const int n1 = c_last - c_first;
        const int nv = (active && nch > 0) ? n1 + (last_folded ? 1 : F) : 0;
        auto v_cta = [&](int v) -> int { return v < n1 ? c_first + v : c_last; };
        auto v_copy = [&](int v) -> int { return v < n1 ? 0 : v - n1; };
        const int nmine = nv > sub ? (nv - sub + wpr - 1) / wpr : 0;
        // With at least one work-line step per CTA every CTA in [c_first, c_last]
        // wrote a partial; only when W < C can some of them be empty.
        const bool every_cta = W >= a.n_ctas;
        auto v_of = [&](int k) -> int { return sub + k * wpr; };
        auto v_m = [&](int v) -> size_t {  // offset of m for virtual slot v
            return static_cast<size_t>(unit + v_cta(v)) * sf + v_copy(v) * R + r;
        };
        auto v_acc = [&](int v) -> size_t {  // offset of this lane's accumulator values
            return static_cast<size_t>(unit + v_cta(v)) * sf + 2 * kRows +
                   static_cast<size_t>(v_copy(v) * R + r) * D + lane * E;
        };
        auto v_work = [&](int v) -> bool {
            return every_cta || cta_has_work(v_cta(v), W, a.n_ctas);
        };
        // One round trip: (m, l) of this warp's first 32 partials (lane k: the
        // k-th) and the accumulator rows of its first four.  Partials are read
        // through L2 only (ld.global.cg): the prefix grid wrote them while this
        // grid was resident.
        // Bit k: the warp's k-th partial exists (one work check per lane, not
        // one per unrolled load below).
        const unsigned have = __ballot_sync(kFull, lane < nmine && v_work(v_of(lane)));
        float m_j = kNegInf, l_j = 0.f;
        if ((have >> lane) & 1u) {
            m_j = __ldcg(a.ws + v_m(v_of(lane)));
            l_j = __ldcg(a.ws + v_m(v_of(lane)) + kRows);
        }
        float v[NF][E];
#pragma unroll
        for (int j = 0; j < NF; ++j) load_acc<E>(a.ws + v_acc(v_of(j)), (have >> j) & 1u, v[j]);
        float mx = fmaxf(m_s, m_j);
#pragma unroll 1
        for (int k = 32 + lane; k < nmine; k += 32)  // rare: more than 32 partials per warp
            if (v_work(v_of(k))) mx = fmaxf(mx, __ldcg(a.ws + v_m(v_of(k))));
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
        if (wpr > 1) {
            if (lane == 0) red_m[warp] = mx;
            __syncthreads();
            for (int s2 = 0; s2 < wpr; ++s2) mx = fmaxf(mx, red_m[wr * wpr + s2]);
        }
        const bool has_keys = mx != kNegInf;
        const float w_s = has_keys ? ptx::ex2(m_s - mx) : 0.f;
        float o[E];
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = acc[e] * w_s;
        float wc = (m_j == kNegInf || !has_keys) ? 0.f : ptx::ex2(m_j - mx);
        float total = l_s * w_s + warp_sum(wc * l_j);
#pragma unroll
        for (int j = 0; j < NF; ++j) {
            const float wj = __shfl_sync(kFull, wc, j);
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] = fmaf(wj, v[j][e], o[e]);
        }
        // Remaining partials of this warp, four accumulator rows per round trip.
#pragma unroll 1
        for (int k0 = 0; k0 < nmine; k0 += 32) {
            if (k0 != 0) {
                const int k = k0 + lane;
                wc = 0.f;
                float lc = 0.f;
                if (k < nmine && v_work(v_of(k))) {
                    const float mm = __ldcg(a.ws + v_m(v_of(k)));
                    wc = (mm == kNegInf) ? 0.f : ptx::ex2(mm - mx);
                    lc = __ldcg(a.ws + v_m(v_of(k)) + kRows);
                }
                total += warp_sum(wc * lc);
            }
            const int nb = min(32, nmine - k0);
#pragma unroll 1
            for (int j0 = (k0 == 0) ? NF : 0; j0 < nb; j0 += 4) {
                float wj[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    wj[j] = __shfl_sync(kFull, wc, j0 + j);
                    load_acc<E>(a.ws + v_acc(v_of(k0 + j0 + j)), j0 + j < nb && wj[j] != 0.f, v[j]);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int e = 0; e < E; ++e) o[e] = fmaf(wj[j], v[j][e], o[e]);
            }
        }
        if (wpr > 1) {
            // Combine the row's warps (all use the same row max mx).
            if (lane == 0) red_l[warp] = total;
#pragma unroll
            for (int e = 0; e < E; ++e) red_o[warp][lane * E + e] = o[e];
            __syncthreads();
            if (sub != 0) continue;
            for (int s2 = 1; s2 < wpr; ++s2) {
                total += red_l[warp + s2];
#pragma unroll
                for (int e = 0; e < E; ++e) o[e] += red_o[warp + s2][lane * E + e];
            }
        }
        if (!active) continue;
        uint16_t* op = a.out + ((static_cast<size_t>(b) * a.T + t) * a.Hq + h) * D + lane * E;
        float* lp = a.lse + (static_cast<size_t>(b) * a.T + t) * a.Hq + h;
        if (!has_keys) {  // no key at all
#pragma unroll
            for (int e = 0; e < E; ++e) op[e] = 0;
            if (lane == 0) *lp = kNegInf;
            continue;
        }
        const float inv = __fdividef(1.f, total);
        if constexpr (E == 4) {
            uint2 pk;
            pk.x = pack_bf16(o[0] * inv, o[1] * inv);
            pk.y = pack_bf16(o[2] * inv, o[3] * inv);
            *reinterpret_cast<uint2*>(op) = pk;
        } else {
            *reinterpret_cast<uint32_t*>(op) = pack_bf16(o[0] * inv, o[1] * inv);
        }
        if (lane == 0) *lp = (mx + log2f(total)) * kLn2;
    }
}

#endif  // !TREE_ATTN_EARLY_TU

template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

using PrefixKernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, PrefixArgs);

// The prefix kernel for a mode (0-3) and a row-copy index (F = 1, 2, 4); the
// explicit-mask form (mode 3) has no early variant.
template <int D, bool EARLY>
PrefixKernel prefix_kernel_for(int mode, int fi) {
    if constexpr (EARLY) {
        const PrefixKernel t[3][3] = {
            {prefix_pass_kernel<D, 1, 0, true>, prefix_pass_kernel<D, 2, 0, true>,
             prefix_pass_kernel<D, 4, 0, true>},
            {prefix_pass_kernel<D, 1, 1, true>, prefix_pass_kernel<D, 2, 1, true>,
             prefix_pass_kernel<D, 4, 1, true>},
            {prefix_pass_kernel<D, 1, 2, true>, prefix_pass_kernel<D, 2, 2, true>,
             prefix_pass_kernel<D, 4, 2, true>}};
        return t[mode][fi];
    } else {
        const PrefixKernel t[4][3] = {
            {prefix_pass_kernel<D, 1, 0, false>, prefix_pass_kernel<D, 2, 0, false>,
             prefix_pass_kernel<D, 4, 0, false>},
            {prefix_pass_kernel<D, 1, 1, false>, prefix_pass_kernel<D, 2, 1, false>,
             prefix_pass_kernel<D, 4, 1, false>},
            {prefix_pass_kernel<D, 1, 2, false>, prefix_pass_kernel<D, 2, 2, false>,
             prefix_pass_kernel<D, 4, 2, false>},
            {prefix_pass_kernel<D, 1, 3, false>, prefix_pass_kernel<D, 2, 3, false>,
             prefix_pass_kernel<D, 4, 3, false>}};
        return t[mode][fi];
    }
}

template <int D, bool EARLY>
cudaError_t launch_prefix_d(const VerifyArgs& v, const void* tmap_k, const void* tmap_v,
                            const void* tmap_tk, const void* tmap_tv, cudaStream_t stream) {
    using S = PrefixShape<D>;
    static int configured_for = -1;  // device on which the smem opt-in was applied
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_for != dev) {
        for (int m = 0; m < (EARLY ? 3 : 4); ++m)
            for (int fi = 0; fi < 3; ++fi) {
                const PrefixKernel k = prefix_kernel_for<D, EARLY>(m, fi);
                e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         S::SMEM_BYTES);
                if (e != cudaSuccess) return e;
            }
        configured_for = dev;
    }
    const int G = v.Hq / v.Hkv;
    const int M = v.T * G;
    PrefixArgs pa;
    pa.block_table = v.block_table;
    pa.seq_lens = v.seq_lens;
    pa.q = v.q;
    pa.ws = v.ws;
    pa.status = v.status;
    pa.B = v.B;
    pa.Hq = v.Hq;
    pa.Hkv = v.Hkv;
    pa.G = G;
    pa.T = v.T;
    pa.M = M;
    pa.RB = (M + kRows - 1) / kRows;
    pa.P = v.P;
    pa.max_pages = v.max_pages;
    pa.num_pages = v.num_pages;
    pa.n_ctas = v.n_ctas;
    pa.scale_log2 = v.scale_log2;
    pa.dense = v.dense;
    pa.dense_cols = v.dense_cols;
    pa.tmode = v.dense != nullptr ? kTreeNone : v.tmode;
    pa.mask = v.mask;
    pa.mask_stride = v.mask_stride;
    pa.parents = v.parents;
    pa.parents_stride = v.parents_stride;
    pa.mask_out = v.mask_out;
    pa.ovh = v.ovh;
    pa.wait_ns = v.wait_ns;
    const CUtensorMap& tk = *static_cast<const CUtensorMap*>(tmap_k);
    const CUtensorMap& tv = *static_cast<const CUtensorMap*>(tmap_v);
    const CUtensorMap& ttk = *static_cast<const CUtensorMap*>(tmap_tk);
    const CUtensorMap& ttv = *static_cast<const CUtensorMap*>(tmap_tv);
    const int F = pa.RB == 1 ? replicas_of(M) : 1;
    const int mode = v.dense != nullptr ? kModeDense : v.tmode;
    const PrefixKernel kernel = prefix_kernel_for<D, EARLY>(mode, F == 4 ? 2 : (F == 2 ? 1 : 0));
    return launch_pdl(kernel, dim3(v.n_ctas), dim3(kPrefixThreads), S::SMEM_BYTES, stream, tk, tv,
                      ttk, ttv, pa);
}

#ifndef TREE_ATTN_EARLY_TU
template <int D>
cudaError_t launch_merge_d(const VerifyArgs& v, cudaStream_t stream) {
    const int G = v.Hq / v.Hkv;
    const int M = v.T * G;
    const int RB = (M + kRows - 1) / kRows;
    MergeArgs ma;
    ma.q = v.q;
    ma.tree_k = v.tree_k;
    ma.tree_v = v.tree_v;
    ma.mask = v.mask;
    ma.seq_lens = v.seq_lens;
    ma.ws = v.ws;
    ma.out = v.out;
    ma.lse = v.lse;
    ma.B = v.B;
    ma.Hq = v.Hq;
    ma.Hkv = v.Hkv;
    ma.G = G;
    ma.T = v.T;
    ma.M = M;
    ma.RB = RB;
    ma.P = v.P;
    ma.max_pages = v.max_pages;
    ma.n_ctas = v.n_ctas;
    ma.scale_log2 = v.scale_log2;
    ma.mask_stride = v.mask_stride;
    ma.tree_in_cache = v.tree_in_cache;
    ma.k_pages = v.k_pages;
    ma.v_pages = v.v_pages;
    ma.block_table = v.block_table;
    ma.num_pages = v.num_pages;
    ma.status = v.status;
    ma.parents = v.parents;
    ma.parents_stride = v.parents_stride;
    ma.mask_out = v.mask_out;
    ma.tmode = v.tmode;
    ma.ovh = v.ovh;
    const Plan plan =
        make_plan(v.B, v.Hq, v.Hkv, v.T, v.P, v.max_pages, v.n_ctas, v.n_ctas, v.tmode);
    const long long units = plan.units;
    const int F = plan.F;
    ma.wpr = plan.merge_wpr;
    ma.rpw = plan.merge_rpw;
    const int rows = M < kRows ? M : kRows;
    const int rows_per_cta = kMergeWarps / ma.wpr * ma.rpw;
    const dim3 grid(static_cast<unsigned>(units), (rows + rows_per_cta - 1) / rows_per_cta);
    using K = void (*)(MergeArgs);
    const K table[3][3] = {
        {suffix_merge_kernel<D, 1, false, false>, suffix_merge_kernel<D, 2, false, false>,
         suffix_merge_kernel<D, 4, false, false>},
        {suffix_merge_kernel<D, 1, false, true>, suffix_merge_kernel<D, 2, false, true>,
         suffix_merge_kernel<D, 4, false, true>},
        {suffix_merge_kernel<D, 1, true, false>, suffix_merge_kernel<D, 2, true, false>,
         suffix_merge_kernel<D, 4, true, false>}};
    const int form = v.tmode == kTreeNone ? 2 : (ma.rpw > 1 ? 1 : 0);
    const K kernel = table[form][F == 4 ? 2 : (F == 2 ? 1 : 0)];
    return launch_pdl(kernel, grid, dim3(32 * kMergeWarps), 0, stream, ma);
}

// ===========================================================================
// Explicit mask of the one-pass form: row (b, t) over cache positions p:
// 1 for the committed prefix (p < L_b), bit p - L_b of the tree mask for the
// tree tokens padded after it, 0 beyond.  16 bytes per thread.
// ===========================================================================
__global__ void __launch_bounds__(256)
    dense_mask_kernel(const uint64_t* __restrict__ mask, int mask_stride,
                      const int32_t* __restrict__ seq_lens, int B, int T, int cols,
                      uint8_t* __restrict__ dense, int32_t* __restrict__ key_lens,
                      int32_t* __restrict__ status) {
    ptx::grid_dep_wait();    // then let the next kernel start: see tree_mask_kernel
    ptx::grid_dep_launch();
    const int row = blockIdx.x;  // b * T + t
    const int b = row / T, t = row % T;
    int L = seq_lens[b];
    const bool bad = L < 0 || static_cast<long long>(L) + T > cols;
    if (L < 0) L = 0;
    uint64_t bits = mask[static_cast<size_t>(b) * mask_stride + t];
    if (T < 64) bits &= (1ull << T) - 1ull;
    const long long p0 = (static_cast<long long>(blockIdx.y) * blockDim.x + threadIdx.x) * 16;
    if (p0 < cols) {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t v = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const long long p = p0 + 4 * q + k;
                uint32_t on = 0;
                if (p < L)
                    on = 1;
                else if (p - L < T)
                    on = static_cast<uint32_t>((bits >> (p - L)) & 1ull);
                v |= on << (8 * k);
            }
            w[q] = v;
        }
        *reinterpret_cast<uint4*>(dense + static_cast<size_t>(row) * cols + p0) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (t == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        key_lens[b] = L + T;
        if (bad) report(status, TREE_ATTN_STATUS_BAD_SEQ_LEN);
    }
}

#endif  // !TREE_ATTN_EARLY_TU

}  // namespace

#ifdef TREE_ATTN_EARLY_TU
// The early-start prefix kernels live in their own translation unit
// (prefix_early.cu includes this file), compiled beside this one.
cudaError_t launch_prefix_early(const VerifyArgs& a, const void* tmap_k, const void* tmap_v,
                                const void* tmap_tk, const void* tmap_tv, cudaStream_t stream) {
    if (a.d == 128)
        return launch_prefix_d<128, true>(a, tmap_k, tmap_v, tmap_tk, tmap_tv, stream);
    return launch_prefix_d<64, true>(a, tmap_k, tmap_v, tmap_tk, tmap_tv, stream);
}
#else
cudaError_t launch_dense_mask_build(const uint64_t* mask, int mask_stride,
                                    const int32_t* seq_lens, int B, int T, int dense_cols,
                                    uint8_t* dense, int32_t* key_lens, int32_t* status,
                                    cudaStream_t stream) {
    const unsigned per_cta = 256 * 16;
    const dim3 grid(static_cast<unsigned>(B) * T, (dense_cols + per_cta - 1) / per_cta);
    return launch_pdl(dense_mask_kernel, grid, dim3(256), 0, stream, mask, mask_stride, seq_lens,
                      B, T, dense_cols, dense, key_lens, status);
}

cudaError_t launch_mask_build(const int32_t* parents, int T, int n_trees, uint64_t* mask,
                              int32_t* status, cudaStream_t stream) {
    return launch_pdl(tree_mask_kernel, dim3(n_trees), dim3(32), 0, stream, parents, T, mask,
                      status);
}

cudaError_t launch_prefix(const VerifyArgs& a, const void* tmap_k, const void* tmap_v,
                          const void* tmap_tk, const void* tmap_tv, cudaStream_t stream) {
    if (a.early && a.dense == nullptr)
        return launch_prefix_early(a, tmap_k, tmap_v, tmap_tk, tmap_tv, stream);
    if (a.d == 128)
        return launch_prefix_d<128, false>(a, tmap_k, tmap_v, tmap_tk, tmap_tv, stream);
    return launch_prefix_d<64, false>(a, tmap_k, tmap_v, tmap_tk, tmap_tv, stream);
}

cudaError_t launch_merge(const VerifyArgs& a, cudaStream_t stream) {
    if (a.d == 128) return launch_merge_d<128>(a, stream);
    return launch_merge_d<64>(a, stream);
}

#endif  // TREE_ATTN_EARLY_TU

}  // namespace treeattn
