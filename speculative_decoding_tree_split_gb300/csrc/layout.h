// layout.h -- plain C++ helpers shared by the host code, the kernels and the
// CPU unit tests of this library (compiles with g++ or nvcc):
//   * tcgen05 shared-memory and instruction descriptors,
//   * the prefix-pass work partition (the "work line") and the slot index of
//     every partial result.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define TA_HD __host__ __device__ __forceinline__
#else
#define TA_HD inline
#endif

namespace treeattn {

// Prefix keys are processed in chunks of 64 tokens: one 128-byte swizzle atom
// of bf16 keys, the N of the S = Q.K^T MMA and the K of the P.V MMA.
constexpr int kChunk = 64;
// Query rows per CTA tile (the M of both MMAs, one TMEM lane per row).
constexpr int kRows = 128;

// ---------------------------------------------------------------------------
// tcgen05 descriptors
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle:
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-47  descriptor version (1 on sm_100-class tensor cores)
//   bits 49-51  base offset (0: every tile starts 1024-byte aligned)
//   bit  52     leading-dimension offset mode (0: relative)
//   bits 61-63  swizzle mode (2 = 128-byte swizzle)
// K-major operands: rows of 128 B (64 bf16 along K), 8-row groups SBO apart;
// LBO unused.  MN-major operands: 64 elements along M/N per 128-B row, LBO
// between such 64-element blocks, SBO between groups of 8 rows along K.
TA_HD uint64_t smem_desc_sw128(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    return static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4) |
           (static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32) |
           (static_cast<uint64_t>(1) << 46) | (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor for tcgen05.mma kind::f16 with bf16 A and B and an
// fp32 accumulator:
//   bits 4-5 D format (1 = f32), bits 7-9 A format (1 = bf16),
//   bits 10-12 B format (1 = bf16), bit 15 A major (1 = MN-major),
//   bit 16 B major (1 = MN-major), bits 17-22 N >> 3, bits 24-28 M >> 4.
TA_HD uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | ((static_cast<uint32_t>(N) >> 3) << 17) |
           ((static_cast<uint32_t>(M) >> 4) << 24);
}

// Byte offset of 16-byte chunk `c` (0..7) of row `r` inside a K-major
// 128-byte-swizzled tile whose rows are 128 B long (the layout TMA writes
// with CU_TENSOR_MAP_SWIZZLE_128B and the tensor core reads).
TA_HD uint32_t sw128_offset(uint32_t r, uint32_t c) {
    return (r >> 3) * 1024u + (r & 7u) * 128u + ((c ^ (r & 7u)) << 4);
}

// ---------------------------------------------------------------------------
// Work line of the prefix pass
// ---------------------------------------------------------------------------
// A "unit" is (sequence b, KV head hk, row block rb); units are numbered
// u = (b * Hkv + hk) * RB + rb.  Unit u owns chunks(b) = ceil(L_b / 64) steps
// of work.  Laying all units' steps end to end gives the work line of length
// W; CTA c of C takes the steps [start(c), start(c+1)), start(c) = c*W/C.
// The piece of unit u handled by CTA c is a "segment"; its partial result
// (m, l, acc) goes to slot u + c, which is unique because moving along the
// work line from one segment to the next increases u, c or both.  At most
// U + C - 1 slots are used.

// Committed prefix length actually used for sequence b: clamped to
// [0, max_pages*P]; `bad` is set when clamping was needed.
TA_HD int clamp_seq_len(int32_t L, int P, int max_pages, bool& bad) {
    const long long cap = static_cast<long long>(max_pages) * P;
    bad = false;
    if (L < 0) {
        bad = true;
        return 0;
    }
    if (L > cap) {
        bad = true;
        return static_cast<int>(cap);
    }
    return L;
}

TA_HD int chunks_of(int L) { return (L + kChunk - 1) / kChunk; }

// Where the draft-tree tokens sit on the work line:
//   kTreeNone     not at all: the prefix pass alone (the merge kernel then
//                 attends the tree tokens: the two-pass form);
//   kTreeChunk    one extra 64-key chunk after the unit's prefix chunks,
//                 loaded from the separate tree K/V buffers (token j in row j);
//   kTreeInCache  the tree tokens follow the prefix in the paged cache
//                 (positions L .. L+T-1), so the unit covers L + T positions.
// In both tree modes the prefix keys stay unmasked and the tree keys are
// masked per query row by the ancestor bits.
enum TreeMode : int { kTreeNone = 0, kTreeChunk = 1, kTreeInCache = 2 };

// Work-line steps of one unit of a sequence with L_raw committed tokens;
// `bad` is set when the lengths had to be clamped to the block table.
TA_HD int unit_chunks(int32_t L_raw, int P, int max_pages, int tmode, int T, bool& bad) {
    const int L = clamp_seq_len(L_raw, P, max_pages, bad);
    if (tmode == kTreeChunk) return chunks_of(L) + 1;
    if (tmode == kTreeInCache) {
        const long long cap = static_cast<long long>(max_pages) * P;
        long long e = static_cast<long long>(L) + T;
        if (e > cap) {
            bad = true;
            e = cap;
        }
        return chunks_of(static_cast<int>(e));
    }
    return chunks_of(L);
}

// n / d for n >= 0, d > 0.  When both fit in 32 bits (every realistic call)
// the quotient comes from one 32-bit unsigned division: on the GPU a 64-bit
// division is a long dependent instruction sequence, and these divisions sit
// on the path from kernel start to the first KV load.  Exact either way.
#if defined(__CUDACC__)
// Out of line on the GPU: one copy of the 64-bit division per kernel instead
// of one inlined at every call site (the inlined sequence is long, and code
// size is latency for kernels that run through their code once per launch).
static __host__ __device__ __noinline__ long long div_nn_wide(long long n, long long d) {
    return n / d;
}
#else
inline long long div_nn_wide(long long n, long long d) { return n / d; }
#endif

TA_HD long long div_nn(long long n, long long d) {
    if (((n | d) >> 32) == 0)
        return static_cast<long long>(static_cast<uint32_t>(n) / static_cast<uint32_t>(d));
    return div_nn_wide(n, d);
}

TA_HD long long cta_start(int c, long long W, int C) {
    return div_nn(static_cast<long long>(c) * W, C);
}

// The CTA whose range holds work-line position x (0 <= x < W).
TA_HD int cta_of(long long x, long long W, int C) {
    return static_cast<int>(div_nn(x * C + C - 1, W));
}

// True when CTA c has work (an empty range happens when W < C).  The merge
// side skips empty CTAs between a unit's first and last CTA: they wrote no
// partial.
TA_HD bool cta_has_work(int c, long long W, int C) {
    return cta_start(c, W, C) < cta_start(c + 1, W, C);
}

// Work-line length of a unit with nch chunks: the chunks, then `ovh` slots
// that stand for the fixed cost of a segment (pipeline restart, epilogue,
// partial store), so that a CTA whose range holds many short units gets
// fewer chunks.  A unit with no chunks takes no room.
TA_HD int unit_len(int nch, int ovh) { return nch > 0 ? nch + ovh : 0; }

struct Segment {
    int b, hk, rb, unit;
    int chunk_begin, chunk_end;  // chunk indices within sequence b
    int32_t len_raw;             // seq_lens[b] as read (not clamped)
};

// Walks the segments of one CTA's range in order.  `seq_lens` is read
// directly (device or host memory, depending on who runs it).
struct Walker {
    const int32_t* seq_lens;
    int B, P, max_pages, units_per_b, RB;
    int tmode, T;    // TreeMode and tree size
    int ovh;         // overhead slots per unit (see unit_len)
    int b;           // current sequence
    long long base;  // work-line position of sequence b's first unit
    int nch;         // chunks per unit of sequence b
    int len;         // work-line length per unit of sequence b
    int32_t lraw;    // seq_lens[b], read once per sequence
    long long x, x1; // current position and end of this CTA's range

    TA_HD int chunks_b(int bb) {
        bool bad;
        lraw = seq_lens[bb];
        return unit_chunks(lraw, P, max_pages, tmode, T, bad);
    }

    TA_HD void init(const int32_t* sl, int B_, int P_, int maxp, int upb, int RB_, int b0,
                    long long base0, long long x0, long long x1_, int tmode_ = kTreeNone,
                    int T_ = 0, int ovh_ = 0) {
        init_known(sl, B_, P_, maxp, upb, RB_, b0, base0, x0, x1_, tmode_, T_, ovh_,
                   (x0 < x1_) ? sl[b0] : 0);
    }

    // As init, with seq_lens[b0] already known (read by the caller's plan).
    TA_HD void init_known(const int32_t* sl, int B_, int P_, int maxp, int upb, int RB_, int b0,
                          long long base0, long long x0, long long x1_, int tmode_, int T_,
                          int ovh_, int32_t lraw_b0) {
        tmode = tmode_;
        T = T_;
        ovh = ovh_;
        seq_lens = sl;
        B = B_;
        P = P_;
        max_pages = maxp;
        units_per_b = upb;
        RB = RB_;
        b = b0;
        base = base0;
        x = x0;
        x1 = x1_;
        lraw = 0;
        nch = 0;
        if (x0 < x1_) {
            bool bad;
            lraw = lraw_b0;
            nch = unit_chunks(lraw_b0, P, max_pages, tmode, T, bad);
        }
        len = unit_len(nch, ovh);
    }

    TA_HD bool next(Segment& s) {
        while (x < x1) {
            while (x >= base + static_cast<long long>(units_per_b) * len) {
                base += static_cast<long long>(units_per_b) * len;
                ++b;
                nch = chunks_b(b);
                len = unit_len(nch, ovh);
            }
            const long long off = x - base;
            const int urel = static_cast<int>(div_nn(off, len));
            const int pos = static_cast<int>(off - static_cast<long long>(urel) * len);
            const long long ubase = base + static_cast<long long>(urel) * len;
            if (pos >= nch) {  // the unit's overhead slots: no chunks
                x = ubase + len;
                continue;
            }
            const long long cend = ubase + nch;
            const long long e = x1 < cend ? x1 : cend;
            s.b = b;
            s.hk = urel / RB;
            s.rb = urel % RB;
            s.unit = b * units_per_b + urel;
            s.chunk_begin = pos;
            s.chunk_end = pos + static_cast<int>(e - x);
            s.len_raw = lraw;
            x = e;
            return true;
        }
        return false;
    }
};

// Serial form of the per-CTA start search (host code and tests): total work
// W and, for CTA c, the sequence b0 holding start(c) and that sequence's
// work-line base.  The kernels compute the same values with warp scans.
inline void plan_serial(const int32_t* seq_lens, int B, int P, int max_pages, int upb, int C,
                        int c, long long& W, int& b0, long long& base0, long long& x0,
                        long long& x1, int tmode = kTreeNone, int T = 0, int ovh = 0) {
    long long tot = 0;
    for (int b = 0; b < B; ++b) {
        bool bad;
        tot += unit_len(unit_chunks(seq_lens[b], P, max_pages, tmode, T, bad), ovh);
    }
    W = tot * upb;
    x0 = cta_start(c, W, C);
    x1 = cta_start(c + 1, W, C);
    b0 = 0;
    base0 = 0;
    long long run = 0;
    for (int b = 0; b < B; ++b) {
        bool bad;
        const long long w = static_cast<long long>(upb) *
                            unit_len(unit_chunks(seq_lens[b], P, max_pages, tmode, T, bad), ovh);
        if (x0 < run + w) {
            b0 = b;
            base0 = run;
            return;
        }
        run += w;
    }
}

// Query-row replication in the prefix pass.  With few query rows per unit
// the 128-row tile holds F copies of them; copy g sits at tile rows
// [g*128/F, (g+1)*128/F) and handles keys [g*128/F, (g+1)*128/F) of every
// 128-key block, so all four softmax warps share the exponentials.  Each copy
// keeps its own (m, l, acc), stored in its own rows of the partial slot.
// Units with more than 128 query rows are split into row blocks (F = 1).
TA_HD int replicas_of(int M) { return M <= 32 ? 4 : (M <= 64 ? 2 : 1); }

// Partial-result slot layout: m[kRows] | l[kRows] | acc[kRows][d] (fp32).
TA_HD long long slot_floats(int d) { return 2LL * kRows + static_cast<long long>(kRows) * d; }

// The kernel selector: every launch choice of a call, from the shapes alone
// (the sequence lengths live on the device and are not read by the host).
// Split-count heuristics pick a number of KV splits that fills the SMs from
// the batch, head count and length (flash-decoding, Dao et al., cited by the
// pith.science verdict record); here the work line is cut into equal
// stretches for a persistent grid, so what remains to choose is:
//   n_ctas     one persistent CTA per SM, but never more CTAs than the
//              largest possible number of 64-token steps (small problems
//              would otherwise launch CTAs with nothing to do);
//   F          query-row copies per tile when one 128-row block holds the
//              unit's rows (small M: the softmax work per CTA is split);
//   tmode      whether the tree tokens ride on the prefix pass (small calls,
//              and calls with no more units than CTAs and two or more row
//              copies) or are attended by the merge kernel;
//   merge_wpr  warps per query row in the merge, from the partials a row
//              expects: prefix CTAs per unit, +1 for a straddled end, +F
//              for the unfolded copies of the last CTA;
//   merge_rpw  rows each merge warp takes in turn (merge without the tree
//              pass, when one row per warp would not fit the SMs at once).
struct Plan {
    int G, M, RB, units, F, n_ctas, merge_wpr;
    int merge_rpw;  // merge rows per warp, taken in turn
    int tmode;  // TreeMode chosen for the call
    int ovh;    // overhead slots per unit on the work line (unit_len)
    long long max_steps;
};

// Merge kernel: warps per CTA, and CTAs its register budget lets an SM hold.
constexpr int kMergeWarps = 4;
constexpr int kMergeResident = 6;

// Overhead slots per unit: a segment switch costs about as much as 2 + F*M/24
// 64-key steps (measured: the epilogue stores F*M rows of partials, then the
// pipeline restarts).
TA_HD int overhead_slots(int F, int M) {
    const int rows = F * (M < kRows ? M : kRows);
    const int o = 2 + rows / 24;
    return o > 8 ? 8 : o;
}

// Where the tree tokens go.  They ride on the prefix pass (one extra step per
// unit) when
//   * the call has at most kTreeInPrefixMaxSteps work-line steps per CTA: it
//     is latency-bound, and the merge's own tree pass sits on its critical
//     path; or
//   * there are no more units than CTAs and the tile holds at least two row
//     copies: the extra steps then cost at most one block per CTA, less than
//     the merge's tree pass over every query row.  (With one row copy the
//     tree-mode softmax spills registers; with more units than CTAs the extra
//     blocks outweigh the merge's work.  Measured on GB300: Llama-3.1-70B layer
//     73.1 -> 69.6 us with the tree on the prefix pass, the B=64 chain
//     360.5 -> 369.2 us and the Maverick layer 96.6 -> 105.1 us.)
// Otherwise the merge kernel attends them.
constexpr int kTreeInPrefixMaxSteps = 32;

// tree_layout: kTreeNone for the prefix pass alone (two-pass API), else where
// the call keeps the tree tokens (kTreeChunk: separate buffers; kTreeInCache:
// padded into the cache); the plan picks that mode or kTreeNone.
TA_HD Plan make_plan(int B, int Hq, int Hkv, int T, int P, int max_pages, int sm_count,
                     int n_ctas_req, int tree_layout = kTreeNone) {
    Plan p;
    p.G = Hq / Hkv;
    p.M = T * p.G;
    p.RB = (p.M + kRows - 1) / kRows;
    p.units = B * Hkv * p.RB;
    p.F = p.RB == 1 ? replicas_of(p.M) : 1;
    const long long prefix_steps =
        static_cast<long long>(p.units) *
        chunks_of(static_cast<int>(static_cast<long long>(max_pages) * P > (1LL << 30)
                                       ? (1LL << 30)
                                       : static_cast<long long>(max_pages) * P));
    auto ctas_for = [&](long long steps) -> int {
        if (n_ctas_req > 0) return n_ctas_req;
        const long long cap = steps > 0 ? steps : 1;
        return sm_count < cap ? sm_count : static_cast<int>(cap);
    };
    p.tmode = kTreeNone;
    const int C = ctas_for(prefix_steps + p.units);
    const bool small_call = prefix_steps <= static_cast<long long>(kTreeInPrefixMaxSteps) * C;
    const bool few_units = p.units <= C && p.F >= 2;
    if (tree_layout != kTreeNone && (small_call || few_units)) p.tmode = tree_layout;
    p.ovh = overhead_slots(p.F, p.M);
    p.max_steps = prefix_steps + (p.tmode == kTreeChunk ? p.units : 0);
    p.n_ctas = ctas_for(p.max_steps);
    const long long units = p.units > 0 ? p.units : 1;
    // Prefix CTAs fold their F row copies in their last segment, so a row
    // sees about one partial per CTA plus the F copies of a straddling CTA.
    const long long expect = p.n_ctas / units + 1 + p.F;
    p.merge_wpr = expect > 12 ? 4 : (expect > 6 ? 2 : 1);
    // Without a tree pass a merge warp's rows are cheap: give each warp
    // several, in turn, rather than launch more CTAs than the SMs hold at
    // once (kMergeResident per SM), whose later waves would wait for the
    // earlier ones.
    p.merge_rpw = 1;
    if (p.tmode != kTreeNone) {
        const long long rows = p.M < kRows ? p.M : kRows;
        const long long per_cta = kMergeWarps / p.merge_wpr;
        const long long ctas = units * ((rows + per_cta - 1) / per_cta);
        const long long cap = static_cast<long long>(sm_count) * kMergeResident;
        p.merge_rpw = static_cast<int>(cap > 0 ? (ctas + cap - 1) / cap : 1);
        if (p.merge_rpw < 1) p.merge_rpw = 1;
    }
    return p;
}

}  // namespace treeattn
