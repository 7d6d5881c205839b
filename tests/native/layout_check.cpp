// CPU check of the prefix-pass work partition in csrc/layout.h:
//   * the segments of all CTAs cover every (unit, chunk) exactly once, with
//     the tree tokens as one extra chunk per unit or as positions after the
//     prefix (the tree modes),
//   * partial-result slots (unit + cta) are unique and < units + CTAs,
//   * the merge side's slot range for a unit (cta_of of the unit's first and
//     last work-line positions) names exactly the CTAs that wrote it,
//   * with F query-row copies per tile, the partials the merge enumerates
//     (one folded partial per CTA before the unit's last CTA, then the last
//     CTA's one folded or F unfolded copies) are exactly those written: a
//     prefix CTA folds its copies in its last segment only,
//   * the descriptor helpers put each field where the bit layout says,
//   * the division helper matches plain 64-bit division on both of its
//     paths, and cta_of inverts cta_start on work lines longer than 2^32.
// Prints "OK" and exits 0, or prints the first failure and exits 1.
#include <cstdio>
#include <cstdlib>
#include <map>
#include <set>
#include <tuple>
#include <utility>
#include <vector>

#include "layout.h"

using namespace treeattn;

static unsigned long long rng_state = 12345;
static unsigned next_rand() {
    rng_state = rng_state * 6364136223846793005ULL + 1442695040888963407ULL;
    return static_cast<unsigned>(rng_state >> 33);
}

#define CHECK(cond, ...)                                     \
    do {                                                     \
        if (!(cond)) {                                       \
            std::printf("FAIL %s:%d: ", __FILE__, __LINE__); \
            std::printf(__VA_ARGS__);                        \
            std::printf("\n");                               \
            return false;                                    \
        }                                                    \
    } while (0)

static bool check_partition(int B, int Hkv, int RB, int P, int maxp, int C, int F, int tmode,
                            int T, int ovh, const std::vector<int32_t>& sl) {
    const int upb = Hkv * RB;
    std::set<std::tuple<int, int, int>> parts;  // (unit, CTA, copy) written
    std::map<std::pair<int, int>, int> covered;  // (unit, chunk) -> count
    std::map<int, std::set<int>> writers;        // unit -> CTAs
    std::set<long long> slots;
    long long W = 0;
    for (int c = 0; c < C; ++c) {
        int b0;
        long long base0, x0, x1;
        plan_serial(sl.data(), B, P, maxp, upb, C, c, W, b0, base0, x0, x1, tmode, T, ovh);
        Walker w;
        w.init(sl.data(), B, P, maxp, upb, RB, b0, base0, x0, x1, tmode, T, ovh);
        Segment s;
        long long done = 0;
        std::vector<Segment> segs;
        while (w.next(s)) {
            segs.push_back(s);
            CHECK(s.chunk_end > s.chunk_begin, "empty segment");
            CHECK(s.unit == (s.b * Hkv + s.hk) * RB + s.rb, "unit index");
            CHECK(s.len_raw == sl[s.b], "segment's cached sequence length");
            bool bad;
            const int nch = unit_chunks(sl[s.b], P, maxp, tmode, T, bad);
            CHECK(s.chunk_end <= nch, "segment past the sequence");
            for (int ch = s.chunk_begin; ch < s.chunk_end; ++ch)
                covered[std::make_pair(s.unit, ch)]++;
            CHECK(slots.insert(static_cast<long long>(s.unit) + c).second, "slot reused");
            CHECK(s.unit + c < B * upb + C, "slot out of range");
            writers[s.unit].insert(c);
            done += s.chunk_end - s.chunk_begin;
        }
        CHECK(done <= x1 - x0, "CTA walked past its range");
        for (size_t k = 0; k < segs.size(); ++k) {
            const bool fold = F > 1 && k + 1 == segs.size();
            for (int g = 0; g < (fold ? 1 : F); ++g)
                parts.insert(std::make_tuple(segs[k].unit, c, g));
        }
    }
    long long base = 0;
    for (int b = 0; b < B; ++b) {
        bool bad;
        const int nch = unit_chunks(sl[b], P, maxp, tmode, T, bad);
        for (int urel = 0; urel < upb; ++urel) {
            const int unit = b * upb + urel;
            for (int ch = 0; ch < nch; ++ch) {
                const int n = covered[std::make_pair(unit, ch)];
                CHECK(n == 1, "unit %d chunk %d covered %d times", unit, ch, n);
            }
            std::set<int> want;
            if (nch > 0) {
                const long long us =
                    base + static_cast<long long>(urel) * unit_len(nch, ovh);
                const int cf = cta_of(us, W, C), cl = cta_of(us + nch - 1, W, C);
                for (int c = cf; c <= cl; ++c)
                    if (cta_has_work(c, W, C)) want.insert(c);
            }
            CHECK(want == writers[unit], "merge-side CTA range mismatch for unit %d", unit);
            // the merge's enumeration of this unit's partials
            std::set<std::tuple<int, int, int>> got, have;
            for (const auto& t : parts)
                if (std::get<0>(t) == unit) have.insert(t);
            if (nch > 0) {
                const long long us =
                    base + static_cast<long long>(urel) * unit_len(nch, ovh);
                const int cf = cta_of(us, W, C), cl = cta_of(us + nch - 1, W, C);
                const bool last_folded =
                    F == 1 || cta_start(cl + 1, W, C) <= us + unit_len(nch, ovh);
                const int n1 = cl - cf;
                const int nv = n1 + (last_folded ? 1 : F);
                for (int v = 0; v < nv; ++v) {
                    const int cta = v < n1 ? cf + v : cl;
                    const int copy = v < n1 ? 0 : v - n1;
                    if (cta_has_work(cta, W, C)) got.insert(std::make_tuple(unit, cta, copy));
                }
            }
            CHECK(got == have, "merge-side partial list mismatch for unit %d (F=%d)", unit, F);
        }
        base += static_cast<long long>(upb) * unit_len(nch, ovh);
    }
    CHECK(base == W, "work-line length");
    return true;
}

static bool check_descriptors() {
    const uint64_t d = smem_desc_sw128(0x12340, 8192, 1024);
    CHECK((d & 0x3FFF) == (0x12340 >> 4), "start address field");
    CHECK(((d >> 16) & 0x3FFF) == 8192 / 16, "LBO field");
    CHECK(((d >> 32) & 0x3FFF) == 1024 / 16, "SBO field");
    CHECK(((d >> 46) & 0x3) == 1, "version field");
    CHECK(((d >> 49) & 0x7) == 0, "base offset field");
    CHECK(((d >> 61) & 0x7) == 2, "swizzle field");
    const uint32_t i = idesc_bf16_f32(128, 64, false, true);
    CHECK(((i >> 4) & 3) == 1 && ((i >> 7) & 7) == 1 && ((i >> 10) & 7) == 1, "formats");
    CHECK(((i >> 15) & 1) == 0 && ((i >> 16) & 1) == 1, "major bits");
    CHECK(((i >> 17) & 0x3F) == 64 / 8 && ((i >> 24) & 0x1F) == 128 / 16, "shape fields");
    // 128-byte swizzle: chunk c of row r lands at chunk c ^ (r % 8) of that row
    for (uint32_t r = 0; r < 16; ++r)
        for (uint32_t c = 0; c < 8; ++c) {
            const uint32_t off = sw128_offset(r, c);
            CHECK(off / 128 == r, "row of swizzled chunk");
            CHECK(((off % 128) / 16) == (c ^ (r % 8)), "swizzled chunk position");
        }
    return true;
}

static bool check_division() {
    for (int i = 0; i < 200000; ++i) {
        const unsigned long long hi = next_rand(), lo = next_rand();
        long long n = static_cast<long long>(((hi << 32) | lo) >> (next_rand() % 64));
        if (n < 0) n = -(n + 1);
        long long d = static_cast<long long>(next_rand() >> (next_rand() % 31)) + 1;
        if (i % 3 == 0) d = (d << (next_rand() % 32)) + 1;
        CHECK(div_nn(n, d) == n / d, "div_nn(%lld, %lld)", n, d);
    }
    // Work lines whose c * W or x * C leave 32 bits.
    for (int i = 0; i < 2000; ++i) {
        const int C = 1 + next_rand() % 300;
        const long long W =
            1 + ((static_cast<long long>(next_rand()) << (next_rand() % 24)) | next_rand());
        const int c = next_rand() % C;
        const long long a = cta_start(c, W, C), b = cta_start(c + 1, W, C);
        CHECK(a == static_cast<long long>(c) * W / C, "cta_start");
        if (a < b) {
            CHECK(cta_of(a, W, C) == c, "cta_of(start) W=%lld C=%d c=%d", W, C, c);
            CHECK(cta_of(b - 1, W, C) == c, "cta_of(end - 1) W=%lld C=%d c=%d", W, C, c);
        }
    }
    return true;
}

int main() {
    if (!check_descriptors()) return 1;
    if (!check_division()) return 1;
    const int Ps[4] = {16, 32, 64, 128};
    for (int trial = 0; trial < 400; ++trial) {
        const int B = 1 + next_rand() % 9;
        const int Hkv = 1 + next_rand() % 4;
        const int RB = 1 + next_rand() % 2;
        const int P = Ps[next_rand() % 4];
        const int maxp = 1 + next_rand() % 12;
        const int C = 1 + next_rand() % 40;
        std::vector<int32_t> sl(B);
        for (int b = 0; b < B; ++b) {
            const unsigned kind = next_rand() % 6;
            if (kind == 0)
                sl[b] = 0;
            else if (kind == 1)
                sl[b] = maxp * P;  // full
            else if (kind == 2)
                sl[b] = maxp * P + 5;  // too long: clamped
            else
                sl[b] = next_rand() % (maxp * P + 1);
        }
        const int T = 1 + next_rand() % 64;
        const int ovh = (trial % 3 == 0) ? 0 : next_rand() % 9;
        for (int tmode = kTreeNone; tmode <= kTreeInCache; ++tmode)
            for (int F = 1; F <= (RB == 1 ? 4 : 1); F *= 2) {
                if (!check_partition(B, Hkv, RB, P, maxp, C, F, tmode, T, ovh, sl)) {
                    std::printf("  at trial %d (B=%d Hkv=%d RB=%d P=%d maxp=%d C=%d F=%d tmode=%d "
                                "T=%d ovh=%d)\n",
                                trial, B, Hkv, RB, P, maxp, C, F, tmode, T, ovh);
                    return 1;
                }
            }
    }
    std::printf("OK\n");
    return 0;
}
