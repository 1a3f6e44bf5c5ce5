// Host-side check of the persistent kernel's work split and of the
// partial-sum bookkeeping of W2 column groups shared by several CTAs, using
// the very functions the kernel calls (awq_split.cuh). For every active
// expert count A, K-part count KP and grid size G the kernel accepts, it
// replays what each CTA publishes and what each CTA gathers, and checks that
// the two agree. Prints "ok <configurations>" and exits 0, or prints the
// first disagreement and exits 1.
#include <cstdio>
#include <vector>

#include "../awq_int4_moe_gb300/csrc/awq_split.cuh"

using namespace awq;

namespace {

constexpr int kGroupsW2 = 10;    // 256-column output groups of the hidden size 2560
constexpr int kMinGrid = 80, kMaxGridSize = 256, kMaxSegments = 256;

int fail(const char *what, int A, int KP, int G, int a, int b)
{
    std::printf("FAIL %s: A=%d KP=%d G=%d (%d, %d)\n", what, A, KP, G, a, b);
    return 1;
}

int check(int A, int KP, int G)
{
    const int per_c = A * KP, U = kGroupsW2 * per_c;
    // the shares tile the list
    if (range_start(0, U, G) != 0 || range_start(G, U, G) != U) return fail("share ends", A, KP, G, 0, 0);
    for (int b = 0; b < G; ++b) {
        const int n = range_start(b + 1, U, G) - range_start(b, U, G);
        if (n < 0 || n > (U + G - 1) / G) return fail("share size", A, KP, G, b, n);
    }
    for (int u = 0; u < U; ++u) {
        const int o = range_owner(u, U, G);
        if (o < 0 || o >= G || range_start(o, U, G) > u || range_start(o + 1, U, G) <= u)
            return fail("owner", A, KP, G, u, o);
    }
    // what every CTA publishes: (partial index, CTA) per shared group
    std::vector<std::vector<std::pair<int, int>>> pub(kGroupsW2);
    for (int b = 0; b < G; ++b) {
        const int r2b = range_start(b, U, G), r2e = range_start(b + 1, U, G);
        if (r2e == r2b) continue;
        const int cg_first = r2b / per_c, cg_last = (r2e - 1) / per_c;
        if (cg_last - cg_first + 1 > 2) return fail("groups per CTA", A, KP, G, b, cg_last - cg_first + 1);
        for (int cg = cg_first; cg <= cg_last; ++cg) {
            const int V0 = cg * per_c;
            const bool whole = V0 >= r2b && V0 + per_c <= r2e;
            const int slot = r2b >= V0 ? 0 : 1;
            if (!whole) pub[cg].push_back({b * 2 + slot, b});
        }
    }
    // what every part gathers
    for (int cg = 0; cg < kGroupsW2; ++cg) {
        const int V0 = cg * per_c;
        const std::vector<std::pair<int, int>> &p = pub[cg];
        if (p.empty()) continue;                  // written out whole by one CTA
        const int nparts = parts_count(V0, per_c, U, G);
        if (nparts != static_cast<int>(p.size())) return fail("part count", A, KP, G, cg, nparts);
        if (nparts > kMaxParts || nparts > 32) return fail("part bound", A, KP, G, cg, nparts);
        const int b_first = range_owner(V0, U, G);
        for (int q = 0; q < nparts; ++q) {
            if (part_index(V0, q, b_first, U, G) != p[q].first) return fail("part index", A, KP, G, cg, q);
            const int b = p[q].second;
            const int q_me = U < G ? range_start(b, U, G) - V0 : b - b_first;
            if (q_me != q) return fail("own part number", A, KP, G, cg, b);
        }
        // the column slices of the parts cover the group once
        int next = 0;
        for (int q = 0; q < nparts; ++q) {
            const int c0 = (q * 256) / nparts, c1 = ((q + 1) * 256) / nparts;
            if (c0 != next || c1 < c0) return fail("column slices", A, KP, G, cg, q);
            next = c1;
        }
        if (next != 256) return fail("column cover", A, KP, G, cg, next);
    }
    return 0;
}

}  // namespace

int main()
{
    long n = 0;
    for (int KP = 1; KP <= 4; KP *= 4)
        for (int A = 1; A <= kMaxSegments; ++A)
            for (int G = kMinGrid; G <= kMaxGridSize; ++G) {
                if (check(A, KP, G)) return 1;
                ++n;
            }
    std::printf("ok %ld\n", n);
    return 0;
}
