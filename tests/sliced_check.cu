// Host-side check of the sliced decode kernel's work split, using the very
// functions the kernel calls (awq_split.cuh). For every active-expert count A
// (A <= grid, the call's admission rule: A <= M * top_k <= grid), pieces per
// segment PJ (inter 160 and 640) and grid size G it checks, per CTA share:
//   - the share spans at most two segments (the kernel's two HW slots);
//   - the op walker emits every piece once, in order, and both W2 halves of
//     every group the share touches once, each after the group's last owned
//     piece plus the lag, and at most kMaxOps ops / kMaxGroups groups;
//   - each group's barrier count (owned pieces) equals the epilogue's
//     arrivals for it;
//   - the contributor rule (CTA c adds to token t when a segment of its share
//     is routed from t) lists exactly the CTAs that own a unit of t's segments.
// Prints "ok <configurations>" and exits 0, or the first failure and exits 1.
#include <cstdio>
#include <vector>

#include "../awq_int4_moe_gb300/csrc/awq_split.cuh"

using namespace awq;

namespace {

constexpr int kMaxOps = 192, kMaxGroups = 32;

int fail(const char *what, int PJ, int A, int G, int b)
{
    std::printf("FAIL %s: PJ=%d A=%d G=%d b=%d\n", what, PJ, A, G, b);
    return 1;
}

int check(int PJ, int A, int G)
{
    const int U = A * PJ;
    for (int b = 0; b < G; ++b) {
        const int r0 = range_start(b, U, G), r1 = range_start(b + 1, U, G);
        const int n13 = r1 - r0;
        if (n13 < 0) return fail("share size", PJ, A, G, b);
        if (n13 > 0 && (r1 - 1) / PJ - r0 / PJ > 1) return fail("segments per share", PJ, A, G, b);
        OpWalker w;
        w.init(r0, r1);
        int piece, gq, hh, next_piece = 0, nops = 0;
        std::vector<int> halves(U / 4 + 2, 0);
        int piece_group_last = -1;
        while (w.next(piece, gq, hh)) {
            ++nops;
            if (piece >= 0) {
                if (piece != next_piece++) return fail("piece order", PJ, A, G, b);
                piece_group_last = piece;
            } else {
                if (gq < r0 / 4 || gq > (r1 - 1) / 4) return fail("group outside share", PJ, A, G, b);
                if (hh != halves[gq]) return fail("half order", PJ, A, G, b);
                ++halves[gq];
                const int last = (4 * gq + 4 < r1 ? 4 * gq + 4 : r1) - 1 - r0;
                if (piece_group_last < last) return fail("W2 before its pieces", PJ, A, G, b);
                if (piece_group_last < n13 - 1 && last > piece_group_last - OpWalker::kLag)
                    return fail("lag", PJ, A, G, b);
            }
        }
        if (next_piece != n13) return fail("pieces missing", PJ, A, G, b);
        if (nops > kMaxOps) return fail("ops bound", PJ, A, G, b);
        if (n13 > 0) {
            const int q0 = r0 >> 2, nq = ((r1 - 1) >> 2) + 1 - q0;
            if (nq > kMaxGroups) return fail("groups bound", PJ, A, G, b);
            for (int q = q0; q < q0 + nq; ++q) {
                if (halves[q] != 2) return fail("halves", PJ, A, G, b);
                const int count = (4 * q + 4 < r1 ? 4 * q + 4 : r1) - (4 * q > r0 ? 4 * q : r0);
                int arrivals = 0;
                for (int u = r0; u < r1; ++u) arrivals += (u >> 2) == q;
                if (count != arrivals || count < 1) return fail("group barrier count", PJ, A, G, b);
            }
        }
    }
    // contributors: segment a's units are owned by CTAs range_owner(a PJ) ..
    // range_owner((a+1) PJ - 1); the kernel's rule looks from the CTA side
    for (int a = 0; a < A; ++a) {
        std::vector<char> by_units(G, 0), by_rule(G, 0);
        for (int u = a * PJ; u < (a + 1) * PJ; ++u) by_units[range_owner(u, U, G)] = 1;
        for (int c = 0; c < G; ++c) {
            const int lo = range_start(c, U, G), hi = range_start(c + 1, U, G);
            if (lo < hi && (lo / PJ == a || (hi - 1) / PJ == a)) by_rule[c] = 1;
        }
        if (by_units != by_rule) return fail("contributors", PJ, A, G, a);
    }
    return 0;
}

}  // namespace

int main()
{
    long n = 0;
    for (int PJ = 20; PJ <= 80; PJ *= 4)
        for (int G = 80; G <= 256; ++G)
            for (int A = 0; A <= 128 && A <= G; ++A) {
                if (check(PJ, A, G)) return 1;
                ++n;
            }
    std::printf("ok %ld\n", n);
    return 0;
}
