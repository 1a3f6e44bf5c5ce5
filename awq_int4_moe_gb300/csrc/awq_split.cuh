// Even split of a flat work list over the CTAs of a persistent grid, and the
// bookkeeping of the parts of a W2 column group that several CTAs share
// (which CTA publishes which partial block, who sums which columns). Host and
// device code alike, so that the arithmetic is checked on the CPU as well.
#pragma once

#include <cstdint>

namespace awq {

// Flat work lists hold at most 10 * 256 * 4 (W2) or 256 * 80 (W13) units
// and the grid is at most 256 CTAs, so every product below fits in 32 bits
// and the divisions are 32-bit unsigned ones.
__host__ __device__ __forceinline__ int range_start(int b, int U, int G)
{
    return static_cast<int>(static_cast<uint32_t>(b * U) / static_cast<uint32_t>(G));
}

// CTA whose share contains unit u (largest b with range_start(b) <= u).
__host__ __device__ __forceinline__ int range_owner(int u, int U, int G)
{
    return static_cast<int>(static_cast<uint32_t>((u + 1) * G - 1) / static_cast<uint32_t>(U));
}

// The parts of a piece [U0, U0 + len) of a list of U units split over G
// CTAs: the CTAs whose shares intersect it, in CTA order. A CTA publishes the
// partial of the first piece of its share in slot 0 and of its last in slot 1.
// With U >= G every CTA has at least one unit, so the parts are the CTAs
// range_owner(U0) .. range_owner(U0 + len - 1), and only the first of them
// can have started before U0. With U < G every CTA has at most one unit, so
// each unit of the piece is its own part, in slot 0.
__host__ __device__ __forceinline__ int parts_count(int U0, int len, int U, int G)
{
    if (U < G) return len;
    return range_owner(U0 + len - 1, U, G) - range_owner(U0, U, G) + 1;
}

// A W2 column group (a tenth of its list) meets at most min(units, G/10 + 2)
// <= 27 CTAs for G <= 256.
constexpr int kMaxParts = 28;

// Partial index (CTA * 2 + slot) of part q; b_first = range_owner(U0, U, G).
__host__ __device__ __forceinline__ int part_index(int U0, int q, int b_first, int U, int G)
{
    if (U < G) return range_owner(U0 + q, U, G) * 2;
    if (q > 0) return (b_first + q) * 2;
    return b_first * 2 + (range_start(b_first, U, G) < U0 ? 1 : 0);
}

// The op sequence of the sliced decode kernel for a share [r0, r1) of its
// unit list (units: segment x 8-column piece, PJ = inter / 8 per segment, a
// multiple of 4). W13 piece i (local index) in order, and after piece i the
// two W2 units (column halves) of every group whose last owned piece is at
// most i - kLag, so that the epilogue has finished those pieces; the rest at
// the end. Groups are 4-unit blocks: global group q covers units [4q, 4q+4).
// The producer and the consumer warps each walk the same sequence.
struct OpWalker {
    static constexpr int kLag = 2;
    int r0, r1, n13, q, q_end, done, pend;   // pieces emitted, second half pending
    __host__ __device__ __forceinline__ void init(int r0_, int r1_)
    {
        r0 = r0_;
        r1 = r1_;
        n13 = r1 - r0;
        q = r0 >> 2;
        q_end = n13 > 0 ? ((r1 - 1) >> 2) + 1 : q;
        done = 0;
        pend = 0;
    }
    // local index of the last owned piece of global group gq
    __host__ __device__ __forceinline__ int last_of(int gq) const
    {
        return (4 * gq + 4 < r1 ? 4 * gq + 4 : r1) - 1 - r0;
    }
    // Next op: false at the end. piece >= 0: W13 piece; else W2 unit (gq, hh).
    __host__ __device__ __forceinline__ bool next(int &piece, int &gq, int &hh)
    {
        if (pend) {
            pend = 0;
            piece = -1;
            gq = q - 1;
            hh = 1;
            return true;
        }
        if (q < q_end && (done >= n13 || last_of(q) <= done - 1 - kLag)) {
            piece = -1;
            gq = q++;
            hh = 0;
            pend = 1;
            return true;
        }
        if (done < n13) {
            piece = done++;
            return true;
        }
        return false;
    }
};

}  // namespace awq
