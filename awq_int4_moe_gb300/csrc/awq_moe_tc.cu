// Steps (a3) and (a4) for prefill-sized batches on the 5th-generation tensor
// cores: grouped W13 + SwiGLU and grouped W2 with tcgen05.mma, weights on the
// UMMA M side (128 rows = weight columns), a work item's token rows on N,
// fp32 accumulators in tensor memory.
//
// Source of the computation: 1Cat-vLLM #520 "Narrow Qwen3.8 AWQ active
// grouped decode", Purpose and Implementation (one launch per stage over all
// active-expert segments, scheduled from the device-side offsets) and Tests
// (the indexed prefill route for larger token counts); #522 "Operator
// results" (W13 + SwiGLU, W2 + weighted top-k reduction). Dequantisation is
// w = (q - zero) * scale as everywhere in the library, with exact products:
// the fp16 scale is split as s = s_hi + s_lo, s_hi keeping 6 of its 10
// stored mantissa bits, so that both (q - zero) * s_hi (at most 4 + 7
// significant bits) and (q - zero) * s_lo (at most 4 + 4) are exact fp16
// values; the A operand holds both, and the two MMAs on the same B rows
// accumulate (q - zero) * s * x exactly into fp32. (A single fp16 weight
// (q - zero) * s would carry a rounding of up to 2^-12 relative, which shows
// in sums that cancel.) |(q - zero) * s| must stay below the fp16 maximum,
// i.e. |s| < 4369. Likewise the activations h between the two GEMMs travel
// as fp16(h) plus the fp16 residue h - fp16(h) (about 22 significant bits):
// W2 multiplies both planes (the s_lo x residue product, below 2^-17 of the
// term, is left out). With h rounded to fp16 alone, large batches put rare
// outputs outside the stage's tolerance.
//
// Both GEMM kernels are persistent and warp-specialised: one CTA per
// multiprocessor walks its share of the units (work item x column tile,
// dealt round-robin), and the roles hand data to each other through
// mbarrier rings, so loads, dequantisation, MMAs and epilogues of different
// K blocks and units overlap:
//   warps 0-7  expand: packed int4 words -> the two fp16 A tiles (s_hi, s_lo
//              parts) of a K block, written straight into tensor memory
//              (tcgen05.st: row m in TMEM lane m, warp w reaches lanes
//              32 (w mod 4) ..; two fp16 of consecutive k per column), so the
//              A operand never passes through shared memory
//   warp 8     producer: TMA copies of the weights (W13: one 3D box of the 8
//              pieces' slices of a K block, and one of their records; W2:
//              bulk copies) and, in W13, cp.async gathers of the item's x rows
//              into the 128-byte-swizzled K-major B tile; in W2, TMA boxes of
//              h rows
//   warp 9     one thread issues the tcgen05.mma and commits
//   warps 10-13 epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//              lanes 32 (w mod 4) ..), the output math, global stores
// Work items: each active segment's rows (sorted-slot order) in chunks of at
// most 64 rows (W13, and W2 at I = 160; 16 for W2 at I = 640).
//
// w13_tc_kernel unit (item, column tile of 8 prepared pieces = 64 gate + 64
// up columns; UMMA row 16p + 8 half + col): 40 K blocks of 64. Epilogue: each
// gate lane pairs with its up lane (8 lanes apart) and stores h = silu(g) * u
// as fp16 in sorted-slot order (and, on the layer path, the residue plane).
// w2_tc_kernel unit (item, 5 output-column tiles of 128): the item's h rows
// of both planes (TMA, 3 boxes of 64 K per 160-row K part and plane) are
// loaded once per unit; per (column tile, K part) the producer bulk-copies
// the 4 x 20 packed lines and 20 record rows; per K block (64, 64, 32 rows of
// K) the MMA thread issues three MMAs per K16 (A_hi B_hi, A_lo B_hi, A_hi
// B_lo) into one of two accumulators; the epilogue writes y[slot][col] =
// router weight * D (fp32). combine_kernel then sums each token's k products
// in slot order and rounds to fp16 -- deterministic, no atomics.
#include <algorithm>

#include <cuda_fp16.h>

#include "awq_dequant.cuh"
#include "awq_launch.cuh"
#include "awq_moe_kernels.cuh"
#include "awq_ptx.cuh"
#include "awq_tc.cuh"

namespace awq {

namespace {

constexpr int kExpandWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kEpiWarp0 = 10;
constexpr int kTcThreads = 14 * 32;
static_assert(kEpiWarp0 + 4 == kTcThreads / 32, "four epilogue warps last (one per TMEM lane quarter)");
constexpr int kMaxUnits = 160;                          // units per CTA (table in shared memory)
constexpr int kKBlock = 64;

// A record's zero as the fp16 pair (1024 + z) and its scale split into the
// exact parts (s_hi, s_hi) and (s_lo, s_lo): s_hi clears the 4 low stored
// mantissa bits, s_lo = s - s_hi (exact: same exponent).
struct SplitRecord {
    uint32_t z2, shi, slo;
};

template <int MB>
__device__ __forceinline__ SplitRecord split_record(const uint8_t *rec)
{
    uint32_t w;
    if constexpr (MB == 4) {
        w = *reinterpret_cast<const uint32_t *>(rec);
    } else {
        w = static_cast<uint32_t>(rec[0]) | (static_cast<uint32_t>(rec[1]) << 8) | (static_cast<uint32_t>(rec[2]) << 16);
    }
    SplitRecord r;
    r.z2 = zero_pair_byte<2>(w);
    const uint32_t s2 = __byte_perm(w, w, 0x1010);
    r.shi = s2 & 0xFFF0FFF0u;
    r.slo = hsub2_u32(s2, r.shi);
    return r;
}

// The eight (q_i - z), i = 0..7 in K order, of one packed word (nibble i =
// k offset i), times s_hi (hi) and s_lo (lo): all sixteen fp16 products exact.
__device__ __forceinline__ void dequant_word_split(uint32_t w, const SplitRecord &m, uint4 &hi, uint4 &lo)
{
    const uint32_t z64 = zero_pair_64(m.z2);
    const uint32_t w8 = w >> 8;
    const uint32_t d0 = hsub2_u32(nib_lo_1024(w), m.z2);    // k 0, 4
    const uint32_t d1 = hsub2_u32(nib_hi_64(w), z64);       // k 1, 5
    const uint32_t d2 = hsub2_u32(nib_lo_1024(w8), m.z2);   // k 2, 6
    const uint32_t d3 = hsub2_u32(nib_hi_64(w8), z64);      // k 3, 7
    const uint32_t e0 = __byte_perm(d0, d1, 0x5410);        // k 0, 1
    const uint32_t e1 = __byte_perm(d2, d3, 0x5410);        // k 2, 3
    const uint32_t e2 = __byte_perm(d0, d1, 0x7632);        // k 4, 5
    const uint32_t e3 = __byte_perm(d2, d3, 0x7632);        // k 6, 7
    hi = make_uint4(hmul2_u32(e0, m.shi), hmul2_u32(e1, m.shi), hmul2_u32(e2, m.shi), hmul2_u32(e3, m.shi));
    lo = make_uint4(hmul2_u32(e0, m.slo), hmul2_u32(e1, m.slo), hmul2_u32(e2, m.slo), hmul2_u32(e3, m.slo));
}

// The eight (q_i - z), i = 0..7 in K order, of one packed word: exact fp16
// integers (the W2 of int4 banks at intermediate 160 applies the scale per
// group to its own accumulator).
__device__ __forceinline__ uint4 dequant_word_int(uint32_t w, uint32_t z2)
{
    const uint32_t z64 = zero_pair_64(z2);
    const uint32_t w8 = w >> 8;
    const uint32_t d0 = hsub2_u32(nib_lo_1024(w), z2);      // k 0, 4
    const uint32_t d1 = hsub2_u32(nib_hi_64(w), z64);       // k 1, 5
    const uint32_t d2 = hsub2_u32(nib_lo_1024(w8), z2);     // k 2, 6
    const uint32_t d3 = hsub2_u32(nib_hi_64(w8), z64);      // k 3, 7
    return make_uint4(__byte_perm(d0, d1, 0x5410), __byte_perm(d2, d3, 0x5410), __byte_perm(d0, d1, 0x7632),
                      __byte_perm(d2, d3, 0x7632));
}

// NVFP4 banks (2-byte records: the E4M3 scales of k 0..15 and k 16..31 of a
// group of 32): the scale pairs (s0, s0) and (s1, s1) as fp16. An E4M3 code
// placed in the fp16 bit fields (sign to bit 15, exponent and mantissa bits
// shifted up by 7) reads as its value times 2^-8 for normal and subnormal
// codes alike; times 256 is exact. (The NaN code is not a valid scale.)
__device__ __forceinline__ void nvfp4_scales(const uint8_t *rec, uint32_t &s0, uint32_t &s1)
{
    const uint32_t r = *reinterpret_cast<const uint16_t *>(rec);
    const uint32_t y = __byte_perm(r, 0u, 0x4140);                     // b0 in byte 0, b1 in byte 2
    const uint32_t raw = ((y & 0x007F007Fu) << 7) | ((y & 0x00800080u) << 8);
    const uint32_t v = hmul2_u32(raw, 0x5C005C00u);                    // x 256
    s0 = __byte_perm(v, v, 0x1010);
    s1 = __byte_perm(v, v, 0x3232);
}

// The eight E2M1 codes of a packed word (nibble i = k offset i) times the
// scale pair s2, as fp16 in K order (exact: at most 2 + 4 significant bits).
// A code's magnitude bits land in fp16 bits 9..11 and its sign in bit 15, which
// reads as the E2M1 value times 2^-14 (the zero-exponent code 1, 0.5, becomes
// the subnormal 2^-15); times 2^14 is exact. Pairs come out as (k_i, k_i+4).
__device__ __forceinline__ uint4 dequant_word_nvfp4(uint32_t w, uint32_t s2)
{
    const uint32_t r0 = ((w << 9) & 0x0E000E00u) | ((w << 12) & 0x80008000u);   // k 0, 4
    const uint32_t r1 = ((w << 5) & 0x0E000E00u) | ((w << 8) & 0x80008000u);    // k 1, 5
    const uint32_t r2 = ((w << 1) & 0x0E000E00u) | ((w << 4) & 0x80008000u);    // k 2, 6
    const uint32_t r3 = ((w >> 3) & 0x0E000E00u) | (w & 0x80008000u);           // k 3, 7
    const uint32_t d0 = hmul2_u32(hmul2_u32(r0, 0x74007400u), s2);
    const uint32_t d1 = hmul2_u32(hmul2_u32(r1, 0x74007400u), s2);
    const uint32_t d2 = hmul2_u32(hmul2_u32(r2, 0x74007400u), s2);
    const uint32_t d3 = hmul2_u32(hmul2_u32(r3, 0x74007400u), s2);
    return make_uint4(__byte_perm(d0, d1, 0x5410), __byte_perm(d2, d3, 0x5410), __byte_perm(d0, d1, 0x7632),
                      __byte_perm(d2, d3, 0x7632));
}

__device__ __forceinline__ int pow2_rows(int n) { return n <= 16 ? 16 : n <= 32 ? 32 : n <= 64 ? 64 : 128; }

// Bounded wait by every lane of a warp; true in all lanes only if all saw
// the phase complete.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t tmo)
{
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, tmo));
}

// Per-unit data every role derives from the unit table: expert, first sorted
// row, row count, column tile (or tile group).
struct UnitInfo {
    int e, row0, nrows, tile;
};

// Fill table[k] (segment, chunk, tile) -> (expert, row0, nrows, tile) for the
// CTA's units; expert -1 marks an id outside [0, E) (the unit is skipped by
// every role, the status is set once).
__device__ void resolve_units(int4 *table, int nu, int C, const StageArgs &args)
{
    for (int k = threadIdx.x; k < nu; k += blockDim.x) {
        const int4 t = table[k];
        const int a = t.x;
        int e = args.active_ids[a];
        const int o0 = args.offsets[a], o1 = args.offsets[a + 1];
        const int row0 = o0 + C * t.y;
        if (e < 0 || e >= args.num_experts) {
            set_status(args.status, AWQ_ERR_BAD_EXPERT_ID);
            e = -1;
        }
        table[k] = make_int4(e, row0, min(C, o1 - row0), t.z);
    }
}

__device__ __forceinline__ UnitInfo unit_at(const int4 *table, int k)
{
    const int4 t = table[k];
    return UnitInfo{t.x, t.y, t.z, t.w};
}

// ------------------------------------------------------------------ W13
constexpr int kStages13 = 10;
constexpr int kKps = kTcKbPerStage13;                    // K blocks per stage
constexpr int kKBlocks13 = kHidden / kKBlock;            // 40
constexpr int kPiecesPerTile = 8;
constexpr int kNA13 = 3;                                 // A buffers, one ring stage (kKps K blocks) each
constexpr int kQBlock = 2 * 4 * kPieceCols * 2 * 4;      // one piece's words of a K block: 512 B
constexpr int kW13Stage = kKps * (kPiecesPerTile * kQBlock + 1024);   // words + records (<= 32 * 4 per piece)
constexpr int kB13 = kTcRows13 * 128;                    // B tile of a K block
static_assert(kKBlocks13 % kKps == 0, "whole stages per unit");

// tensor memory: accumulators [0, 2 kTcRows13), A buffers from there, one per
// ring stage: 64 columns per K block (s_hi part, then s_lo part)
constexpr uint32_t kTmemCols13 = 512;
constexpr uint32_t kTmemA13 = 2 * kTcRows13;
static_assert(kTmemA13 + 64 * kTcKbPerStage13 * 3 <= kTmemCols13, "A buffers fit the allocation");

struct Lay13 {
    static constexpr int b = 0;                          // B tiles (1024-aligned)
    static constexpr int w = b + kStages13 * kKps * kB13;   // weight stages
    static constexpr int table = w + kStages13 * kW13Stage;
    static constexpr int tok = table + kMaxUnits * 16;
    static constexpr int bars = tok + kTcRows13 * 4;
    static constexpr int nbars = 2 * kStages13 + 2 * kNA13 + 4 + 1;
    static constexpr int misc = bars + nbars * 8;
    static constexpr int total = misc + 16 + 4 * 16;
};

int smem13() { return Lay13::total + 1024; }

}  // namespace

// grid = multiprocessors, kTcThreads threads
// tq13 / tm13: the prepared W13 bank as [piece][K block][512 B of words] /
// [piece][K block][32 mb bytes of records], boxes of 8 pieces x 1 K block.
template <int MB, int INTER>
__global__ void __launch_bounds__(kTcThreads, 1)
w13_tc_kernel(const __grid_constant__ CUtensorMap tq13, const __grid_constant__ CUtensorMap tm13, StageArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    constexpr int PJ = INTER / kPieceCols;
    constexpr int kTiles = (PJ + kPiecesPerTile - 1) / kPiecesPerTile;
    constexpr int kMBlock = 2 * 16 * MB;                  // one piece's records of a K block
    constexpr bool kNv = MB == 2;                         // NVFP4 banks: one exact A plane
    uint8_t *sb = smem + Lay13::b;
    uint8_t *sw = smem + Lay13::w;
    int4 *table = reinterpret_cast<int4 *>(smem + Lay13::table);
    int32_t *s_tok = reinterpret_cast<int32_t *>(smem + Lay13::tok);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lay13::bars);
    uint64_t *empty = full + kStages13;
    uint64_t *a_full = empty + kStages13;
    uint64_t *a_empty = a_full + kNA13;
    uint64_t *acc_full = a_empty + kNA13;                 // [2]
    uint64_t *acc_empty = acc_full + 2;                   // [2]
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Lay13::misc);
    int32_t *s_warp = reinterpret_cast<int32_t *>(smem + Lay13::misc + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t tmo = args.timeout_ns;

    if (tid == 0) {
        for (int s = 0; s < kStages13; ++s) {
            mbar_init(&full[s], 1 + 32);      // the copies' expect_tx arrival + every producer lane's gather
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < kNA13; ++b) {
            mbar_init(&a_full[b], kExpandWarps);
            mbar_init(&a_empty[b], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 0) tc_alloc(tmem_slot, kTmemCols13);
    if (tid == 0) {
        prefetch_tmap(&tq13);
        prefetch_tmap(&tm13);
    }
    grid_dependency_wait();
    if (tid == 0) trace_start(args.trace, 0);
    const int A = *args.num_active;
    const int nu = build_unit_table<kTcThreads>(A, args.offsets, kTcRows13, kTiles, gridDim.x, blockIdx.x, table,
                                                kMaxUnits, s_warp);
    resolve_units(table, nu, kTcRows13, args);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ---------------- producer: words, records, gathered x rows ----------------
        // Gather slots of this lane: 16-byte chunk c = lane mod 8 of rows
        // r_j = lane / 8 + 4 j, j < 8 (the item's <= 32 rows x 8 chunks of a
        // K block), addresses fixed for the whole unit.
        static_assert(kTcRows13 == 32, "eight gather slots per lane cover 32 rows");
        const int gc = lane & 7;
        int g = 0;
        bool alive = true;
        for (int k = 0; k < nu && alive; ++k) {
            const UnitInfo u = unit_at(table, k);
            if (u.e < 0) continue;
            for (int r = lane; r < u.nrows; r += 32) s_tok[r] = args.sorted_slots[u.row0 + r] / args.top_k;
            __syncwarp();
            const uint16_t *src[8];
            uint32_t dst[8];
            uint32_t valid = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int r = (lane >> 3) + 4 * j;
                const bool v = r < u.nrows;
                valid |= (v ? 1u : 0u) << j;
                src[j] = args.x + static_cast<int64_t>(v ? s_tok[r] : 0) * kHidden + gc * 8;
                dst[j] = sw128_offset(r, gc);
            }
            for (int kb = 0; kb < kKBlocks13; kb += kKps, ++g) {
                const int s = g % kStages13;
                if (g >= kStages13 && !warp_wait(&empty[s], ((g / kStages13) - 1) & 1, tmo)) {
                    if (lane == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                    alive = false;
                    break;
                }
                uint8_t *q = sw + s * kW13Stage;
                if (lane == 0) {
                    // the 8 pieces' slices of K blocks kb .. kb + kKps - 1 as
                    // [piece][K block][words] (pieces past the tile's last read
                    // as another expert's or as zero fill: their rows are never
                    // stored)
                    const int piece0 = u.e * PJ + kPiecesPerTile * u.tile;
                    mbar_arrive_expect_tx(&full[s], kKps * kPiecesPerTile * (kQBlock + kMBlock));
                    tma_load_3d(q, &tq13, &full[s], 0, kb, piece0);
                    tma_load_3d(q + kKps * kPiecesPerTile * kQBlock, &tm13, &full[s], 0, kb, piece0);
                }
                // the item's rows of K blocks kb .. kb + kKps - 1
                const uint32_t bs = smem_u32(sb + s * kKps * kB13);
#pragma unroll
                for (int sub = 0; sub < kKps; ++sub)
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (valid & (1u << j))
                            cp_async_16(bs + sub * kB13 + dst[j], src[j] + (kb + sub) * kKBlock);
                cp_async_arrive_noinc(&full[s]);
            }
            __syncwarp();
        }
        cp_async_wait_group<0>();
        // the MMAs' releases of the last stages arrive before the CTA exits
        // (a wait that runs out ends the drain: the consumers have stopped)
        if (lane == 0 && alive) {
            bool drained = true;
            for (int j = max(0, g - kStages13); j < g && drained; ++j)
                drained = mbar_wait_bounded(&empty[j % kStages13], (j / kStages13) & 1, tmo);
        }
    } else if (warp < kExpandWarps) {
        // ---------------- expand ----------------
        // thread = UMMA row m = 32 (warp mod 4) + lane = 16p + 8 half + c
        // (piece p, gate/up half, column c); warp / 4 = g2 picks the K half
        // (group 2 kb + g2). In the prepared piece, column c and half sit at
        // index ci = 2c + half of every 16 words / records: the thread's
        // record is 16 g2 + ci and its words t = 0..3 are 64 g2 + 16 t + ci;
        // word t covers k = 32 g2 + 8 t .. + 7 -> TMEM columns 16 g2 + 4 t .. + 3.
        const int quarter = warp & 3, g2 = warp >> 2;
        const int p = 2 * quarter + (lane >> 4);
        const int ci = 2 * (lane & 7) + ((lane >> 3) & 1);
        const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
        // A ring stage at a time: both K blocks' words are loaded and
        // expanded together (independent chains), then one wait for the
        // tensor-memory stores.
        int gs = 0;                                             // ring stages
        bool alive = true;
        for (int k = 0; k < nu && alive; ++k) {
            const UnitInfo u = unit_at(table, k);
            if (u.e < 0) continue;
            for (int kb = 0; kb < kKBlocks13; kb += kKps, ++gs) {
                const int s = gs % kStages13, ab = gs % kNA13;
                bool good = mbar_wait_bounded(&full[s], (gs / kStages13) & 1, tmo);
                if (good && gs >= kNA13) good = mbar_wait_bounded(&a_empty[ab], ((gs / kNA13) - 1) & 1, tmo);
                if (!__all_sync(0xffffffffu, good)) {
                    if (lane == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                    alive = false;
                    break;
                }
                tc_fence_after();
                // words [piece][sub][128], then records [piece][sub][32 MB]
                const uint8_t *q = sw + s * kW13Stage + p * kKps * kQBlock + (64 * g2 + ci) * 4;
                const uint8_t *rec_at = sw + s * kW13Stage + kKps * kPiecesPerTile * kQBlock + p * kKps * kMBlock +
                                        (16 * g2 + ci) * MB;
                const uint32_t at = tmem + lane_base + kTmemA13 + 64 * kKps * ab + 16 * g2;
                uint32_t w[kKps][4];
#pragma unroll
                for (int sub = 0; sub < kKps; ++sub)
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        w[sub][t] = *reinterpret_cast<const uint32_t *>(q + sub * kQBlock + 16 * t * 4);
#pragma unroll
                for (int sub = 0; sub < kKps; ++sub) {
                    if constexpr (kNv) {
                        uint32_t s0, s1, rh[16];
                        nvfp4_scales(rec_at + sub * kMBlock, s0, s1);
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const uint4 v = dequant_word_nvfp4(w[sub][t], t < 2 ? s0 : s1);   // words 0, 1: k 0..15
                            rh[4 * t] = v.x, rh[4 * t + 1] = v.y, rh[4 * t + 2] = v.z, rh[4 * t + 3] = v.w;
                        }
                        tc_st16(at + 64 * sub, rh);
                    } else {
                        const SplitRecord rec = split_record<MB>(rec_at + sub * kMBlock);
                        uint32_t rh[16], rl[16];
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            uint4 hi, lo;
                            dequant_word_split(w[sub][t], rec, hi, lo);
                            rh[4 * t] = hi.x, rh[4 * t + 1] = hi.y, rh[4 * t + 2] = hi.z, rh[4 * t + 3] = hi.w;
                            rl[4 * t] = lo.x, rl[4 * t + 1] = lo.y, rl[4 * t + 2] = lo.z, rl[4 * t + 3] = lo.w;
                        }
                        tc_st16(at + 64 * sub, rh);
                        tc_st16(at + 64 * sub + 32, rl);
                    }
                }
                tc_wait_st();                                   // the stage's K blocks are in TMEM
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[ab]);
            }
        }
        // the MMAs' releases of the last A buffers arrive before the CTA exits
        const int stages_done = gs;
        if (lane == 0 && alive)
            for (int j = max(0, stages_done - kNA13); j < stages_done; ++j)
                if (!mbar_wait_bounded(&a_empty[j % kNA13], (j / kNA13) & 1, tmo)) break;
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issue (one thread) ----------------
        if (lane == 0) {
            int g = 0, ui = 0;
            bool issued = false;
            for (int k = 0; k < nu; ++k) {
                const UnitInfo u = unit_at(table, k);
                if (u.e < 0) continue;
                const int buf = ui & 1;
                if (ui >= 2 && !mbar_wait_bounded(&acc_empty[buf], ((ui >> 1) - 1) & 1, tmo)) {
                    set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                    break;
                }
                tc_fence_after();
                const uint32_t idesc = umma_idesc_f16(128, pow2_rows(u.nrows));
                const uint32_t dt = tmem + static_cast<uint32_t>(buf * kTcRows13);
                bool ok = true;
                for (int kb = 0; kb < kKBlocks13; kb += kKps, ++g) {      // g: ring stages
                    const int s = g % kStages13, ab = g % kNA13;
                    if (!mbar_wait_bounded(&a_full[ab], (g / kNA13) & 1, tmo) ||
                        !mbar_wait_bounded(&full[s], (g / kStages13) & 1, tmo)) {
                        ok = false;
                        break;
                    }
                    // the gathered x rows were written through the generic proxy
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    tc_fence_after();
#pragma unroll
                    for (int sub = 0; sub < kKps; ++sub) {
                        const uint32_t a0 = tmem + kTmemA13 + 64 * (kKps * ab + sub);
                        const uint32_t b0 = smem_u32(sb + (s * kKps + sub) * kB13);
#pragma unroll
                        for (int kk = 0; kk < kKBlock / 16; ++kk) {
                            const uint64_t bd = umma_desc_sw128(b0 + 32 * kk);
                            tc_mma_f16_tmem_a(dt, a0 + 8 * kk, bd, idesc, (kb + sub > 0 || kk > 0) ? 1u : 0u);
                            if constexpr (!kNv) tc_mma_f16_tmem_a(dt, a0 + 32 + 8 * kk, bd, idesc, 1u);
                        }
                    }
                    tc_commit(&empty[s]);
                    tc_commit(&a_empty[ab]);
                    issued = true;
                }
                if (!ok) {
                    set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                    break;
                }
                tc_commit(&acc_full[buf]);
                ++ui;
            }
            // every MMA issued here has completed before TMEM is freed
            if (issued) {
                tc_commit(drain);
                mbar_wait_bounded(drain, 0, tmo);
            }
        }
    } else {
        // ---------------- epilogue: TMEM -> SwiGLU -> h ----------------
        const int quarter = warp & 3;
        const int r = 32 * quarter + lane;                 // UMMA row of this lane
        const int p = r >> 4, hr = (r >> 3) & 1, cc = r & 7;
        int ui = 0;
        for (int k = 0; k < nu; ++k) {
            const UnitInfo u = unit_at(table, k);
            if (u.e < 0) continue;
            const int buf = ui & 1;
            if (!warp_wait(&acc_full[buf], (ui >> 1) & 1, tmo)) {
                if (lane == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                break;
            }
            tc_fence_after();
            const int np = min(kPiecesPerTile, PJ - kPiecesPerTile * u.tile);
            const int col = kPieceCols * (kPiecesPerTile * u.tile + p) + cc;
            const int nb = pow2_rows(u.nrows);
            const float gs = MB == 2 ? args.global_scale[2 * u.e] : 1.0f;   // NVFP4 W13 global
            for (int n0 = 0; n0 < nb; n0 += 16) {
                uint32_t v[16];
                tc_ld16(tmem + (static_cast<uint32_t>(32 * quarter) << 16) + static_cast<uint32_t>(buf * kTcRows13 + n0),
                        v);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float mine = __uint_as_float(v[j]) * gs;
                    const float other = __shfl_xor_sync(0xffffffffu, mine, 8);   // up of a gate row
                    const int n = n0 + j;
                    if (hr == 0 && p < np && n < u.nrows) {
                        const float hv = silu_f(mine) * other;
                        const uint16_t hi = f2h_bits(hv);
                        const int64_t at = static_cast<int64_t>(u.row0 + n) * INTER + col;
                        args.h_out[at] = hi;
                        if (args.h_lo) args.h_lo[at] = f2h_bits(hv - __half2float(__ushort_as_half(hi)));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
            ++ui;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tc_dealloc(tmem, kTmemCols13);
    if (tid == 0) trace_end(args.trace, 0);
}

// ------------------------------------------------------------------ W2
namespace {

constexpr int kStages2 = 4;
constexpr int kTilesPerUnit2 = 5;                        // 128-column output tiles per unit (large batches)
static_assert(kHidden / 128 % kTilesPerUnit2 == 0, "whole units per work item");
constexpr int kNA2 = 2;
constexpr int kQUnit2 = 4 * kW2TileKK * 128;             // 4 x 20 lines: 10240 B
constexpr int kW2Stage = kQUnit2 + 4 * 5 * 32 * 4;       // + 20 record rows (<= 4-byte records)
constexpr int kBUnit2 = 3 * 2 * 64 * 128;                // h boxes of a unit: KP x 3 x 2 planes x rows x 128 B

// Two schemes. Split scale (intermediate 640; NVFP4 with its exact single
// plane): A = (q - z) s split into exact s_hi and s_lo planes, one
// accumulator per output tile. Per group (int4 banks at intermediate 160):
// A = (q - z), an exact single plane, and one accumulator per 32-k group of
// the 160-k part, so the scale of each (group, column) multiplies the
// group's fp32 sum in the epilogue -- half the MMAs of the split scale
// (one per K16 instead of two). Work items are then at most 16 rows, so the
// five group accumulators of both buffers fit in tensor memory.
__host__ __device__ constexpr bool w2_per_group(int inter, int mb) { return mb != 2 && inter == 160; }
__host__ __device__ constexpr int w2_rows(int inter, int mb) { return w2_per_group(inter, mb) ? 16 : tc_rows2(inter); }

// tensor memory, split scale: two accumulators of 2 C2 columns in [0, 4 C2)
// (the products with the item's fp16(h) rows, then with its residue rows:
// the two h planes are one B operand of 2 nb rows), A buffers from 256 (64
// columns each: s_hi part, then s_lo part). Per group: two accumulators of
// 5 groups x 32 columns (16 fp16(h) rows, 16 residue rows) in [0, 320), A
// buffers of a whole 160-k tile (80 columns) from 320, so the MMA thread
// waits and commits once per tile.
constexpr uint32_t kTmemCols2 = 512;
constexpr uint32_t kTmemA2 = 256;
static_assert(4 * tc_rows2(160) <= kTmemA2 && 4 * tc_rows2(640) <= kTmemA2, "accumulators below the A buffers");
static_assert(kTmemA2 + kNA2 * 64 <= kTmemCols2, "A buffers fit the allocation");
constexpr uint32_t kGrpAcc2 = 5 * 32;                   // per-group scheme: one accumulator buffer
constexpr uint32_t kGrpA2 = 2 * kGrpAcc2;               // its A buffers (one 160-k tile each)
static_assert(kGrpA2 + kNA2 * 80 <= kTmemCols2, "per-group accumulators and A buffers fit the allocation");

struct Lay2 {
    static constexpr int b = 0;                          // 2 unit buffers of h boxes (1024-aligned)
    static constexpr int w = b + 2 * kBUnit2;
    static constexpr int table = w + kStages2 * kW2Stage;
    static constexpr int bars = table + kMaxUnits * 16;
    static constexpr int nbars = 2 * kStages2 + 2 * 2 + 2 * kNA2 + 4 + 1;
    static constexpr int misc = bars + nbars * 8;
    static constexpr int total = misc + 16 + 4 * 16;
};

int smem2() { return Lay2::total + 1024; }

}  // namespace

// grid = multiprocessors, kTcThreads threads
// TPU: 128-column output tiles per unit (5, or 1 when there are too few
// units of 5 to occupy the grid: small batches).
template <int MB, int INTER, int TPU>
__global__ void __launch_bounds__(kTcThreads, 1)
w2_tc_kernel(const __grid_constant__ CUtensorMap th16, const __grid_constant__ CUtensorMap th32,
             const __grid_constant__ CUtensorMap th64, const __grid_constant__ CUtensorMap th128, StageArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    constexpr int KP = INTER / 160;
    constexpr int kUnits = kHidden / 128 / TPU;           // units per work item
    constexpr bool kGrp = w2_per_group(INTER, MB);        // per-group accumulators (else split scale)
    constexpr int C2 = w2_rows(INTER, MB);
    constexpr int kMUnit = 4 * 5 * 32 * MB;
    constexpr bool kNv = MB == 2;                         // NVFP4 banks: one exact A plane
    // one A buffer per whole 160-k tile (one MMA-thread wait and two commits
    // per tile): the per-group scheme and NVFP4 banks (one exact plane) at
    // intermediate 160; per K block otherwise
    constexpr bool kTileA = INTER == 160 && (kGrp || kNv);
    constexpr uint32_t kAccStride = kGrp ? kGrpAcc2 : 2 * C2;   // TMEM columns of one accumulator buffer
    constexpr uint32_t kAOff = kGrp ? kGrpA2 : kTmemA2;         // first A buffer
    constexpr uint32_t kAStride = kTileA ? 80 : 64;             // TMEM columns of one A buffer
    static_assert(kAOff + kNA2 * kAStride <= kTmemCols2, "A buffers fit the allocation");
    uint8_t *sbh = smem + Lay2::b;
    uint8_t *sw = smem + Lay2::w;
    int4 *table = reinterpret_cast<int4 *>(smem + Lay2::table);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lay2::bars);
    uint64_t *empty = full + kStages2;
    uint64_t *b_full = empty + kStages2;                  // [2] unit buffers of h boxes
    uint64_t *b_empty = b_full + 2;
    uint64_t *a_full = b_empty + 2;
    uint64_t *a_empty = a_full + kNA2;
    uint64_t *acc_full = a_empty + kNA2;                  // [2]
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Lay2::misc);
    int32_t *s_warp = reinterpret_cast<int32_t *>(smem + Lay2::misc + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t tmo = args.timeout_ns;

    if (tid == 0) {
        for (int s = 0; s < kStages2; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&b_full[b], 1);
            mbar_init(&b_empty[b], 1);
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        for (int b = 0; b < kNA2; ++b) {
            mbar_init(&a_full[b], kExpandWarps);
            mbar_init(&a_empty[b], 1);
        }
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 0) tc_alloc(tmem_slot, kTmemCols2);
    grid_dependency_wait();
    if (tid == 0) trace_start(args.trace, 1);
    const int A = *args.num_active;
    const int S = args.M * args.top_k;
    const int nu = build_unit_table<kTcThreads>(A, args.offsets, C2, kUnits, gridDim.x, blockIdx.x, table,
                                                kMaxUnits, s_warp);
    resolve_units(table, nu, C2, args);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            // ---------------- producer: h boxes per unit, weights per (tile, K part) ----------------
            int gw = 0, ui = 0;
            bool alive = true;
            for (int k = 0; k < nu && alive; ++k) {
                const UnitInfo u = unit_at(table, k);
                if (u.e < 0) continue;
                const int nb = pow2_rows(u.nrows), bbox = nb * 128, ub = ui & 1;
                const CUtensorMap *th = nb == 16 ? &th16 : nb == 32 ? &th32 : nb == 64 ? &th64 : &th128;
                if (ui >= 2 && !mbar_wait_bounded(&b_empty[ub], ((ui >> 1) - 1) & 1, tmo)) {
                    set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                    break;
                }
                // box (kp, kbl, plane): plane 0 = fp16(h) rows, plane 1 = residue rows (S below)
                mbar_arrive_expect_tx(&b_full[ub], KP * 3 * 2 * bbox);
                for (int kp = 0; kp < KP; ++kp)
                    for (int b = 0; b < 3; ++b)
                        for (int pl = 0; pl < 2; ++pl)
                            tma_load_2d(sbh + ub * kBUnit2 + ((kp * 3 + b) * 2 + pl) * bbox, th, &b_full[ub],
                                        160 * kp + 64 * b, pl * S + u.row0);
                for (int wu = 0; wu < TPU * KP; ++wu, ++gw) {
                    const int s = gw % kStages2;
                    if (gw >= kStages2 && !mbar_wait_bounded(&empty[s], ((gw / kStages2) - 1) & 1, tmo)) {
                        set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                        alive = false;
                        break;
                    }
                    const int ct = u.tile * TPU + wu / KP, kp = wu % KP;
                    // 4 consecutive 32-column tiles of (e, kp): 80 lines, 20 record rows
                    const int64_t tile0 = (static_cast<int64_t>(u.e) * KP + kp) * kColTiles + 4 * ct;
                    uint8_t *q = sw + s * kW2Stage;
                    mbar_arrive_expect_tx(&full[s], kQUnit2 + kMUnit);
                    bulk_load(q, reinterpret_cast<const uint8_t *>(args.w2_q) + tile0 * kW2TileKK * 128, kQUnit2,
                              &full[s]);
                    bulk_load(q + kQUnit2, args.w2_meta + tile0 * 5 * 32 * MB, kMUnit, &full[s]);
                }
                ++ui;
            }
            // the last units' boxes and the MMAs' releases of the last stages
            // arrive before the CTA exits (a wait that runs out ends the drain)
            bool drained = alive;
            for (int j = max(0, ui - 2); j < ui && drained; ++j)
                drained = mbar_wait_bounded(&b_empty[j & 1], (j >> 1) & 1, tmo);
            for (int j = max(0, gw - kStages2); j < gw && drained; ++j)
                drained = mbar_wait_bounded(&empty[j % kStages2], (j / kStages2) & 1, tmo);
        }
    } else if (warp < kExpandWarps) {
        // ---------------- expand ----------------
        // thread: output column m = tid mod 128 of the tile (UMMA row, TMEM
        // lane; warp mod 4 = m / 32); in K block kbl of a part, the packed
        // rows r = 8 kbl + 4 rh + i, i < 4 (rh = tid / 128), which share the
        // record of group 2 kbl + rh; row r covers TMEM columns 16 rh + 4 i ..
        const int m = tid & 127, rh = tid >> 7;
        const int t4 = m >> 5, c32 = m & 31;
        const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        int gk = 0, gw = 0;
        bool alive = true;
        for (int k = 0; k < nu && alive; ++k) {
            const UnitInfo u = unit_at(table, k);
            if (u.e < 0) continue;
            for (int wu = 0; wu < TPU * KP && alive; ++wu, ++gw) {
                const int s = gw % kStages2;
                if constexpr (kTileA) {
                    // the whole 160-k tile into one A buffer: this thread's groups
                    // rh, rh + 2 (, 4), group g at TMEM columns 16 g ..
                    const int ab = gk % kNA2;
                    bool good = mbar_wait_bounded(&full[s], (gw / kStages2) & 1, tmo);
                    if (good && gk >= kNA2) good = mbar_wait_bounded(&a_empty[ab], ((gk / kNA2) - 1) & 1, tmo);
                    if (!__all_sync(0xffffffffu, good)) {
                        if (lane == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                        alive = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t *q = sw + s * kW2Stage;
#pragma unroll
                    for (int gi = 0; gi < 3; ++gi) {
                        const int grp = rh + 2 * gi;
                        if (grp < 5) {                             // (warp-uniform)
                            const uint8_t *rec_at = q + kQUnit2 + (t4 * 5 + grp) * 32 * MB + c32 * MB;
                            uint32_t rq[16];
                            if constexpr (kNv) {
                                // e2m1 x e4m3 of the word's 16-k block: exact
                                uint32_t s0, s1;
                                nvfp4_scales(rec_at, s0, s1);
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const int r = 4 * grp + i;
                                    const uint4 v = dequant_word_nvfp4(
                                        *reinterpret_cast<const uint32_t *>(q + (t4 * kW2TileKK + r) * 128 + c32 * 4),
                                        i < 2 ? s0 : s1);
                                    rq[4 * i] = v.x, rq[4 * i + 1] = v.y, rq[4 * i + 2] = v.z, rq[4 * i + 3] = v.w;
                                }
                            } else {
                                uint32_t w;
                                if constexpr (MB == 4) {
                                    w = *reinterpret_cast<const uint32_t *>(rec_at);
                                } else {
                                    w = static_cast<uint32_t>(rec_at[0]) | (static_cast<uint32_t>(rec_at[1]) << 8) |
                                        (static_cast<uint32_t>(rec_at[2]) << 16);
                                }
                                const uint32_t z2 = zero_pair_byte<2>(w);
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const int r = 4 * grp + i;
                                    const uint4 v = dequant_word_int(
                                        *reinterpret_cast<const uint32_t *>(q + (t4 * kW2TileKK + r) * 128 + c32 * 4),
                                        z2);
                                    rq[4 * i] = v.x, rq[4 * i + 1] = v.y, rq[4 * i + 2] = v.z, rq[4 * i + 3] = v.w;
                                }
                            }
                            tc_st16(tmem + lane_base + kAOff + kAStride * ab + 16 * grp, rq);
                        }
                    }
                    tc_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&a_full[ab]);
                    ++gk;
                } else {
                for (int kbl = 0; kbl < 3; ++kbl, ++gk) {
                    const int ab = gk % kNA2;
                    bool good = true;
                    if (kbl == 0) good = mbar_wait_bounded(&full[s], (gw / kStages2) & 1, tmo);
                    if (good && gk >= kNA2) good = mbar_wait_bounded(&a_empty[ab], ((gk / kNA2) - 1) & 1, tmo);
                    if (!__all_sync(0xffffffffu, good)) {
                        if (lane == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                        alive = false;
                        break;
                    }
                    tc_fence_after();
                    const int grp = 2 * kbl + rh;                  // group of this thread's rows
                    if (grp < 5) {                                 // (warp-uniform: rh = warp / 4)
                        const uint8_t *q = sw + s * kW2Stage;
                        const uint8_t *rec_at = q + kQUnit2 + (t4 * 5 + grp) * 32 * MB + c32 * MB;
                        const uint32_t at = tmem + lane_base + kAOff + kAStride * ab + 16 * rh;
                        if constexpr (kNv) {
                            uint32_t s0, s1, rhi[16];
                            nvfp4_scales(rec_at, s0, s1);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int r = 4 * grp + i;
                                const uint32_t w =
                                    *reinterpret_cast<const uint32_t *>(q + (t4 * kW2TileKK + r) * 128 + c32 * 4);
                                const uint4 v = dequant_word_nvfp4(w, i < 2 ? s0 : s1);   // rows 0, 1: k 0..15
                                rhi[4 * i] = v.x, rhi[4 * i + 1] = v.y, rhi[4 * i + 2] = v.z, rhi[4 * i + 3] = v.w;
                            }
                            tc_st16(at, rhi);
                        } else {
                            const SplitRecord rec = split_record<MB>(rec_at);
                            uint32_t rhi[16], rlo[16];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int r = 4 * grp + i;
                                const uint32_t w =
                                    *reinterpret_cast<const uint32_t *>(q + (t4 * kW2TileKK + r) * 128 + c32 * 4);
                                uint4 hi, lo;
                                dequant_word_split(w, rec, hi, lo);
                                rhi[4 * i] = hi.x, rhi[4 * i + 1] = hi.y, rhi[4 * i + 2] = hi.z, rhi[4 * i + 3] = hi.w;
                                rlo[4 * i] = lo.x, rlo[4 * i + 1] = lo.y, rlo[4 * i + 2] = lo.z, rlo[4 * i + 3] = lo.w;
                            }
                            tc_st16(at, rhi);
                            tc_st16(at + 32, rlo);
                        }
                        tc_wait_st();
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&a_full[ab]);
                }
                }   // per K block
            }
        }
        // the MMAs' releases of the last A buffers arrive before the CTA exits
        if (lane == 0 && alive)
            for (int j = max(0, gk - kNA2); j < gk; ++j)
                if (!mbar_wait_bounded(&a_empty[j % kNA2], (j / kNA2) & 1, tmo)) break;
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issue (one thread) ----------------
        if (lane == 0) {
            int gk = 0, gw = 0, gc = 0, ui = 0;
            bool issued = false, ok = true;
            for (int k = 0; k < nu && ok; ++k) {
                const UnitInfo u = unit_at(table, k);
                if (u.e < 0) continue;
                const int nb = pow2_rows(u.nrows), ub = ui & 1;
                // N = 2 nb: the plane-1 (residue) box follows the plane-0 box,
                // so one B operand carries both planes' rows
                const uint32_t idesc = umma_idesc_f16(128, 2 * nb);
                if (!mbar_wait_bounded(&b_full[ub], (ui >> 1) & 1, tmo)) {
                    ok = false;
                    break;
                }
                for (int ctl = 0; ctl < TPU && ok; ++ctl, ++gc) {
                    const int buf = gc & 1;
                    if (gc >= 2 && !mbar_wait_bounded(&acc_empty[buf], ((gc >> 1) - 1) & 1, tmo)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dt = tmem + static_cast<uint32_t>(buf) * kAccStride;
                    if constexpr (kTileA) {
                        // one A buffer holds the tile's 160 k: ten K16 MMAs, one wait
                        // and two commits. Per group: (q - z) x [h | h residue] into
                        // the accumulator of group kk / 2 (its first K16 starts it);
                        // NVFP4: the exact weights x [h | h residue] into one.
                        const int s = gw % kStages2, ab = gk % kNA2;
                        if (!mbar_wait_bounded(&a_full[ab], (gk / kNA2) & 1, tmo)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a0 = tmem + kAOff + kAStride * ab;
                        const uint32_t bh = smem_u32(sbh + ub * kBUnit2);
#pragma unroll
                        for (int kk = 0; kk < 10; ++kk) {
                            const uint64_t bd = umma_desc_sw128(bh + (kk >> 2) * 2 * nb * 128 + 32 * (kk & 3));
                            if constexpr (kGrp)
                                tc_mma_f16_tmem_a(dt + 32 * (kk >> 1), a0 + 8 * kk, bd, idesc, (kk & 1) ? 1u : 0u);
                            else
                                tc_mma_f16_tmem_a(dt, a0 + 8 * kk, bd, idesc, kk > 0 ? 1u : 0u);
                        }
                        tc_commit(&a_empty[ab]);
                        tc_commit(&empty[s]);
                        issued = true;
                        ++gk;
                        ++gw;
                        tc_commit(&acc_full[buf]);
                    } else {
                    for (int kp = 0; kp < KP && ok; ++kp, ++gw) {
                        const int s = gw % kStages2;
                        for (int kbl = 0; kbl < 3; ++kbl, ++gk) {
                            const int ab = gk % kNA2;
                            if (!mbar_wait_bounded(&a_full[ab], (gk / kNA2) & 1, tmo)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint32_t a0 = tmem + kAOff + kAStride * ab;
                            const uint32_t bk = smem_u32(sbh + ub * kBUnit2 + (kp * 3 + kbl) * 2 * nb * 128);
                            const int nk16 = kbl < 2 ? 4 : 2;      // K 160 = 64 + 64 + 32
                            for (int kk = 0; kk < nk16; ++kk) {
                                const uint64_t bd = umma_desc_sw128(bk + 32 * kk);
                                // A_hi x [h | h residue], then A_lo x [h | h residue]
                                tc_mma_f16_tmem_a(dt, a0 + 8 * kk, bd, idesc, (kp > 0 || kbl > 0 || kk > 0) ? 1u : 0u);
                                if constexpr (!kNv) tc_mma_f16_tmem_a(dt, a0 + 32 + 8 * kk, bd, idesc, 1u);
                            }
                            tc_commit(&a_empty[ab]);
                            if (kbl == 2) tc_commit(&empty[s]);
                            issued = true;
                        }
                    }
                    if (ok) tc_commit(&acc_full[buf]);
                    }   // per K block
                }
                if (ok) tc_commit(&b_empty[ub]);
                ++ui;
            }
            if (!ok) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
            // every MMA issued here has completed before TMEM is freed
            if (issued) {
                tc_commit(drain);
                mbar_wait_bounded(drain, 0, tmo);
            }
        }
    } else {
        // ---------------- epilogue: TMEM -> y[slot][col] = weight * D ----------------
        const int quarter = warp & 3;
        int gc = 0;
        bool alive = true;
        for (int k = 0; k < nu && alive; ++k) {
            const UnitInfo u = unit_at(table, k);
            if (u.e < 0) continue;
            // the slots and router weights of the unit's rows n = lane, lane + 32
            int sl0 = 0, sl1 = 0;
            float wt0 = 0.f, wt1 = 0.f;
            const float gs = MB == 2 ? args.global_scale[2 * u.e + 1] : 1.0f;   // NVFP4 W2 global
            if (lane < u.nrows) {
                sl0 = args.sorted_slots[u.row0 + lane];
                wt0 = args.topk_weights[sl0] * gs;
            }
            if (lane + 32 < u.nrows) {
                sl1 = args.sorted_slots[u.row0 + lane + 32];
                wt1 = args.topk_weights[sl1] * gs;
            }
            const int nb = pow2_rows(u.nrows);
            for (int ctl = 0; ctl < TPU; ++ctl, ++gc) {
                const int buf = gc & 1;
                // per-group scheme: this lane's column's five group scales, loaded
                // (L2: the producer's copy of the records) before the wait
                float sc[5];
                if constexpr (kGrp) {
                    const int t32 = 4 * (u.tile * TPU + ctl) + quarter;     // 32-column tile
                    const uint8_t *rec = args.w2_meta + (static_cast<int64_t>(u.e) * kColTiles + t32) * 5 * 32 * MB +
                                         lane * MB;
#pragma unroll
                    for (int g5 = 0; g5 < 5; ++g5) {
                        const uint32_t sb = static_cast<uint32_t>(__ldg(rec + g5 * 32 * MB)) |
                                            (static_cast<uint32_t>(__ldg(rec + g5 * 32 * MB + 1)) << 8);
                        sc[g5] = half_bits_to_float(sb);
                    }
                }
                if (!warp_wait(&acc_full[buf], (gc >> 1) & 1, tmo)) {
                    if (lane == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                    alive = false;
                    break;
                }
                tc_fence_after();
                float *ycol = args.y + 128 * (u.tile * TPU + ctl) + 32 * quarter + lane;
                const uint32_t dq = tmem + (static_cast<uint32_t>(32 * quarter) << 16) + static_cast<uint32_t>(buf) * kAccStride;
                if constexpr (kGrp) {
                    // y = sum over the groups of scale * (fp16(h) part + residue part)
                    float yv[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) yv[j] = 0.f;
#pragma unroll 1
                    for (int g5 = 0; g5 < 5; ++g5) {            // (not unrolled: 128 registers a thread)
                        uint32_t v[16], r[16];
                        tc_ld16(dq + 32 * g5, v);
                        tc_ld16(dq + 32 * g5 + 16, r);
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            yv[j] = fmaf(sc[g5], __uint_as_float(v[j]) + __uint_as_float(r[j]), yv[j]);
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int slot = __shfl_sync(0xffffffffu, sl0, j);
                        const float w = __shfl_sync(0xffffffffu, wt0, j);
                        if (j < u.nrows) ycol[static_cast<int64_t>(slot) * kHidden] = w * yv[j];
                    }
                }
                for (int n0 = 0; n0 < nb && !kGrp; n0 += 16) {
                    uint32_t v[16], r[16];
                    tc_ld16(dq + static_cast<uint32_t>(n0), v);          // x fp16(h) rows
                    tc_ld16(dq + static_cast<uint32_t>(nb + n0), r);     // x residue rows
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = n0 + j;
                        const int slot = __shfl_sync(0xffffffffu, n < 32 ? sl0 : sl1, n & 31);
                        const float w = __shfl_sync(0xffffffffu, n < 32 ? wt0 : wt1, n & 31);
                        if (n < u.nrows)
                            ycol[static_cast<int64_t>(slot) * kHidden] = w * (__uint_as_float(v[j]) + __uint_as_float(r[j]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[buf]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tc_dealloc(tmem, kTmemCols2);
    if (tid == 0) trace_end(args.trace, 1);
}

// out[t][c] = fp16(sum over j of y[t k + j][c]), j in order; 4 columns per thread.
__global__ void combine_kernel(const float *y, uint16_t *out, int32_t M, int32_t top_k, uint64_t *trace)
{
    grid_dependency_wait();
    if (threadIdx.x == 0) trace_start(trace, 2);
    const int64_t n4 = static_cast<int64_t>(M) * (kHidden / 4);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / (kHidden / 4);
        const int c4 = static_cast<int>(i - t * (kHidden / 4));
        const float4 *src = reinterpret_cast<const float4 *>(y + t * top_k * kHidden) + c4;
        float4 acc = __ldcs(src);
        for (int j = 1; j < top_k; ++j) {
            const float4 v = __ldcs(src + j * (kHidden / 4));
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        uint2 o;
        o.x = static_cast<uint32_t>(f2h_bits(acc.x)) | (static_cast<uint32_t>(f2h_bits(acc.y)) << 16);
        o.y = static_cast<uint32_t>(f2h_bits(acc.z)) | (static_cast<uint32_t>(f2h_bits(acc.w)) << 16);
        *reinterpret_cast<uint2 *>(out + t * kHidden + 4 * c4) = o;
    }
    if (trace) {
        __syncthreads();
        if (threadIdx.x == 0) trace_end(trace, 2);
    }
}

// The unit tables hold at most kMaxUnits units per CTA: refuse a grid too
// small for the largest routing the call's shape allows.
static bool units_fit(int S, int E, int C, int tiles, int grid)
{
    const int64_t units = static_cast<int64_t>(max_work_items(S, E, C)) * tiles;
    return grid > 0 && units <= static_cast<int64_t>(kMaxUnits) * grid;
}

awq_status launch_w13_tc(int mb, int S, int sms, cudaStream_t st, const CUtensorMap &tq13, const CUtensorMap &tm13,
                         const StageArgs &a)
{
    const int smem = smem13();
    void (*kernel)(const CUtensorMap, const CUtensorMap, StageArgs);
    if (a.inter == 160)
        kernel = mb == 4 ? w13_tc_kernel<4, 160> : mb == 3 ? w13_tc_kernel<3, 160> : w13_tc_kernel<2, 160>;
    else
        kernel = mb == 4 ? w13_tc_kernel<4, 640> : mb == 3 ? w13_tc_kernel<3, 640> : w13_tc_kernel<2, 640>;
    const int tiles = (a.inter / kPieceCols + kPiecesPerTile - 1) / kPiecesPerTile;
    if (!units_fit(S, a.num_experts, kTcRows13, tiles, sms)) return AWQ_ERR_UNSUPPORTED_SHAPE;
    awq_status r = set_smem(kernel, smem);
    if (r) return r;
    return launch(kernel, dim3(sms), dim3(kTcThreads), smem, 1, st, tq13, tm13, a);
}

awq_status launch_w2_tc(int mb, int S, int sms, cudaStream_t st, const CUtensorMap (&th)[4], const StageArgs &a)
{
    const int smem = smem2();
    void (*kernel)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, StageArgs);
    // Units of one 128-column tile when units of five would leave every CTA
    // with at most one (small batches: most CTAs idle, each busy one working
    // through five tiles), else units of five (the item's h boxes loaded once
    // per five tiles; measured faster from about 8 tokens up). The bound on
    // the items is the host's: the routing is on the device.
    const int64_t items = max_work_items(S, a.num_experts, w2_rows(a.inter, mb));
    const bool one = a.inter == 160 && items * (kHidden / 128 / kTilesPerUnit2) <= sms &&
                     units_fit(S, a.num_experts, w2_rows(a.inter, mb), kHidden / 128, sms);
    if (a.inter == 160 && one)
        kernel = mb == 4 ? w2_tc_kernel<4, 160, 1> : mb == 3 ? w2_tc_kernel<3, 160, 1> : w2_tc_kernel<2, 160, 1>;
    else if (a.inter == 160)
        kernel = mb == 4 ? w2_tc_kernel<4, 160, kTilesPerUnit2> : mb == 3 ? w2_tc_kernel<3, 160, kTilesPerUnit2>
                                                                          : w2_tc_kernel<2, 160, kTilesPerUnit2>;
    else
        kernel = mb == 4 ? w2_tc_kernel<4, 640, kTilesPerUnit2> : mb == 3 ? w2_tc_kernel<3, 640, kTilesPerUnit2>
                                                                          : w2_tc_kernel<2, 640, kTilesPerUnit2>;
    if (!units_fit(S, a.num_experts, w2_rows(a.inter, mb), one ? kHidden / 128 : kHidden / 128 / kTilesPerUnit2,
                   sms))
        return AWQ_ERR_UNSUPPORTED_SHAPE;
    awq_status r = set_smem(kernel, smem);
    if (r) return r;
    return launch(kernel, dim3(sms), dim3(kTcThreads), smem, 1, st, th[0], th[1], th[2], th[3], a);
}

awq_status launch_combine(int M, int top_k, const float *y, uint16_t *out, uint64_t *trace, cudaStream_t st)
{
    const int64_t work = static_cast<int64_t>(M) * (kHidden / 4);
    const int blocks = static_cast<int>(std::min<int64_t>((work + 255) / 256, 152 * 8));
    return launch(combine_kernel, dim3(blocks), dim3(256), 0, 1, st, y, out, M, top_k, trace);
}

}  // namespace awq
