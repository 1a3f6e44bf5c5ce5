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
// Work items: each active segment's rows (sorted-slot order) in chunks of at
// most 64 rows (W13) / 128 rows (W2; 32 at I = 640), numbered segment by
// segment; a CTA
// finds its item from the CSR offsets. Operands are K-major with the 128-byte
// swizzle: 64 fp16 of K per 128-byte row.
//
// w13_tc_kernel: CTA (column tile c, item) computes the 8 prepared pieces
// 8c .. 8c+7 (64 gate + 64 up columns; UMMA row 16p + 8 half + col) for the
// item's rows. Per 64-wide K block a producer warp bulk-copies the pieces'
// packed words and records and gathers the rows' x chunks with cp.async
// into the swizzled B tile; eight warps (warp p = piece p) expand the int4
// words into the two 128 x 64 fp16 A tiles (s_hi and s_lo parts; one 16-byte
// chunk per packed word), and one thread issues eight K16 MMAs. The epilogue reads the accumulator with tcgen05.ld
// (warp w reads TMEM lanes 32 (w mod 4) ..), pairs each gate row with its up
// row (8 lanes apart) and stores h = silu(gate) * up as fp16, sorted-slot
// order (and, on the layer path, the residue plane).
//
// w2_tc_kernel: CTA (group of 10 output-column tiles of 128, item) keeps the
// item's h rows of both planes resident (TMA, 3 boxes of 64 K per 160-row K
// part and plane) and
// streams, per (column tile, K part), the 4 x 20 packed lines and 20 record
// rows of the prepared bank. Per K block of the part (64, 64, 32 rows of K)
// eight warps expand them into the two 128 x 64 A tiles, one thread issues
// the K16 MMAs into one of two TMEM accumulators, and the epilogue of the
// previous column tile
// (y[slot][col] = router weight * D, fp32) overlaps the current MMAs.
// combine_kernel then sums each token's k products in slot order and rounds
// to fp16 -- deterministic, no atomics.
#include <algorithm>

#include <cuda_fp16.h>

#include "awq_dequant.cuh"
#include "awq_launch.cuh"
#include "awq_moe_kernels.cuh"
#include "awq_ptx.cuh"
#include "awq_tc.cuh"

namespace awq {

namespace {

constexpr int kTcExpandWarps = 8;
constexpr int kTcThreads = (kTcExpandWarps + 1) * 32;   // + producer warp
constexpr int kTcExpand = kTcExpandWarps * 32;
constexpr int kTcProducer = kTcExpandWarps;
constexpr int kBarExpand = 1;                           // named barrier of the expand warps
constexpr int kTileA = 128 * 128;                       // 128 rows x 64 fp16

// ------------------------------------------------------------------ W13
constexpr int kStages13 = 3;
constexpr int kKBlock = 64;
constexpr int kKBlocks13 = kHidden / kKBlock;            // 40
constexpr int kPiecesPerTile = 8;
constexpr int kQBlock = 2 * 4 * kPieceCols * 2 * 4;     // one piece's words of a K block: 512 B
constexpr int kQm13 = kPiecesPerTile * kQBlock + 1024;  // words + records (<= 32 * 4 per piece)
constexpr int kB13 = kTcRows13 * 128;                   // B tile of a K block
constexpr int kABuf = 2 * kTileA;                       // A tiles of the s_hi and s_lo parts

struct Lay13 {
    static constexpr int a = 0;
    static constexpr int b = 2 * kABuf;
    static constexpr int qm = b + kStages13 * kB13;
    static constexpr int tok = qm + kStages13 * kQm13;
    static constexpr int bars = tok + kTcRows13 * 4;
    static constexpr int misc = bars + (2 * kStages13 + 2 + 1) * 8;
    static constexpr int total = misc + 64;
};

int smem13() { return Lay13::total + 1024; }

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

__device__ __forceinline__ int pow2_rows(int n) { return n <= 16 ? 16 : n <= 32 ? 32 : n <= 64 ? 64 : 128; }

}  // namespace

// grid (ceil(PJ / 8) column tiles, max work items), kTcThreads threads
template <int MB, int INTER>
__global__ void __launch_bounds__(kTcThreads, 1) w13_tc_kernel(StageArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    constexpr int PJ = INTER / kPieceCols;
    constexpr int kMeta13 = piece_meta_bytes(MB);
    constexpr int kMBlock = 2 * 16 * MB;                  // one piece's records of a K block
    uint8_t *sa = smem + Lay13::a;
    uint8_t *sb = smem + Lay13::b;
    uint8_t *sqm = smem + Lay13::qm;
    int32_t *s_tok = reinterpret_cast<int32_t *>(smem + Lay13::tok);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lay13::bars);
    uint64_t *empty = full + kStages13;
    uint64_t *mma_done = empty + kStages13;               // [2] A buffer free again
    uint64_t *acc_done = mma_done + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Lay13::misc);
    int32_t *s_res = reinterpret_cast<int32_t *>(smem + Lay13::misc + 8);
    int32_t *s_warp = reinterpret_cast<int32_t *>(smem + Lay13::misc + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x;
    const uint64_t tmo = args.timeout_ns;

    grid_dependency_wait();
    if (tid == 0) trace_start(args.trace, 0);
    const int A = *args.num_active;
    find_work_item<kTcThreads>(blockIdx.y, A, args.offsets, kTcRows13, s_warp, s_res);
    const int a = s_res[0];
    if (a < 0) return;
    const int e = args.active_ids[a];
    const int row0 = args.offsets[a] + kTcRows13 * s_res[1];
    const int nrows = min(kTcRows13, args.offsets[a + 1] - row0);
    if (e < 0 || e >= args.num_experts) {
        if (tid == 0) set_status(args.status, AWQ_ERR_BAD_EXPERT_ID);
        return;
    }
    const int nb = pow2_rows(nrows);
    const int np = min(kPiecesPerTile, PJ - kPiecesPerTile * tile);
    const uint32_t tcols = nb < 32 ? 32 : nb;
    for (int r = tid; r < nrows; r += kTcThreads) s_tok[r] = args.sorted_slots[row0 + r] / args.top_k;
    if (tid == 0) {
        for (int s = 0; s < kStages13; ++s) {
            mbar_init(&full[s], 2);      // the copies' expect_tx arrival + the gathered rows' arrival
            mbar_init(&empty[s], 1);
        }
        mbar_init(&mma_done[0], 1);
        mbar_init(&mma_done[1], 1);
        mbar_init(acc_done, 1);
        fence_barrier_init();
    }
    if (warp == 0) tc_alloc(tmem_slot, tcols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTcProducer) {
        // ---------------- producer: packed words, records, gathered x rows ----------------
        int issued = 0;
        bool alive = true;
        for (int kb = 0; kb < kKBlocks13; ++kb) {
            const int s = kb % kStages13;
            if (kb >= kStages13) {
                const bool freed = mbar_wait_bounded(&empty[s], ((kb / kStages13) - 1) & 1, tmo);
                if (!__all_sync(0xffffffffu, freed)) {
                    if (lane == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                    alive = false;
                    break;
                }
            }
            uint8_t *q = sqm + s * kQm13;
            uint8_t *m = q + kPiecesPerTile * kQBlock;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[s], np * (kQBlock + kMBlock));
                for (int p = 0; p < np; ++p) {
                    const int64_t gp = static_cast<int64_t>(e) * PJ + kPiecesPerTile * tile + p;
                    bulk_load(q + p * kQBlock,
                              reinterpret_cast<const uint8_t *>(args.w13_q) + gp * kPieceQ + kb * kQBlock, kQBlock,
                              &full[s]);
                    bulk_load(m + p * kMBlock, args.w13_meta + gp * kMeta13 + kb * kMBlock, kMBlock, &full[s]);
                }
            }
            // rows r < nrows, 16-byte chunk c of the K block: (r, c) = i / 8, i % 8
            const uint32_t bs = smem_u32(sb + s * kB13);
            for (int i = lane; i < nrows * 8; i += 32) {
                const int r = i >> 3, c = i & 7;
                cp_async_16(bs + sw128_offset(r, c),
                            args.x + static_cast<int64_t>(s_tok[r]) * kHidden + kb * kKBlock + c * 8);
            }
            cp_async_commit();
            ++issued;
            if (kb >= 1) {
                // the rows of K block kb - 1 have landed: make them visible to
                // the tensor core (async proxy) and release that stage (one
                // block behind the issue, so the consumers never wait for a
                // later block's stage to free up)
                cp_async_wait_group<1>();
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[(kb - 1) % kStages13]);
            }
        }
        cp_async_wait_group<0>();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (alive && lane == 0) mbar_arrive(&full[(kKBlocks13 - 1) % kStages13]);
        // let the weight copies still in flight land, and the MMAs' releases of
        // the last stages arrive, before the CTA exits (a wait that runs out
        // ends the drain: the consumers have stopped)
        if (lane == 0) {
            bool drained = true;
            for (int kb = max(0, issued - kStages13); kb < issued && drained; ++kb)
                drained = mbar_wait_bounded(&full[kb % kStages13], (kb / kStages13) & 1, tmo);
            for (int kb = max(0, issued - kStages13); kb < issued && drained; ++kb)
                drained = mbar_wait_bounded(&empty[kb % kStages13], (kb / kStages13) & 1, tmo);
        }
    } else {
        // ---------------- expand + MMA issue ----------------
        // warp p expands piece p; lane (group g2, column c, half) owns record
        // lane of the K block and its four words t = 0..3 (word index
        // 64 g2 + 16 t + lane mod 16) -> UMMA row 16p + 8 half + c, 16-byte
        // chunk 4 g2 + t of the row
        const int p = warp;
        const int half = lane & 1, c = (lane >> 1) & 7, g2 = lane >> 4;
        const int arow = 16 * p + 8 * half + c;
        const uint32_t idesc = umma_idesc_f16(128, nb);
        bool ok = true, issued = false;
        for (int kb = 0; kb < kKBlocks13; ++kb) {
            const int s = kb % kStages13, ab = kb & 1;
            bool good = mbar_wait_bounded(&full[s], (kb / kStages13) & 1, tmo);
            // A buffer ab was last read by the MMAs of K block kb - 2
            if (good && kb >= 2) good = mbar_wait_bounded(&mma_done[ab], ((kb - 2) >> 1) & 1, tmo);
            if (good && p < np) {
                const uint8_t *q = sqm + s * kQm13 + p * kQBlock;
                const SplitRecord rec = split_record<MB>(sqm + s * kQm13 + kPiecesPerTile * kQBlock + p * kMBlock + lane * MB);
                uint8_t *at = sa + ab * kABuf;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(q + (64 * g2 + 16 * t + (lane & 15)) * 4);
                    uint4 hi, lo;
                    dequant_word_split(w, rec, hi, lo);
                    const uint32_t off = sw128_offset(arow, 4 * g2 + t);
                    *reinterpret_cast<uint4 *>(at + off) = hi;
                    *reinterpret_cast<uint4 *>(at + kTileA + off) = lo;
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (!named_barrier_and(kBarExpand, kTcExpand, good)) {
                ok = false;
                break;
            }
            if (tid == 0) {
                tc_fence_after();
                const uint32_t a0 = smem_u32(sa + ab * kABuf), b0 = smem_u32(sb + s * kB13);
#pragma unroll
                for (int k = 0; k < kKBlock / 16; ++k) {
                    const uint64_t bd = umma_desc_sw128(b0 + 32 * k);
                    tc_mma_f16(tmem, umma_desc_sw128(a0 + 32 * k), bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    tc_mma_f16(tmem, umma_desc_sw128(a0 + kTileA + 32 * k), bd, idesc, 1u);
                }
                tc_commit(&mma_done[ab]);
                tc_commit(&empty[s]);
                issued = true;
            }
        }
        if (tid == 0 && issued) tc_commit(acc_done);
        if (!ok && tid == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
        // ---------------- epilogue: TMEM -> SwiGLU -> h ----------------
        const bool done = ok && mbar_wait_bounded(acc_done, 0, tmo);
        if (__all_sync(0xffffffffu, done)) {
            tc_fence_after();
            const int r = 32 * (warp & 3) + lane;             // UMMA row of this lane
            const int p = r >> 4, hr = (r >> 3) & 1, cc = r & 7;
            const int col = kPieceCols * (kPiecesPerTile * tile + p) + cc;
            for (int n0 = 16 * (warp >> 2); n0 < nb; n0 += 32) {
                uint32_t v[16];
                tc_ld16(tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + static_cast<uint32_t>(n0), v);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float mine = __uint_as_float(v[j]);
                    const float other = __shfl_xor_sync(0xffffffffu, mine, 8);   // up of a gate row
                    const int n = n0 + j;
                    if (hr == 0 && p < np && n < nrows) {
                        const float hv = silu_f(mine) * other;
                        const uint16_t hi = f2h_bits(hv);
                        const int64_t at = static_cast<int64_t>(row0 + n) * INTER + col;
                        args.h_out[at] = hi;
                        if (args.h_lo) args.h_lo[at] = f2h_bits(hv - __half2float(__ushort_as_half(hi)));
                    }
                }
            }
        } else if (ok && lane == 0) {
            set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
        }
        // every MMA this CTA issued has completed, and its commits have
        // arrived, before its TMEM and shared memory are released
        if (tid == 0 && issued) {
            if (!done) mbar_wait_bounded(acc_done, 0, tmo);
            else
                for (int kb = kKBlocks13 - 2; kb < kKBlocks13; ++kb)
                    mbar_wait_bounded(&mma_done[kb & 1], (kb >> 1) & 1, tmo);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tc_dealloc(tmem, tcols);
    if (tid == 0) trace_end(args.trace, 0);
}

// ------------------------------------------------------------------ W2
namespace {

constexpr int kStages2 = 3;
constexpr int kTilesPerCta2 = 10;                        // 128-column output tiles per CTA
constexpr int kCtGroups2 = kHidden / 128 / kTilesPerCta2;   // 2
constexpr int kQUnit2 = 4 * kW2TileKK * 128;             // 4 x 20 lines: 10240 B
constexpr int kMUnitMax2 = 4 * 5 * 32 * 4;               // 20 record rows (4-byte records)
constexpr int kBBytes2 = 2 * 3 * 128 * 128;              // resident h boxes: KP x 3 x 2 planes x rows x 128 B

struct Lay2 {
    static constexpr int b = 0;
    static constexpr int a = b + kBBytes2;                 // 2 buffers x (s_hi, s_lo) A tiles
    static constexpr int wq = a + 2 * kABuf;
    static constexpr int wstage = kQUnit2 + kMUnitMax2;
    static constexpr int slot = wq + kStages2 * wstage;
    static constexpr int wgt = slot + 128 * 4;
    static constexpr int bars = wgt + 128 * 4;
    static constexpr int misc = bars + (2 * kStages2 + 1 + 2 + 2 + 1) * 8;
    static constexpr int total = misc + 64;
};

int smem2() { return Lay2::total + 1024; }

}  // namespace

// grid (kCtGroups2, max work items), kTcThreads threads
template <int MB, int INTER>
__global__ void __launch_bounds__(kTcThreads, 1)
w2_tc_kernel(const __grid_constant__ CUtensorMap th16, const __grid_constant__ CUtensorMap th32,
             const __grid_constant__ CUtensorMap th64, const __grid_constant__ CUtensorMap th128, StageArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    constexpr int KP = INTER / 160;
    constexpr int C2 = tc_rows2(INTER);
    constexpr int kWUnits = kTilesPerCta2 * KP;             // weight units (column tile, K part)
    constexpr int kUnits = 3 * kWUnits;                     // K blocks of 64, 64, 32 rows per unit
    constexpr int kMUnit = 4 * 5 * 32 * MB;
    uint8_t *sbh = smem + Lay2::b;
    uint8_t *sa = smem + Lay2::a;
    uint8_t *sw = smem + Lay2::wq;
    int32_t *s_slot = reinterpret_cast<int32_t *>(smem + Lay2::slot);
    float *s_wgt = reinterpret_cast<float *>(smem + Lay2::wgt);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lay2::bars);
    uint64_t *empty = full + kStages2;
    uint64_t *bfull = empty + kStages2;
    uint64_t *mma_done = bfull + 1;                         // [2] A buffers
    uint64_t *acc_full = mma_done + 2;                      // [2] accumulators
    uint64_t *drain = acc_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Lay2::misc);
    int32_t *s_res = reinterpret_cast<int32_t *>(smem + Lay2::misc + 8);
    int32_t *s_warp = reinterpret_cast<int32_t *>(smem + Lay2::misc + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ct0 = blockIdx.x * kTilesPerCta2;
    const uint64_t tmo = args.timeout_ns;

    grid_dependency_wait();
    if (tid == 0) trace_start(args.trace, 1);
    const int A = *args.num_active;
    find_work_item<kTcThreads>(blockIdx.y, A, args.offsets, C2, s_warp, s_res);
    const int a = s_res[0];
    if (a < 0) return;
    const int e = args.active_ids[a];
    const int row0 = args.offsets[a] + C2 * s_res[1];
    const int nrows = min(C2, args.offsets[a + 1] - row0);
    if (e < 0 || e >= args.num_experts) {
        if (tid == 0) set_status(args.status, AWQ_ERR_BAD_EXPERT_ID);
        return;
    }
    const int nb = pow2_rows(nrows);
    const uint32_t tcols = 2 * nb < 32 ? 32 : 2 * nb;
    for (int r = tid; r < nrows; r += kTcThreads) {
        const int sl = args.sorted_slots[row0 + r];
        s_slot[r] = sl;
        s_wgt[r] = args.topk_weights[sl];
    }
    if (tid == 0) {
        for (int s = 0; s < kStages2; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(bfull, 1);
        mbar_init(&mma_done[0], 1);
        mbar_init(&mma_done[1], 1);
        mbar_init(&acc_full[0], 1);
        mbar_init(&acc_full[1], 1);
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == 0) tc_alloc(tmem_slot, tcols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int bbox = nb * 128;                               // bytes of one h box

    if (warp == kTcProducer) {
        if (lane == 0) {
            const CUtensorMap *th = nb == 16 ? &th16 : nb == 32 ? &th32 : nb == 64 ? &th64 : &th128;
            // box (kp, kbl, plane): plane 0 = fp16(h) rows, plane 1 = residue rows (S below)
            const int S = args.M * args.top_k;
            mbar_arrive_expect_tx(bfull, KP * 3 * 2 * bbox);
            for (int kp = 0; kp < KP; ++kp)
                for (int b = 0; b < 3; ++b)
                    for (int pl = 0; pl < 2; ++pl)
                        tma_load_2d(sbh + ((kp * 3 + b) * 2 + pl) * bbox, th, bfull, 160 * kp + 64 * b, pl * S + row0);
            int issued = 0;
            for (int u = 0; u < kWUnits; ++u) {
                const int s = u % kStages2;
                if (u >= kStages2 && !mbar_wait_bounded(&empty[s], ((u / kStages2) - 1) & 1, tmo)) {
                    set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                    break;
                }
                const int ct = ct0 + u / KP, kp = u % KP;
                // 4 consecutive 32-column tiles of (e, kp): 80 lines, 20 record rows
                const int64_t tile0 = (static_cast<int64_t>(e) * KP + kp) * kColTiles + 4 * ct;
                uint8_t *q = sw + s * Lay2::wstage;
                mbar_arrive_expect_tx(&full[s], kQUnit2 + kMUnit);
                bulk_load(q, reinterpret_cast<const uint8_t *>(args.w2_q) + tile0 * kW2TileKK * 128, kQUnit2, &full[s]);
                bulk_load(q + kQUnit2, args.w2_meta + tile0 * 5 * 32 * MB, kMUnit, &full[s]);
                ++issued;
            }
            // let the copies still in flight land, and the MMAs' releases of the
            // last stages arrive, before the CTA exits (a wait that runs out
            // ends the drain: the consumers have stopped)
            bool drained = mbar_wait_bounded(bfull, 0, tmo);
            for (int u = max(0, issued - kStages2); u < issued && drained; ++u)
                drained = mbar_wait_bounded(&full[u % kStages2], (u / kStages2) & 1, tmo);
            for (int u = max(0, issued - kStages2); u < issued && drained; ++u)
                drained = mbar_wait_bounded(&empty[u % kStages2], (u / kStages2) & 1, tmo);
        }
    } else {
        // thread: output column m = tid mod 128 of the tile (UMMA row); in K
        // block kbl of a part, the packed rows r = 8 kbl + 4 rh + i, i < 4
        // (rh = tid / 128), which share the record of group 2 kbl + rh
        const int m = tid & 127, rh = tid >> 7;
        const int t4 = m >> 5, c32 = m & 31;
        const uint32_t idesc = umma_idesc_f16(128, nb);
        bool ok = true, issued = false;
        auto epilogue = [&](int ctl) {
            // y[slot][128 ct + m] = weight * D[m][n] for the item's rows n
            const int buf = ctl & 1;
            const bool got = ok && mbar_wait_bounded(&acc_full[buf], (ctl >> 1) & 1, tmo);
            if (!__all_sync(0xffffffffu, got)) {
                if (ok && lane == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                ok = false;
                return;
            }
            tc_fence_after();
            float *ycol = args.y + 128 * (ct0 + ctl) + 32 * (warp & 3) + lane;
            for (int n0 = 16 * (warp >> 2); n0 < nb; n0 += 32) {
                uint32_t v[16];
                tc_ld16(tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + static_cast<uint32_t>(buf * nb + n0), v);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int n = n0 + j;
                    if (n < nrows) ycol[static_cast<int64_t>(s_slot[n]) * kHidden] = s_wgt[n] * __uint_as_float(v[j]);
                }
            }
            tc_fence_before();
        };
        for (int u = 0; u < kUnits; ++u) {
            const int kbl = u % 3, wu = u / 3, ab = u & 1;
            const int ctl = wu / KP, kp = wu % KP, s = wu % kStages2;
            bool good = ok;
            if (good && kbl == 0) good = mbar_wait_bounded(&full[s], (wu / kStages2) & 1, tmo);
            if (good && u == 0) good = mbar_wait_bounded(bfull, 0, tmo);
            if (good && u >= 2) good = mbar_wait_bounded(&mma_done[ab], ((u - 2) >> 1) & 1, tmo);
            const int g = 2 * kbl + rh;                     // group of this thread's rows
            if (good && g < 5) {
                const uint8_t *q = sw + s * Lay2::wstage;
                const SplitRecord rec = split_record<MB>(q + kQUnit2 + (t4 * 5 + g) * 32 * MB + c32 * MB);
                uint8_t *at = sa + ab * kABuf;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 4 * g + i;
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(q + (t4 * kW2TileKK + r) * 128 + c32 * 4);
                    uint4 hi, lo;
                    dequant_word_split(w, rec, hi, lo);
                    const uint32_t off = sw128_offset(m, r & 7);
                    *reinterpret_cast<uint4 *>(at + off) = hi;
                    *reinterpret_cast<uint4 *>(at + kTileA + off) = lo;
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (!named_barrier_and(kBarExpand, kTcExpand, good)) {
                if (ok && tid == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                ok = false;
                break;
            }
            if (tid == 0) {
                tc_fence_after();
                const uint32_t a0 = smem_u32(sa + ab * kABuf);
                const uint32_t bk = smem_u32(sbh + (kp * 3 + kbl) * 2 * bbox);
                const uint32_t dt = tmem + static_cast<uint32_t>((ctl & 1) * nb);
                const int nk16 = kbl < 2 ? 4 : 2;           // K 160 = 64 + 64 + 32
                for (int k = 0; k < nk16; ++k) {
                    const uint64_t ahi = umma_desc_sw128(a0 + 32 * k);
                    const uint64_t bhi = umma_desc_sw128(bk + 32 * k);
                    tc_mma_f16(dt, ahi, bhi, idesc, (kp > 0 || kbl > 0 || k > 0) ? 1u : 0u);
                    tc_mma_f16(dt, umma_desc_sw128(a0 + kTileA + 32 * k), bhi, idesc, 1u);
                    tc_mma_f16(dt, ahi, umma_desc_sw128(bk + bbox + 32 * k), idesc, 1u);
                }
                tc_commit(&mma_done[ab]);
                if (kbl == 2) tc_commit(&empty[s]);
                if (kbl == 2 && kp == KP - 1) tc_commit(&acc_full[ctl & 1]);
                issued = true;
            }
            // the previous tile's epilogue overlaps this tile's MMAs
            if (kbl == 0 && kp == 0 && ctl > 0) epilogue(ctl - 1);
        }
        if (ok) epilogue(kTilesPerCta2 - 1);
        // every MMA this CTA issued has completed, and its commits have
        // arrived, before its TMEM and shared memory are released
        if (tid == 0 && issued) {
            if (!ok) {
                tc_commit(drain);
                mbar_wait_bounded(drain, 0, tmo);
            } else {
                for (int u = kUnits - 2; u < kUnits; ++u)
                    if (u >= 0) mbar_wait_bounded(&mma_done[u & 1], (u >> 1) & 1, tmo);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tc_dealloc(tmem, tcols);
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

awq_status launch_w13_tc(int mb, int S, cudaStream_t st, const StageArgs &a)
{
    const int smem = smem13();
    void (*kernel)(StageArgs);
    if (a.inter == 160)
        kernel = mb == 4 ? w13_tc_kernel<4, 160> : w13_tc_kernel<3, 160>;
    else
        kernel = mb == 4 ? w13_tc_kernel<4, 640> : w13_tc_kernel<3, 640>;
    awq_status r = set_smem(kernel, smem);
    if (r) return r;
    const int tiles = (a.inter / kPieceCols + kPiecesPerTile - 1) / kPiecesPerTile;
    const dim3 grid(tiles, max_work_items(S, a.num_experts, kTcRows13));
    return launch(kernel, grid, dim3(kTcThreads), smem, 1, st, a);
}

awq_status launch_w2_tc(int mb, int S, cudaStream_t st, const CUtensorMap (&th)[4], const StageArgs &a)
{
    const int smem = smem2();
    void (*kernel)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, StageArgs);
    if (a.inter == 160)
        kernel = mb == 4 ? w2_tc_kernel<4, 160> : w2_tc_kernel<3, 160>;
    else
        kernel = mb == 4 ? w2_tc_kernel<4, 640> : w2_tc_kernel<3, 640>;
    awq_status r = set_smem(kernel, smem);
    if (r) return r;
    const dim3 grid(kCtGroups2, max_work_items(S, a.num_experts, tc_rows2(a.inter)));
    return launch(kernel, grid, dim3(kTcThreads), smem, 1, st, th[0], th[1], th[2], th[3], a);
}

awq_status launch_combine(int M, int top_k, const float *y, uint16_t *out, uint64_t *trace, cudaStream_t st)
{
    const int64_t work = static_cast<int64_t>(M) * (kHidden / 4);
    const int blocks = static_cast<int>(std::min<int64_t>((work + 255) / 256, 152 * 8));
    return launch(combine_kernel, dim3(blocks), dim3(256), 0, 1, st, y, out, M, top_k, trace);
}

}  // namespace awq
