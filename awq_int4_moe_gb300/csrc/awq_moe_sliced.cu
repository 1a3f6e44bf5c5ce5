// The whole expert stage of one decode layer call (routing, W13 + SwiGLU,
// W2 + router-weighted top-k reduction) as ONE persistent cooperative kernel
// for up to 8 tokens, with W2 sliced along K together with W13.
//
// Source of the computation: 1Cat-vLLM #520 "Narrow Qwen3.8 AWQ active
// grouped decode", Purpose and Implementation (active-expert segments,
// offsets-based scheduling, one pass per stage, grouped-active exact W2
// reduction); 1Cat-vLLM #522 "Coalesce AWQ QPN W13 compact metadata loads and
// enable compact metadata by default", Purpose (3-byte records read as
// aligned 32-bit words); Leonccaa/1Cat-vLLM #12 "Add opt-in native-g32 AWQ
// QPN M1 dispatch", Purpose and stack (int32 top-10 ids and fp32 router
// weights as the stage's inputs).
//
// Why sliced. h = silu(x W13_gate) * (x W13_up) is elementwise in the
// intermediate column, and out = sum_j w_j h_j W2 sums over intermediate rows.
// So the CTA that computes intermediate columns [8p, 8p+8) of a segment can
// multiply them straight into rows [8p, 8p+8) of the segment's W2: no CTA
// waits for another's W13 results. The price is one cross-CTA sum of the
// partial outputs at the end, which costs one grid barrier.
//
// Schedule. One CTA per SM (grid = SM count, cooperative launch: all CTAs
// co-resident). The flat list of units (segment a, piece p: 8 gate + 8 up
// W13 columns over the whole K) is split into equal contiguous shares; the
// units of one 32-row W2 group are 4 consecutive units (segments hold a
// multiple of 4), so a share's groups and its W2 work follow from its bounds
// by arithmetic alone. A CTA runs, in one shared-memory ring filled by a
// producer warp:
//   W13 pieces   -- the prepared 20 KB piece + its metadata (bulk copies);
//   W2 units     -- (segment, 32-row group, column half): the rows of the
//                   group this CTA owns (one 5 KB TMA box per 8-row word row,
//                   40 column tiles of 128 bytes) + the group's metadata row
//                   for those columns;
// interleaved so that a group's W2 units follow its last piece by two pieces
// (the epilogue has finished them by then). Consumer warps (8) expand int4
// in registers and run MMAs with the weights on M, tokens on N (N = token
// index: 8 columns cover every token): m16n8k16 over whole 32-row groups for
// W13, m16n8k8 per owned 8-row word row for W2 (so rows of a group that
// another CTA owns cost nothing). Two epilogue warps sum the consumer
// warps' W13 tiles, apply SwiGLU and the router weights and store the
// weighted activations HW[token][k] of the segment in shared memory, zero
// for tokens not routed to it and for rows this CTA does not own.
//
// W2 accumulates in registers for the whole CTA (each consumer warp owns ten
// 32-column output tiles for every token), then the CTA writes its fp32
// partial output P[cta][token < M][2560] for the tokens its segments touch.
// After a grid barrier each CTA sums a share of the output over the
// contributing CTAs of each token (listed by the epilogue warps at the start,
// from the routing alone), in a fixed order: the result is deterministic run
// to run, with no atomics on data.
//
// Tile mode (few active experts: A * K parts <= 24). Then every token is
// routed to nearly every CTA's segments and the partial outputs would need a
// sum over ~G contributors per output element. Instead the epilogue writes
// the weighted activations HW to global memory, all CTAs pass the grid
// barrier, and CTA c < 80 computes the 32-column output tile c over every
// segment (its W2 lines prefetched into the ring's free stages during W13)
// and writes it directly. No partial outputs, no final sum.
//
// Every wait is bounded by the call's timeout and reports
// AWQ_ERR_DEVICE_TIMEOUT through the status word.
#include <cuda_fp16.h>

#include "awq_dequant.cuh"
#include "awq_launch.cuh"
#include "awq_moe_kernels.cuh"
#include "awq_ptx.cuh"
#include "awq_router.cuh"
#include "awq_split.cuh"

namespace awq {

namespace {

// Consumer warps: 8. With the producer and two epilogue warps that is 11
// warps, at most 3 on each of the 4 schedulers, whose 16K-register files then
// allow 168 registers a thread: the x fragments (40), the W2 accumulators (80)
// and the loads of several groups in flight. (The group step is bound by the
// integer pipe, not by latency: more warps with fewer registers do not run
// it faster, and each op's bookkeeping is paid once per warp.)
constexpr int kCW = 8;
constexpr int kProducer = kCW;                   // producer warp
constexpr int kEpi = kCW + 1;                    // first of two epilogue warps
constexpr int kThreads = (kCW + 3) * 32;         // 352
constexpr int kCThreads = kCW * 32;
constexpr int kGPW = kGroups13 / kCW;            // W13 groups per consumer warp (10)
constexpr int kStageBytes = 25600;               // 25 x 1 KB: a piece (q + meta) or a W2 unit
constexpr int kStages = 7;
constexpr int kSlots = 2;                        // W13 hand-off slots (piece i -> slot i % 2)
constexpr int kMaxTok = kSlicedMaxTokens;        // 8
constexpr int kMaxSlotsS = kMaxTok * kMaxTopK;   // 128
constexpr int kMaxGroups = 32;                   // W2 groups of one share (<= 80 pieces / 4 + 2)
constexpr int kUnitTiles = 40;                   // 32-column tiles per W2 unit
constexpr int kRowBlock = kUnitTiles * 128;      // 5120: one word row of a unit
constexpr int kUnitQ = 4 * kRowBlock;            // 20480
// A W2 unit's 40 column tiles go to consumer warp w as tiles w + 8x, x =
// 0..4; accumulator tile 5h + x of half h.
constexpr int kTPW = kUnitTiles / kCW;           // 5
constexpr int kAcc = 2 * kTPW;                   // 10
static_assert(kGroups13 % kCW == 0 && kUnitTiles % kCW == 0, "work splits evenly over the consumer warps");
// Tile mode: at most kTileMaxAK (segment, K part) pairs; a ring stage holds
// kTSlots of them, each the tile's 20 lines (1 KB-aligned 3 KB slot, 128-byte
// swizzle) and 5 metadata rows (640-byte slots after the line slots).
constexpr int kTileMaxAK = 24;
constexpr int kTSlots = 6;
constexpr int kTQSlot = 3072;
constexpr int kTMetaOff = kTSlots * kTQSlot;     // 18432
constexpr int kTMetaSlot = 640;
static_assert(kTMetaOff + kTSlots * kTMetaSlot <= kStageBytes, "tile-mode chunk fits a stage");
constexpr int kBarC = 1;                         // named barrier of the consumer warps
constexpr int kBarE = 2;                         // named barrier of the two epilogue warps
static_assert(kUnitQ + kUnitTiles * 32 * 4 <= kStageBytes, "W2 unit fits a stage");
static_assert(kPieceQ + piece_meta_bytes(4) <= kStageBytes, "W13 piece fits a stage");

// HW row stride: 2I bytes padded to 64 mod 128 so that the eight token rows
// of one B-fragment load fall in distinct banks.
__host__ __device__ constexpr int hw_row(int inter) { return inter == 160 ? 320 : 1344; }

struct Layout {
    int bars, red, hbuf, hw, route, contrib, gbars, total;
};

__host__ __device__ inline int rup(int v, int a) { return (v + a - 1) / a * a; }

__host__ __device__ inline Layout layout(int inter)
{
    Layout L;
    L.bars = kStages * kStageBytes;
    L.red = rup(L.bars + (2 * kStages + 2 * kSlots) * 8, 128);   // ring and hand-off barriers
    L.hbuf = L.red + kSlots * kCW * 32 * 16;                       // hand-off slots
    L.hw = L.hbuf + 2 * 8 * 8 * 4;                                 // SwiGLU buffer per epilogue warp
    L.route = L.hw + 2 * 8 * hw_row(inter);                        // two segment slots
    // s_ids, s_w, act, tm [128 each], bitmap[32], wpre[32], misc[16]
    L.contrib = rup(L.route + (4 * kMaxSlotsS + 32 + 32 + 16) * 4, 16);
    // per token: contributor mask [8 words], count, list [256 int16]
    L.gbars = rup(L.contrib + kMaxTok * (8 * 4 + 4 + 256 * 2), 8);
    L.total = L.gbars + (kMaxGroups + 2) * 8;      // per-group HW-ready barriers, lists-ready, epilogue-done
    return L;
}

__device__ __forceinline__ void red_add_release_u64(uint64_t *p, uint64_t v)
{
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_acquire_gpu_u64(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t ld_relaxed_gpu_u64(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *m, uint64_t *bar, int c0, int c1,
                                            int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// D = A * B + C, m16n8k8, fp16 inputs, fp32 accumulate (PTX ISA fragment
// layout of mma.m16n8k8 .row.col). A pure function of its registers.
__device__ __forceinline__ void mma_1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0, const float (&c)[4])
{
    asm("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, {%7, %8, %9, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(b0), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// Per-lane constants of the row-granular W2 step. In an 8-row word row each
// lane t takes the nibble pair (t, t + 4) of a column's word -- k rows t and
// t + 4 of the 8, the pair the HW chunk holds at elements (2t, 2t + 1) -- as
// (1024 + q) (t even: nibbles at bits 8(t/2) + 0..3) or (64 + q) (t odd:
// bits 8(t/2) + 4..7) with one shift and one lop3.
struct RowLane {
    uint32_t shift, mask, magic;
    bool odd;
};

__device__ __forceinline__ RowLane row_lane(int t)
{
    RowLane r;
    r.shift = 8u * static_cast<uint32_t>(t >> 1);
    r.odd = (t & 1) != 0;
    r.mask = r.odd ? 0x00F000F0u : 0x000F000Fu;
    r.magic = r.odd ? 0x54005400u : 0x64006400u;
    return r;
}

__device__ __forceinline__ uint32_t nib_pair(uint32_t w, const RowLane &rl)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w >> rl.shift), "r"(rl.mask), "r"(rl.magic));
    return r;
}

// One W2 unit's tiles of consumer warp `warp`: tiles warp + 8x (x = 0..4) of
// the unit's 40, into accumulator tiles kTPW * H + x. Only the word rows
// [lo, hi) this CTA owns are read and multiplied (one m16n8k8 per row and
// 16-column half), chained through the accumulator of the group, then scaled
// once per column. Row r of the unit lies at r * 5120; lane (g, t) reads
// columns 4Qg .. 4Qg+3 of the tile. hb[r]: the lane's B fragment of row r
// (HW of token g, k rows t and t + 4 of word row r).
template <int MB, int H>
__device__ __forceinline__ void w2_unit_rows(float (&acc)[kAcc][2][4], const uint8_t *base, const uint32_t (&hb)[4],
                                             int lo, int hi, int warp, int Qg, const RowLane &rl)
{
#pragma unroll
    for (int x = 0; x < kTPW; ++x) {
        const int tl = warp + kCW * x;
        const Meta4<MB> mt = meta4_of<MB>(load_meta4_raw<MB>(base + kUnitQ + (tl * 32 + 4 * Qg) * MB));
        uint32_t zp[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) zp[c] = rl.odd ? zero_pair_64(mt.z2[c]) : mt.z2[c];
        float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            if (r < lo || r >= hi) continue;
            const uint4 q = *reinterpret_cast<const uint4 *>(base + r * kRowBlock + tl * 128 + Qg * 16);
            mma_1688(t0, hsub2_u32(nib_pair(q.x, rl), zp[0]), hsub2_u32(nib_pair(q.y, rl), zp[1]), hb[r], t0);
            mma_1688(t1, hsub2_u32(nib_pair(q.z, rl), zp[2]), hsub2_u32(nib_pair(q.w, rl), zp[3]), hb[r], t1);
        }
        float(&a)[2][4] = acc[kTPW * H + x];
        const float s0 = half_bits_to_float(mt.s[0]), s1 = half_bits_to_float(mt.s[1]);
        const float s2 = half_bits_to_float(mt.s[2]), s3 = half_bits_to_float(mt.s[3]);
        a[0][0] = fmaf(s0, t0[0], a[0][0]);
        a[0][1] = fmaf(s0, t0[1], a[0][1]);
        a[0][2] = fmaf(s1, t0[2], a[0][2]);
        a[0][3] = fmaf(s1, t0[3], a[0][3]);
        a[1][0] = fmaf(s2, t1[0], a[1][0]);
        a[1][1] = fmaf(s2, t1[1], a[1][1]);
        a[1][2] = fmaf(s3, t1[2], a[1][2]);
        a[1][3] = fmaf(s3, t1[3], a[1][3]);
    }
}

}  // namespace

// TILE: the host has proven tile mode (M * top_k * K parts <= kTileMaxAK, so
// A * K parts is too); the flat-mode code is then compiled out, which frees
// registers (134-140 instead of 168) and shortens the call.
template <int MB, int INTER, bool TILE>
__global__ void __launch_bounds__(kThreads, 1)
sliced_layer_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tm_map,
                    const __grid_constant__ CUtensorMap t1q, const __grid_constant__ CUtensorMap t1m, SlicedArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    constexpr int kMeta13 = piece_meta_bytes(MB);
    constexpr int PJ = INTER / kPieceCols;         // pieces per segment
    constexpr int KP = INTER / 160;                // 160-row K parts of W2
    constexpr int HWR = hw_row(INTER);
    const int M = args.M, k = args.top_k, E = args.num_experts;
    const Layout Lo = layout(INTER);
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lo.bars);
    uint64_t *empty = full + kStages;
    uint64_t *red_full = empty + kStages;          // [kSlots] consumer warps -> epilogue warp (slot & 1)
    uint64_t *red_empty = red_full + kSlots;       // [kSlots]
    float *red = reinterpret_cast<float *>(smem + Lo.red);
    float *hbuf = reinterpret_cast<float *>(smem + Lo.hbuf);
    uint8_t *hw = smem + Lo.hw;                    // [2 slots][8 tokens][HWR]
    int32_t *s_ids = reinterpret_cast<int32_t *>(smem + Lo.route);
    float *s_w = reinterpret_cast<float *>(s_ids + kMaxSlotsS);
    int32_t *act = reinterpret_cast<int32_t *>(s_w + kMaxSlotsS);
    uint32_t *tm = reinterpret_cast<uint32_t *>(act + kMaxSlotsS);
    uint32_t *bitmap = tm + kMaxSlotsS;
    int32_t *wpre = reinterpret_cast<int32_t *>(bitmap + 32);
    int32_t *s_misc = wpre + 32;
    uint32_t *cm = reinterpret_cast<uint32_t *>(smem + Lo.contrib);      // [8 tokens][8 words] contributor CTAs
    int32_t *cnt = reinterpret_cast<int32_t *>(cm + kMaxTok * 8);        // [8] contributors per token
    int16_t *clist = reinterpret_cast<int16_t *>(cnt + kMaxTok);          // [8][256] contributors in CTA order
    uint64_t *hw_full = reinterpret_cast<uint64_t *>(smem + Lo.gbars);   // [kMaxGroups] a W2 group's HW rows ready
    uint64_t *lists_ready = hw_full + kMaxGroups;
    uint64_t *epi_done = lists_ready + 1;          // tile mode: both epilogue warps have published HW
    uint64_t *const trace = args.trace ? args.trace + static_cast<int64_t>(blockIdx.x) * AWQ_TRACE_POINTS : nullptr;
    auto stamp = [&](int pnt) {
        if (trace) trace[pnt] = global_timer_ns();
    };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int G = gridDim.x, b = blockIdx.x;
    const int S = M * k;
    const uint64_t tmo = args.timeout_ns;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&red_full[s], kCW);
            mbar_init(&red_empty[s], 1);
        }
        mbar_init(lists_ready, 2);
        mbar_init(epi_done, 2);
        fence_barrier_init();
        stamp(0);
        prefetch_tmap(&tq);
        prefetch_tmap(&tm_map);
        prefetch_tmap(&t1q);
        prefetch_tmap(&t1m);
    }
    if (tid < 32) bitmap[tid] = 0;
    for (int i = tid; i < kMaxSlotsS; i += kThreads) tm[i] = 0;
    // both HW slots start at zero: rows of tokens not routed to a segment and
    // rows of W2 this CTA does not own must multiply as zeros
    for (int i = tid * 16; i < 2 * 8 * HWR; i += kThreads * 16)
        *reinterpret_cast<uint4 *>(hw + i) = make_uint4(0, 0, 0, 0);
    grid_dependency_wait();
    grid_launch_dependents();
    // epoch of the grid barrier: the arrival count is a 64-bit total over all
    // calls on this workspace, G per call, and no other CTA of this call can
    // have arrived G times yet
    uint64_t epoch = 0;                            // thread 0 arrives and waits for the barrier
    if (tid == 0) {
        stamp(1);
        epoch = ld_relaxed_gpu_u64(args.gbar) / static_cast<uint64_t>(G);
    }

    // ---------------- routing in shared memory ----------------
    if (args.logits) {
        for (int tok = warp; tok < M; tok += kThreads / 32)
            warp_router_topk<kRouterExperts / 32>(args.logits + static_cast<int64_t>(tok) * kRouterExperts, k,
                                                  lane, s_ids + tok * k, s_w + tok * k);
        __syncthreads();
        if (tid < S) {
            const int e = s_ids[tid];
            atomicOr(&bitmap[e >> 5], 1u << (e & 31));
            if (b == 0) {
                args.topk_ids_out[tid] = e;
                args.topk_weights_out[tid] = s_w[tid];
            }
        }
    } else if (tid < S) {
        int e = args.topk_ids[tid];
        if (e < 0 || e >= E) {
            if (b == 0) set_status(args.status, AWQ_ERR_BAD_EXPERT_ID);
            e = -1;
        }
        s_ids[tid] = e;
        s_w[tid] = args.topk_weights[tid];
        if (e >= 0) atomicOr(&bitmap[e >> 5], 1u << (e & 31));
    }
    __syncthreads();
    if (tid < 32) {
        const int c = __popc(bitmap[tid]);
        int v = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, o);
            if (tid >= o) v += y;
        }
        wpre[tid] = v - c;
        if (tid == 31) s_misc[0] = v;               // A
    }
    __syncthreads();
    const int A = s_misc[0];
    const int U = A * PJ;
    const int r0 = range_start(b, U, G), r1 = range_start(b + 1, U, G);
    const int n13 = r1 - r0;
    const int a_first = r0 / PJ;
    const int q0 = r0 >> 2;                        // first W2 group of the share (global index)
    const bool tmode = TILE || A * KP <= kTileMaxAK;   // all CTAs agree: A comes from the same routing
    // tile mode: CTA b < 80 owns output tile b over every (segment, K part)
    const int n_chunks = (tmode && b < kColTiles) ? (A * KP + kTSlots - 1) / kTSlots : 0;
    uint16_t *const hwg = reinterpret_cast<uint16_t *>(args.part);   // tile mode: HW[a][8 tokens][I]
    if (tid < S && s_ids[tid] >= 0) {
        const int e = s_ids[tid];
        const int a = wpre[e >> 5] + __popc(bitmap[e >> 5] & ((1u << (e & 31)) - 1u));
        act[a] = e;
        atomicOr(&tm[a], 1u << (tid / k));
    }
    // group q's HW rows are ready once the epilogue has finished each of its
    // owned pieces (one arrival each); each barrier completes one phase
    if (n13 > 0 && tid < ((r1 - 1) >> 2) + 1 - q0) {
        const int gq = q0 + tid;
        mbar_init(&hw_full[tid], min(4 * gq + 4, r1) - max(4 * gq, r0));
    }
    __syncthreads();
    if (tid == 0) stamp(2);

    if (warp == kProducer) {
        // ================================ producer ================================
        OpWalker wk;
        wk.init(r0, r1);
        int piece, gq, hh;
        for (int kk = 0;; ++kk) {
            // tile mode: the share's pieces, then the W2 tile chunks
            if (tmode) {
                if (kk >= n13 + n_chunks) break;
                piece = kk < n13 ? kk : -1;
                gq = kk - n13;
            } else if (!wk.next(piece, gq, hh)) {
                break;
            }
            const int s = kk % kStages;
            const uint32_t ph = (kk / kStages) & 1;
            int freed = 0;
            if (lane == 0) freed = mbar_wait_bounded(&empty[s], ph ^ 1, tmo) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, freed, 0)) {
                if (lane == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                break;
            }
            uint8_t *dst = ring + s * kStageBytes;
            if (lane == 0) {
                if (piece >= 0) {
                    const int u = r0 + piece, a = u / PJ, j = u - a * PJ;
                    const int64_t gp = static_cast<int64_t>(act[a]) * PJ + j;     // prepared piece
                    mbar_arrive_expect_tx(&full[s], kPieceQ + kMeta13);
                    bulk_load(dst, reinterpret_cast<const uint8_t *>(args.w13_q) + gp * kPieceQ, kPieceQ, &full[s]);
                    bulk_load(dst + kPieceQ, args.w13_meta + gp * kMeta13, kMeta13, &full[s]);
                } else if (tmode) {
                    // chunk gq: (segment, K part) pairs kTSlots * gq .. of tile b
                    const int p0 = kTSlots * gq, np = min(kTSlots, A * KP - p0);
                    mbar_arrive_expect_tx(&full[s], np * (kW2TileKK * 128 + 5 * 32 * MB));
                    for (int sl = 0; sl < np; ++sl) {
                        const int a = (p0 + sl) / KP, kp = p0 + sl - a * KP;
                        const int tile = (act[a] * KP + kp) * kColTiles + b;
                        tma_load_2d(dst + sl * kTQSlot, &t1q, &full[s], 0, tile * kW2TileKK);
                        tma_load_2d(dst + kTMetaOff + sl * kTMetaSlot, &t1m, &full[s], 0, tile * 5);
                    }
                } else {
                    const int a = (4 * gq) / PJ, gg = (4 * gq - a * PJ) >> 2;
                    const int lo = max(4 * gq, r0) - 4 * gq, hi = min(4 * gq + 4, r1) - 4 * gq;
                    const int tile0 = (act[a] * KP + gg / 5) * kColTiles + kUnitTiles * hh;
                    const int row0 = 4 * (gg % 5);
                    mbar_arrive_expect_tx(&full[s], (hi - lo) * kRowBlock + kUnitTiles * 32 * MB);
                    for (int r = lo; r < hi; ++r) tma_load_3d(dst + r * kRowBlock, &tq, &full[s], 0, row0 + r, tile0);
                    tma_load_3d(dst + kUnitQ, &tm_map, &full[s], 0, gg % 5, tile0);
                }
            }
            __syncwarp();
        }
        return;
    }

    if (warp >= kEpi) {
        // ================================ epilogue ================================
        const int e0 = warp - kEpi;
        // Contributors of every token for the final sum, while the first
        // pieces are in flight: CTA c contributes to token t when its share
        // holds a piece of a segment routed from t (a share spans at most two
        // segments). One ballot per (token, 32 CTAs).
        for (int w = e0; w < 8 && !tmode; w += 2) {
            const int c = 32 * w + lane;
            uint32_t m = 0;
            if (c < G) {
                const int c_lo = range_start(c, U, G), c_hi = range_start(c + 1, U, G);
                if (c_lo < c_hi) m = tm[c_lo / PJ] | tm[(c_hi - 1) / PJ];
            }
            for (int tok = 0; tok < M; ++tok) {
                const uint32_t word = __ballot_sync(0xffffffffu, m >> tok & 1);
                if (lane == 0) cm[tok * 8 + w] = word;
            }
        }
        named_barrier_sync(kBarE, 64);
        for (int tok = e0; tok < M && !tmode; tok += 2) {
            const uint32_t w = lane < 8 ? cm[tok * 8 + lane] : 0u;
            const int c = __popc(w);
            int v = c;
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += y;
            }
            int pos = v - c;
            for (uint32_t rest = w; rest; rest &= rest - 1)
                clist[tok * 256 + pos++] = static_cast<int16_t>(lane * 32 + __ffs(rest) - 1);
            if (lane == 7) cnt[tok] = v;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_count(lists_ready, 1);

        float *hb = hbuf + e0 * 64;                // [8 tokens][8 columns]
        int cur_a = -1;
        float wsum = 0.f;                          // lane < M: token lane's router weight on the segment
        for (int i = e0; i < n13; i += 2) {
            const int u = r0 + i, a = u / PJ, j = u - a * PJ;
            if (a != cur_a) {
                cur_a = a;
                const int e = act[a];
                wsum = 0.f;
                if (lane < M && (tm[a] >> lane & 1))
                    for (int q = 0; q < k; ++q)
                        if (s_ids[lane * k + q] == e) wsum += s_w[lane * k + q];
            }
            const int rslot = i % kSlots;
            if (!mbar_wait_bounded(&red_full[rslot], (i / kSlots) & 1, tmo)) {
                set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                return;
            }
            const float *rs = red + rslot * (kCW * 32 * 4);
            float4 sum = *reinterpret_cast<const float4 *>(rs + lane * 4);
#pragma unroll
            for (int w = 1; w < kCW; ++w) {
                const float4 v = *reinterpret_cast<const float4 *>(rs + (w * 32 + lane) * 4);
                sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
            }
            // lane (g, t): gate of column g for tokens 2t, 2t+1 in x, y; up in z, w
            hb[(2 * t) * 8 + g] = silu_f(sum.x) * sum.z;
            hb[(2 * t + 1) * 8 + g] = silu_f(sum.y) * sum.w;
            __syncwarp();
            if (lane == 0) mbar_arrive_count(&red_empty[rslot], 1);
            if (lane < 8) {
                // token row `lane`, chunk j (k rows 8j..8j+7) in MMA fragment
                // order: columns 0,4,1,5,2,6,3,7
                const float wv = lane < M ? wsum : 0.f;
                uint32_t pk[4];
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    pk[c] = static_cast<uint32_t>(f2h_bits(wv * hb[lane * 8 + c])) |
                            (static_cast<uint32_t>(f2h_bits(wv * hb[lane * 8 + c + 4])) << 16);
                if (tmode)
                    *reinterpret_cast<uint4 *>(hwg + (static_cast<int64_t>(a) * 8 + lane) * INTER + j * 8) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                else
                    *reinterpret_cast<uint4 *>(hw + (a - a_first) * 8 * HWR + lane * HWR + j * 16) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            __syncwarp();
            if (!tmode && lane == 0) mbar_arrive_count(&hw_full[(u >> 2) - q0], 1);
            if (i + 2 >= n13) stamp(9);
        }
        if (tmode) {
            // this warp's HW rows happen before the arrival (release), which
            // thread 0 acquires before its device-scope fence and its arrival
            // at the grid barrier
            __syncwarp();
            if (lane == 0) mbar_arrive_count(epi_done, 1);
        }
        return;
    }

    // ================================ consumers ================================
    // ok: results valid. dead: a wait for a copy ran out (later copy waits are
    // skipped). epi_dead: a wait for the epilogue ran out (later ones are
    // skipped). Waits on the epilogue only clear ok, so the ring is still
    // drained and no copy is in flight when the CTA leaves the op loop.
    bool ok = true, dead = false, epi_dead = false;
    int st_idx = 0;
    uint32_t st_ph = 0;
    auto wait_stage = [&]() {
        if (!dead && !mbar_wait_bounded(&full[st_idx], st_ph, tmo)) {
            ok = false;
            dead = true;
            set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
        }
    };
    auto next_stage = [&]() {
        if (++st_idx == kStages) {
            st_idx = 0;
            st_ph ^= 1;
        }
    };
    // x fragments of every token (row g of the N = 8 token block), this
    // warp's ten K groups: loaded once, used by every piece of the share
    uint4 xf[kGPW];
    {
        const uint16_t *xr = args.x + static_cast<int64_t>(g < M ? g : 0) * kHidden + warp * kGPW * kGroup + t * 8;
#pragma unroll
        for (int gi = 0; gi < kGPW; ++gi)
            xf[gi] = g < M ? permute_k8(ld_nc_v4(xr + gi * kGroup)) : make_uint4(0, 0, 0, 0);
    }
    const RowLane rl = row_lane(t);
    const int Qg = (g >> 1) | ((g & 1) << 2);
    // W2 accumulators: ten 32-column tiles per warp, two 16-column halves each
    float acc[kAcc][2][4];
#pragma unroll
    for (int s = 0; s < kAcc; ++s)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[s][h][v] = 0.f;

    OpWalker wk;
    wk.init(r0, r1);
    if (tmode) wk.q_end = wk.q;                    // tile mode: W13 pieces only
    int piece, gq, hh;
    while (wk.next(piece, gq, hh)) {
        if (piece >= 0) {
            // ---- W13 piece: this warp's ten K groups of the 16-row tile ----
            const int i = piece;
            wait_stage();
            if (i == 0 && tid == 0) stamp(3);
            const uint8_t *base = ring + st_idx * kStageBytes;
            float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int gi = 0; gi < kGPW; ++gi) {
                const int grp = warp * kGPW + gi;
                const uint2 q = *reinterpret_cast<const uint2 *>(base + ((grp * 4 + t) * kPieceCols + g) * 8);
                const MetaPair m = load_meta_pair_p<MB>(base + kPieceQ + (grp * kPieceCols + g) * 2 * MB);
                group_tile_mma(a4, q.x, q.y, m.zg2, m.zu2, half_bits_to_float(m.sg), half_bits_to_float(m.su),
                               xf[gi]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_count(&empty[st_idx], 1);
            next_stage();
            const int slot = i % kSlots;
            if (!epi_dead && !mbar_wait_bounded(&red_empty[slot], ((i / kSlots) & 1) ^ 1, tmo)) {
                ok = false;
                epi_dead = true;
                set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
            }
            *reinterpret_cast<float4 *>(red + slot * (kCW * 32 * 4) + (warp * 32 + lane) * 4) =
                make_float4(a4[0], a4[1], a4[2], a4[3]);
            __syncwarp();
            if (lane == 0) mbar_arrive_count(&red_full[slot], 1);
            if (i == n13 - 1 && tid == 0) stamp(4);
        } else {
            // ---- W2 unit: the group's owned rows x 40 column tiles ----
            const int a = (4 * gq) / PJ, gg = (4 * gq - a * PJ) >> 2;
            // the epilogue has finished every owned piece of the group
            if (!epi_dead && !mbar_wait_bounded(&hw_full[gq - q0], 0, tmo)) {
                ok = false;
                epi_dead = true;
                set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
            }
            wait_stage();
            const uint8_t *base = ring + st_idx * kStageBytes;
            const int lo = max(4 * gq, r0) - 4 * gq, hi = min(4 * gq + 4, r1) - 4 * gq;
            // B fragments of the owned word rows: token g, k rows t and t + 4
            const uint8_t *hgrp = hw + (a - a_first) * 8 * HWR + g * HWR + (4 * gg) * 16 + 4 * t;
            uint32_t hb[4];
#pragma unroll
            for (int r = 0; r < 4; ++r)
                hb[r] = (r >= lo && r < hi) ? *reinterpret_cast<const uint32_t *>(hgrp + r * 16) : 0u;
            if (hh == 0)
                w2_unit_rows<MB, 0>(acc, base, hb, lo, hi, warp, Qg, rl);
            else
                w2_unit_rows<MB, 1>(acc, base, hb, lo, hi, warp, Qg, rl);
            __syncwarp();
            if (lane == 0) mbar_arrive_count(&empty[st_idx], 1);
            next_stage();
        }
    }
    if (tid == 0) stamp(5);

    if (tmode) {
        // ---------------- tile mode: grid barrier, then W2 tiles ----------------
        if (tid == 0) {
            bool fine = mbar_wait_bounded(epi_done, 0, tmo);
            stamp(6);
            if ((args.debug_flags & 1) && b == 0) {
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 2 * tmo) sleep_ns(1000);
            }
            // release: the epilogue warps' HW stores are ordered before it by
            // their arrival on epi_done, which this thread acquired
            red_add_release_u64(args.gbar, 1ull);
            const uint64_t target = (epoch + 1) * static_cast<uint64_t>(G);
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire_gpu_u64(args.gbar) < target) {
                if (global_timer_ns() - t0 > tmo) {
                    fine = false;
                    break;
                }
                sleep_ns(20);
            }
            if (!fine) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
            s_misc[4] = fine ? 1 : 0;
            stamp(7);
        }
        named_barrier_sync(kBarC, kCThreads);
        if (n_chunks == 0) return;
        // W2 of tile b over every (segment, K part): items (pair, group) of
        // each chunk dealt over the warps; the HW B fragments of every item of
        // every chunk are loaded from L2 first, all in flight at once
        float tacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        constexpr int kItems = (kTSlots * 5 + kCW - 1) / kCW;   // 4 per chunk
        constexpr int kMaxChunks = (kTileMaxAK + kTSlots - 1) / kTSlots;
        uint4 xb[kMaxChunks][kItems];
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c)
#pragma unroll
            for (int x = 0; x < kItems; ++x) {
                const int it = warp + kCW * x, sl = it / 5, gg = it - sl * 5;
                const int pr = kTSlots * c + sl;
                xb[c][x] = make_uint4(0, 0, 0, 0);
                if (c < n_chunks && sl < kTSlots && pr < A * KP) {
                    const int a = pr / KP, kp = pr - a * KP;
                    xb[c][x] = __ldcg(reinterpret_cast<const uint4 *>(
                        hwg + (static_cast<int64_t>(a) * 8 + g) * INTER + (4 * (5 * kp + gg) + t) * 8));
                }
            }
#pragma unroll
        for (int c = 0; c < kMaxChunks; ++c) {
            if (c >= n_chunks) break;
            wait_stage();
            const uint8_t *base = ring + st_idx * kStageBytes;
            const int p0 = kTSlots * c, np = min(kTSlots, A * KP - p0);
#pragma unroll
            for (int x = 0; x < kItems; ++x) {
                const int it = warp + kCW * x, sl = it / 5, gg = it - sl * 5;
                if (sl >= np) continue;
                const int L = 4 * gg + t;
                const uint4 q = *reinterpret_cast<const uint4 *>(base + sl * kTQSlot + L * 128 + ((Qg ^ (L & 7)) << 4));
                const Meta4<MB> mt = meta4_of<MB>(load_meta4_raw<MB>(base + kTMetaOff + sl * kTMetaSlot + gg * 32 * MB + Qg * 4 * MB));
                group_tile_mma(tacc[0], q.x, q.y, mt.z2[0], mt.z2[1], half_bits_to_float(mt.s[0]),
                               half_bits_to_float(mt.s[1]), xb[c][x]);
                group_tile_mma(tacc[1], q.z, q.w, mt.z2[2], mt.z2[3], half_bits_to_float(mt.s[2]),
                               half_bits_to_float(mt.s[3]), xb[c][x]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_count(&empty[st_idx], 1);
            next_stage();
        }
        // the warps' partial tiles, summed in warp order. They go to the idle
        // W13 hand-off slots: the ring may still be read by slower warps (a
        // chunk can occupy any stage).
        float4 *tp = reinterpret_cast<float4 *>(red);               // [kCW warps][2 halves][32 lanes]
        static_assert(kSlots * kCW * 32 * 16 >= kCW * 2 * 32 * 16, "partial tiles fit the hand-off slots");
        tp[(warp * 2 + 0) * 32 + lane] = make_float4(tacc[0][0], tacc[0][1], tacc[0][2], tacc[0][3]);
        tp[(warp * 2 + 1) * 32 + lane] = make_float4(tacc[1][0], tacc[1][1], tacc[1][2], tacc[1][3]);
        named_barrier_sync(kBarC, kCThreads);
        if (warp < 2 && s_misc[4]) {
            const int hh = warp;
            float4 sum = tp[hh * 32 + lane];
            for (int w = 1; w < kCW; ++w) {
                const float4 v = tp[(w * 2 + hh) * 32 + lane];
                sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
            }
            const float vals[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int tok = 2 * t + (v & 1);
                const int col = 32 * b + 4 * Qg + 2 * hh + (v >> 1);
                if (tok < M) args.out[static_cast<int64_t>(tok) * kHidden + col] = f2h_bits(vals[v]);
            }
        }
        if (tid == 0) stamp(8);
        return;
    }

    // ---------------- partial output of this CTA ----------------
    // Lane (g, t) holds, per tile, columns 4Qg .. 4Qg+3 of tokens 2t and
    // 2t+1: one 16-byte store per token, a warp's stores are 128-byte rows.
    uint32_t cmask = 0;
    if (n13 > 0) cmask = tm[a_first] | tm[(r1 - 1) / PJ];
    float *P = args.part + static_cast<int64_t>(b) * M * kHidden;     // [M tokens][H]
    if (n13 > 0) {
#pragma unroll
        for (int s = 0; s < kAcc; ++s) {
            const int col = 32 * (kUnitTiles * (s / kTPW) + warp + kCW * (s % kTPW)) + 4 * Qg;
            if (cmask >> (2 * t) & 1)
                *reinterpret_cast<float4 *>(P + (2 * t) * kHidden + col) =
                    make_float4(acc[s][0][0], acc[s][0][2], acc[s][1][0], acc[s][1][2]);
            if (cmask >> (2 * t + 1) & 1)
                *reinterpret_cast<float4 *>(P + (2 * t + 1) * kHidden + col) =
                    make_float4(acc[s][0][1], acc[s][0][3], acc[s][1][1], acc[s][1][3]);
        }
    }

    // ---------------- grid barrier ----------------
    named_barrier_sync(kBarC, kCThreads);
    if (tid == 0) {
        stamp(6);
        if ((args.debug_flags & 1) && b == 0) {
            // test hook: arrive only after the other CTAs' wait has run out
            const uint64_t t0 = global_timer_ns();
            while (global_timer_ns() - t0 < 2 * tmo) sleep_ns(1000);
        }
        // release: the CTA's partial-output stores are ordered before it by
        // the barrier above
        red_add_release_u64(args.gbar, 1ull);
        const uint64_t target = (epoch + 1) * static_cast<uint64_t>(G);
        bool fine = true;
        const uint64_t t0 = global_timer_ns();
        while (ld_acquire_gpu_u64(args.gbar) < target) {
            if (global_timer_ns() - t0 > tmo) {
                fine = false;
                break;
            }
            sleep_ns(20);
        }
        // the contributor lists (epilogue warps) are complete
        if (!mbar_wait_bounded(lists_ready, 0, tmo)) fine = false;
        if (!fine) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
        s_misc[4] = fine ? 1 : 0;
        stamp(7);
    }
    named_barrier_sync(kBarC, kCThreads);

    // ---------------- final sum over the contributing CTAs ----------------
    // Work items (token, 128-column chunk), an equal share per CTA; each
    // item's contributors are split over `nparts` warps (strided), each lane
    // four columns, 8 loads of a lane in flight at once; the parts are then
    // added in a fixed order.
    float4 *partial = reinterpret_cast<float4 *>(ring);              // [kCW warps][32] (the ring is free)
    constexpr int kChunks = kHidden / 128;                          // 20
    const int n_items = M * kChunks;
    const int i0 = range_start(b, n_items, G), n_it = range_start(b + 1, n_items, G) - i0;
    const int nparts = n_it > 0 ? kCW / n_it : 0;
    if (warp < n_it * nparts) {
        const int item = i0 + warp / nparts, part = warp % nparts;
        const int tok = item / kChunks, ch = item - tok * kChunks;
        const int n = cnt[tok];
        const int16_t *lst = clist + tok * 256;
        const float4 *src = reinterpret_cast<const float4 *>(args.part + tok * kHidden + ch * 128) + lane;
        const int64_t cstride = static_cast<int64_t>(M) * kHidden / 4;     // in float4
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int qb = part; qb < n; qb += 8 * nparts) {
            float4 v[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int q = qb + r * nparts;
                v[r] = q < n ? __ldcg(src + lst[q] * cstride) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                sum.x += v[r].x; sum.y += v[r].y; sum.z += v[r].z; sum.w += v[r].w;
            }
        }
        partial[warp * 32 + lane] = sum;
    }
    named_barrier_sync(kBarC, kCThreads);
    if (warp < n_it && s_misc[4]) {
        const int item = i0 + warp;
        const int tok = item / kChunks, ch = item - tok * kChunks;
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int p = 0; p < nparts; ++p) {
            const float4 v = partial[(warp * nparts + p) * 32 + lane];
            sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
        }
        const uint32_t lo = static_cast<uint32_t>(f2h_bits(sum.x)) | (static_cast<uint32_t>(f2h_bits(sum.y)) << 16);
        const uint32_t hi = static_cast<uint32_t>(f2h_bits(sum.z)) | (static_cast<uint32_t>(f2h_bits(sum.w)) << 16);
        *reinterpret_cast<uint2 *>(args.out + static_cast<int64_t>(tok) * kHidden + ch * 128 + lane * 4) =
            make_uint2(lo, hi);
    }
    if (tid == 0) stamp(8);
    (void)ok;
}

int sliced_smem_bytes(int inter) { return layout(inter).total + 1024; }

awq_status launch_sliced(int mb, int sms, cudaStream_t st, const CUtensorMap &tq, const CUtensorMap &tm,
                         const CUtensorMap &t1q, const CUtensorMap &t1m, const SlicedArgs &a)
{
    const int smem = sliced_smem_bytes(a.inter);
    void (*kernel)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, SlicedArgs);
    // at most M * top_k active experts: tile mode is certain below the bound
    const bool tile = static_cast<int64_t>(a.M) * a.top_k * (a.inter / 160) <= kTileMaxAK;
    if (a.inter == 160 && tile)
        kernel = mb == 4 ? sliced_layer_kernel<4, 160, true> : sliced_layer_kernel<3, 160, true>;
    else if (a.inter == 160)
        kernel = mb == 4 ? sliced_layer_kernel<4, 160, false> : sliced_layer_kernel<3, 160, false>;
    else
        kernel = mb == 4 ? sliced_layer_kernel<4, 640, false> : sliced_layer_kernel<3, 640, false>;
    awq_status r = set_smem(kernel, smem);
    if (r) return r;
    return launch_ex(kernel, dim3(sms), dim3(kThreads), smem, 1, true, st, tq, tm, t1q, t1m, a);
}

}  // namespace awq
