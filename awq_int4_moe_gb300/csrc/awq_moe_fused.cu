// The whole expert stage of one decode layer call (routing, W13 + SwiGLU,
// W2 + router-weighted top-k reduction) as ONE persistent kernel, for up to
// 16 tokens.
//
// Source of the computation: 1Cat-vLLM #520 "Narrow Qwen3.8 AWQ active
// grouped decode", Purpose and Implementation (active-expert segments,
// offsets-based scheduling, one pass per stage, grouped-active exact W2
// reduction); 1Cat-vLLM #522 "Coalesce AWQ QPN W13 compact metadata loads and
// enable compact metadata by default", Purpose (3-byte {fp16 scale, u8 zero}
// records read as aligned 32-bit words).
//
// Prologue. Every CTA rebuilds the routing it needs from the <= 256 slots in
// shared memory: a bitmap of the active experts (segment a is the a-th set
// bit, so segments come in ascending expert order) and, per segment, the mask
// of tokens routed to it. No sort is needed because this kernel never exposes
// sorted slots. Given router logits instead of top-k ids, the CTA first runs
// the router itself (one warp per token; 1Cat-vLLM #12 "Add opt-in
// native-g32 AWQ QPN M1 dispatch", Purpose and stack: int32 top-10 ids and
// fp32 router weights are the stage's inputs).
//
// Schedule. One CTA per SM (grid = SM count). Each CTA takes a contiguous,
// equal share of two flat work lists, whose units are single contiguous
// blocks of the prepared banks (awq_moe_prepare_weights):
//   W13 pieces (segment a, 8 gate + 8 up columns, whole K)                 25 KB
//   W2  units  (256-column output group, segment a, 160-row K part)          25 KB
// A producer warp streams them (bulk copies for W13, 128-byte swizzled TMA
// tiles for W2) into a ring of shared-memory stages; the consumer warps (16
// for one 8-token block, 10 for two) dequantise in registers and run m16n8k16
// tensor-core MMAs with the weights on the M side and tokens on the N side.
//
// W13. A piece is one 16-row tile (rows 0-7 gate, 8-15 up) over the whole K,
// so it needs no cross-CTA reduction: each consumer warp accumulates its
// share of the 80 K groups with the segment's x fragments held in registers
// (loaded once per segment), and the epilogue warps (slot e of the two hand-off
// slots to epilogue warp e) sum the warps' tiles in a fixed order, apply
// SwiGLU (a lane holds the gate and the up value of the same column and
// token) and store the router-weighted activations
// HW[a][t][:] = (sum of the router weights of token t's slots on segment a) *
// h[a][t][:], each 8-column octet in the MMA fragment order of the W2 K
// permutation. Each epilogue warp announces its finished pieces once, with a
// release.
//
// W2, flat mode. Warp w owns output tile w % 8 of the unit's 256-column group
// (one 16-column half of it with 16 warps). Once every W13 piece of the grid
// is announced, the producer copies each unit's activation rows into the
// unit's stage, counted by the same barrier as its weights. All segments of
// a group accumulate in registers with tokens as the MMA N dimension. A group
// that lies inside one CTA's share is written directly; for a group split
// between CTAs every part publishes a partial, and once all are in, each part
// sums its own slice of the columns over the partials in CTA order, so
// results are deterministic with no atomics on data.
//
// W2, tile mode (few active experts: 10 A KP <= grid). CTA c < 80 owns the
// 32-column output tile c over every segment, four segments per unit; the
// units' activations are copied at once when the W13 pieces are all
// announced, the warps wait for all units and expand every group in one
// pass, and add their partials in shared memory in a fixed order. No
// cross-CTA exchange after the hand-over.
//
// NVFP4 banks (MB = 2: prepared 2-byte records, the E4M3 scales of the two
// 16-k blocks of a group of 32): both modes (tile-mode units of 3 segments,
// whose stages also hold the residue rows). A lane's packed word
// covers 8 consecutive k of one block, so it takes that block's scale; each
// weight enters the MMA as the exact fp16 product e2m1 * scale * 2^-7, the
// W13 sums are multiplied by 2^7 * the expert's W13 global scale before
// SwiGLU, the W2 global scale is folded into the expert's HW rows, and the
// W2 outputs are multiplied by 2^7. HW goes out as fp16 plus its fp16
// residue (a second plane) and W2 multiplies both: one fp16 rounding of HW is
// too coarse for NVFP4 layers (about one output in 20,000 then falls outside
// the stage's tolerance).
//
// The cross-CTA waits (W2 on all W13 pieces, split groups on their parts) are
// bounded by a timeout; the grid is one CTA per SM, launched cooperatively so
// that all CTAs are resident at once. Two counter
// sets alternate between calls (a per-CTA sense word says which is current);
// each call zeroes the other one, so a zero-filled workspace stays usable
// call after call, a timed-out call included.
#include <cuda_fp16.h>

#include "awq_dequant.cuh"
#include "awq_launch.cuh"
#include "awq_moe_kernels.cuh"
#include "awq_nvfp4.cuh"
#include "awq_ptx.cuh"
#include "awq_router.cuh"
#include "awq_split.cuh"

namespace awq {

namespace {

// Consumer warps: 16 for one 8-token block (NT = 1), 10 for two. In W13 a
// warp takes 80 / CW consecutive groups of a piece, fully unrolled with its x
// fragments in registers; more warps per scheduler hide more of the
// dequantise -> MMA latency. In W2 warps 0-7 own the unit's eight tiles; with
// 16 warps, warps 8-15 take the second 16-column half of the same tiles.
__host__ __device__ constexpr int consumer_warps(int NT) { return NT == 1 ? 16 : 10; }
// Epilogue warps: one warp cannot keep up with the hand-offs (16 consumer
// warps, or 10 with two token blocks), so two share them (warp e takes the
// pieces of hand-off slot e).
__host__ __device__ constexpr int epilogue_warps(int) { return 2; }
__host__ __device__ constexpr int fused_threads(int NT) { return (consumer_warps(NT) + 1 + epilogue_warps(NT)) * 32; }
constexpr int kMaxSlotsF = kFusedMaxTokens * kMaxTopK;           // 256
static_assert(kGroups13 % consumer_warps(1) == 0 && kGroups13 % consumer_warps(2) == 0, "groups split evenly");
// W2 unit: 8 consecutive 32-column tiles (warp w <-> tile w) of one segment,
// one 160-row K part (5 groups): 160 lines [tile][20 rows][32 words] + 40
// metadata rows [tile][group][32 records].
constexpr int kW2Tiles = kFusedW2Tiles;
constexpr int kW2KK = 20;
constexpr int kW2Groups = 5;
constexpr int kW2Q = kW2Tiles * kW2KK * 128;                        // 20 KB
constexpr int kColGroups = kHidden / (32 * kW2Tiles);               // 10
constexpr int kBarCompute = 1;
// W2 activations of one unit: MP rows x 160 fp16 (320 B rows: 20 chunks,
// bank-conflict free), after the unit's weights in the same stage.
constexpr int kHwRow = kW2Groups * kGroup * 2;                      // 320
constexpr int kHwOff = kW2Q + kW2Tiles * kW2Groups * 32 * 4;        // 25600

__host__ __device__ constexpr int round_up(int v, int a) { return (v + a - 1) / a * a; }
// One ring stage holds a W13 piece or a W2 unit with its activations; a
// multiple of 1 KB (the 128-byte swizzle repeats every 1 KB).
// NVFP4 banks (MB = 2) carry the fp16 residue of HW as a second plane of
// activation rows after the first, so their stages are larger and fewer.
__host__ __device__ constexpr int hw_planes(int MB) { return MB == 2 ? 2 : 1; }
__host__ __device__ constexpr int fused_stage_bytes(int NT, int MB = 4)
{
    return round_up(kHwOff + hw_planes(MB) * 8 * NT * kHwRow, 1024);
}
static_assert(kPieceQ + piece_meta_bytes(4) <= fused_stage_bytes(1), "W13 piece fits");
__host__ __device__ constexpr int fused_stages(int NT, int MB = 4)
{
    return MB == 2 ? (NT == 1 ? 6 : 5) : (NT == 1 ? 7 : 6);
}
// Tile mode (few active experts, one token block): CTA c < 80 owns 32-column
// output tile c over every segment. A unit is (tile_segs(MB) segments, 160-row
// K part): 4 segments, or 3 for NVFP4 banks, whose stages also hold the
// residue plane. Its stage holds per segment s the tile's 20 lines (1 KB-
// aligned 3 KB slot at 3072 s), 5 metadata rows (at tile_meta + 640 s) and MP
// activation rows (at tile_hw + 8 * 320 s; NVFP4: their residue rows after all
// segments' rows).
constexpr int kTSegs = 4;                      // segment slots of the consumer warps
constexpr int kTQSlot = 3072;
constexpr int kTMetaSlot = 640;
__host__ __device__ constexpr int tile_segs(int MB) { return MB == 2 ? 3 : kTSegs; }
__host__ __device__ constexpr int tile_meta(int MB) { return tile_segs(MB) * kTQSlot; }       // 12288 (9216)
__host__ __device__ constexpr int tile_hw(int MB) { return tile_meta(MB) + tile_segs(MB) * kTMetaSlot; }   // 14848 (11136)
static_assert(tile_hw(4) + kTSegs * 8 * kHwRow <= fused_stage_bytes(1), "tile-mode unit fits");
static_assert(tile_hw(2) + hw_planes(2) * tile_segs(2) * 8 * kHwRow <= fused_stage_bytes(1, 2), "NVFP4 tile-mode unit fits");
// A CTA's tile-mode units are all resident at once (with its at most 2 W13
// pieces: 10 A KP <= grid bounds the pieces per CTA by 2 at I = 160 and 640).
constexpr int kTMaxUnits = 4;
static_assert(kTMaxUnits + 2 <= fused_stages(1) && kTMaxUnits + 2 <= fused_stages(1, 2),
              "tile-mode units and pieces fit the ring together");
static_assert(kW2Tiles <= consumer_warps(2), "one consumer warp per W2 tile");

struct Layout {
    int bars, red, hbuf, route, total;
};

// One hand-off slot: every consumer warp's W13 tile for one piece
// ([warp][n NT][lane][4] floats); two slots alternate.
__host__ __device__ constexpr int red_slot_bytes(int NT) { return consumer_warps(NT) * NT * 32 * 16; }

// Shared-memory layout (offsets from the 1024-aligned base). Stage s starts at
// s * fused_stage_bytes(NT, MB).
__host__ __device__ inline Layout fused_layout(int NT, int MB = 4)
{
    Layout L;
    const int stages = fused_stages(NT, MB);
    L.bars = stages * fused_stage_bytes(NT, MB);
    L.red = round_up(L.bars + (2 * stages + 4) * 8, 128);
    L.hbuf = L.red + 2 * red_slot_bytes(NT);
    L.route = L.hbuf + epilogue_warps(NT) * 16 * kPieceCols * 4;   // one SwiGLU buffer per epilogue warp
    // s_ids[256], s_w[256], act[256], tm[256], bitmap[32], wpre[32], misc[16]
    L.total = L.route + (4 * kMaxSlotsF + 32 + 32 + 16) * 4;
    return L;
}

__device__ __forceinline__ void red_add_release(int32_t *p, int v)
{
    asm volatile("red.add.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Release pattern for several counters: one fence, then relaxed adds.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void red_add_relaxed(int32_t *p, int v)
{
    asm volatile("red.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded spin until *p >= target (acquire).
__device__ __forceinline__ bool wait_counter(const int32_t *p, int target, uint64_t limit_ns)
{
    if (ld_acquire_gpu(p) >= target) return true;
    const uint64_t t0 = global_timer_ns();
    while (ld_acquire_gpu(p) < target) {
        if (global_timer_ns() - t0 > limit_ns) return false;
        sleep_ns(32);
    }
    return true;
}

// j-th (0-based) set bit of a token mask, or -1.
__device__ __forceinline__ int nth_token(uint32_t mask, int j)
{
    if (j >= __popc(mask)) return -1;
    return static_cast<int>(__fns(mask, 0, j + 1));
}

}  // namespace

template <int MB, int NT>
__global__ void __launch_bounds__(fused_threads(NT), 1)
fused_layer_kernel(const __grid_constant__ CUtensorMap t2q, const __grid_constant__ CUtensorMap t2m,
                   const __grid_constant__ CUtensorMap t2q1, const __grid_constant__ CUtensorMap t2m1,
                   FusedArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    constexpr int kStages = fused_stages(NT, MB);
    constexpr int kStageBytes = fused_stage_bytes(NT, MB);
    constexpr int MP = 8 * NT;                     // token rows of HW per segment
    constexpr int kMeta13 = piece_meta_bytes(MB);
    constexpr int kConsumerWarps = consumer_warps(NT);
    constexpr int kConsumerThreads = kConsumerWarps * 32;
    constexpr int kProducerWarp = kConsumerWarps;
    constexpr int kEpilogueWarp = kConsumerWarps + 1;          // first epilogue warp
    constexpr int kEpilogueWarps = epilogue_warps(NT);
    constexpr int kFusedThreads = fused_threads(NT);
    constexpr int kGroupsPerWarp = kGroups13 / kConsumerWarps;     // W13 groups of a warp
    constexpr int kW2Split = kConsumerWarps / kW2Tiles;            // warps per W2 tile (1 or 2)
    static_assert(kW2Split == 1 || kW2Split == 2, "one or two warps per W2 tile");
    const int M = args.M, k = args.top_k, E = args.num_experts, I = args.inter;
    const int PJ = I / kPieceCols, KP = I / 160;   // W13 pieces per expert, W2 K parts
    const Layout Lo = fused_layout(NT, MB);
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lo.bars);
    uint64_t *empty = full + kStages;
    uint64_t *red_full = empty + kStages;          // [2] consumer warps -> epilogue
    uint64_t *red_empty = red_full + 2;            // [2] epilogue -> consumer warps
    float *red = reinterpret_cast<float *>(smem + Lo.red);
    float *hbuf = reinterpret_cast<float *>(smem + Lo.hbuf);   // [epilogue warp][MP][8] SwiGLU of one piece
    int32_t *s_ids = reinterpret_cast<int32_t *>(smem + Lo.route);     // expert of slot, -1 if invalid
    float *s_w = reinterpret_cast<float *>(s_ids + kMaxSlotsF);       // router weight of slot
    int32_t *act = reinterpret_cast<int32_t *>(s_w + kMaxSlotsF);     // expert of segment
    uint32_t *tm = reinterpret_cast<uint32_t *>(act + kMaxSlotsF);    // token mask of segment
    uint32_t *bitmap = tm + kMaxSlotsF;                               // active experts
    int32_t *wpre = reinterpret_cast<int32_t *>(bitmap + 32);         // set bits before word
    int32_t *s_misc = wpre + 32;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int G = gridDim.x, b = blockIdx.x;
    const int S = M * k;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&red_full[s], kConsumerWarps);
            mbar_init(&red_empty[s], 1);
        }
        fence_barrier_init();
        prefetch_tmap(&t2q);
        prefetch_tmap(&t2m);
        prefetch_tmap(&t2q1);
        prefetch_tmap(&t2m1);
    }
    if (tid < 32) bitmap[tid] = 0;
    for (int i = tid; i < kMaxSlotsF; i += kFusedThreads) tm[i] = 0;
    grid_dependency_wait();
    grid_launch_dependents();
    if (tid == kFusedThreads - 1) s_misc[5] = args.sense[b];

    // ---------------- routing in shared memory ----------------
    if (args.logits) {
        // the router itself: one warp per token, every CTA alike
        for (int tok = warp; tok < M; tok += kFusedThreads / 32)
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
    if (tid < S && s_ids[tid] >= 0) {
        const int e = s_ids[tid];
        const int a = wpre[e >> 5] + __popc(bitmap[e >> 5] & ((1u << (e & 31)) - 1u));
        act[a] = e;
        atomicOr(&tm[a], 1u << (tid / k));
    }
    __syncthreads();

    // Counter set of this call. Every CTA flips its sense word once per call,
    // so all CTAs agree on it; the set of the previous call is idle and is
    // zeroed here for the next call (no end-of-call count is needed).
    const int sp = s_misc[5] & 1;
    int32_t *const done13 = args.sync + sp;                 // finished W13 pieces
    int32_t *const cnt2 = args.cnt2 + sp * kColGroups;      // published W2 partials per group
    if (tid == kFusedThreads - 1) {
        args.sense[b] = sp ^ 1;
        if (b == 0) {
            args.sync[sp ^ 1] = 0;
            for (int c = 0; c < kColGroups; ++c) args.cnt2[(sp ^ 1) * kColGroups + c] = 0;
        }
    }

    const int A = s_misc[0];
    const int U13 = A * PJ;
    // Tile mode when the flat W2 list would give every CTA at most one unit:
    // then each split column group would gather 10+ partials from as many CTAs,
    // while 80 tile owners need no cross-CTA exchange at all.
    constexpr int kTSegsU = tile_segs(MB);         // segments per tile-mode unit
    constexpr int kTMeta = tile_meta(MB), kTHw = tile_hw(MB);
    const bool tmode = NT == 1 && kColGroups * A * KP <= G && G >= kColTiles &&
                       (A + kTSegsU - 1) / kTSegsU * KP <= kTMaxUnits;
    const int U2 = tmode ? 0 : kColGroups * A * KP;
    const int r13b = range_start(b, U13, G), r13e = range_start(b + 1, U13, G);
    const int r2b = range_start(b, U2, G), r2e = range_start(b + 1, U2, G);
    const int n13 = r13e - r13b;
    const int n2 = tmode ? (b < kColTiles ? (A + kTSegsU - 1) / kTSegsU * KP : 0) : r2e - r2b;
    const uint64_t tmo = args.timeout_ns;
    const int per_c = A * KP;                      // W2 units per 256-column group

    if (warp == kProducerWarp) {
        // ================================ producer ================================
        // W13 pieces, then W2 units (weights as soon as a stage is free). A W2
        // unit's stage also receives its activation rows HW[a][0..MP)[kp part],
        // one bulk copy per row, counted by the same barrier; those copies go
        // out once every W13 piece of the grid is announced, while the warp
        // waits for stages or after its last weight copy.
        int w2_issued = 0, hw_next = 0;
        bool hw_ready = false, live = true;
        // issue the pending activation copies; false if the wait ran out
        auto pump_hw = [&](bool block) -> bool {
            if (hw_next >= w2_issued) return true;
            if (!hw_ready) {
                int ready = 0;
                if (lane == 0) ready = block ? (wait_counter(done13, U13, tmo) ? 1 : 2) : (ld_acquire_gpu(done13) >= U13);
                ready = __shfl_sync(0xffffffffu, ready, 0);
                if (ready == 2) {
                    if (lane == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                    return false;
                }
                if (!ready) return true;
                hw_ready = true;
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            for (; hw_next < w2_issued; ++hw_next) {
                const int i = n13 + hw_next;
                uint8_t *stage = ring + (i % kStages) * kStageBytes;
                // With one K part (I = 160) a segment's MP rows, and consecutive
                // segments, are contiguous in HW: one copy per unit (tile mode:
                // every pending unit at once, one lane each). With four, each
                // row's 160-column part is a separate 320-byte copy.
                if (tmode && KP == 1) {
                    const int u = hw_next + lane;
                    if (u < w2_issued) {
                        const int nseg = min(kTSegsU, A - u * kTSegsU);
                        const int iu = n13 + u;
                        const int64_t off = static_cast<int64_t>(u * kTSegsU) * MP * I;
                        uint8_t *dst = ring + (iu % kStages) * kStageBytes + kTHw;
                        bulk_load(dst, args.hw + off, nseg * MP * kHwRow, &full[iu % kStages]);
                        if (MB == 2)       // NVFP4: the residue rows after all segments' rows
                            bulk_load(dst + kTSegsU * MP * kHwRow, args.hw_lo + off, nseg * MP * kHwRow,
                                      &full[iu % kStages]);
                    }
                    hw_next = w2_issued;
                    break;
                }
                if (tmode) {
                    const int sgrp = hw_next / KP, kp = hw_next - sgrp * KP;
                    const int nseg = min(kTSegsU, A - sgrp * kTSegsU);
                    const int64_t off = static_cast<int64_t>(sgrp * kTSegsU) * MP * I + kp * 160;
                    for (int r = lane; r < nseg * MP; r += 32) {
                        bulk_load(stage + kTHw + r * kHwRow, args.hw + off + static_cast<int64_t>(r) * I, kHwRow,
                                  &full[i % kStages]);
                        if (MB == 2)
                            bulk_load(stage + kTHw + (kTSegsU * MP + r) * kHwRow,
                                      args.hw_lo + off + static_cast<int64_t>(r) * I, kHwRow, &full[i % kStages]);
                    }
                } else {
                    const int rem = (r2b + hw_next) % per_c;
                    const int a = rem / KP, kp = rem - a * KP;
                    const int64_t off = static_cast<int64_t>(a) * MP * I + kp * 160;
                    const uint16_t *src = args.hw + off;
                    if (KP == 1) {
                        if (lane == 0) bulk_load(stage + kHwOff, src, MP * kHwRow, &full[i % kStages]);
                        if (MB == 2 && lane == 1)      // NVFP4: the residue rows after them
                            bulk_load(stage + kHwOff + MP * kHwRow, args.hw_lo + off, MP * kHwRow, &full[i % kStages]);
                    } else if (lane < MP) {
                        bulk_load(stage + kHwOff + lane * kHwRow, src + static_cast<int64_t>(lane) * I, kHwRow,
                                  &full[i % kStages]);
                        if (MB == 2)
                            bulk_load(stage + kHwOff + (MP + lane) * kHwRow,
                                      args.hw_lo + off + static_cast<int64_t>(lane) * I, kHwRow, &full[i % kStages]);
                    }
                }
            }
            return true;
        };
        for (int i = 0; i < n13 + n2 && live; ++i) {
            const int s = i % kStages;
            const uint32_t ph = (i / kStages) & 1;
            const uint64_t t0 = global_timer_ns();
            while (true) {                                   // wait for a free stage
                int freed = 0;
                if (lane == 0) freed = mbar_try_wait(&empty[s], ph ^ 1) ? 1 : 0;
                if (__shfl_sync(0xffffffffu, freed, 0)) break;
                if (!pump_hw(false) || global_timer_ns() - t0 > tmo) {
                    if (lane == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                    live = false;
                    break;
                }
            }
            if (!live) break;
            uint8_t *dst = ring + s * kStageBytes;
            if (lane == 0) {
                if (i < n13) {
                    const int u = r13b + i;
                    const int a = u / PJ, j = u - a * PJ;
                    const int64_t gp = static_cast<int64_t>(act[a]) * PJ + j;   // prepared piece
                    mbar_arrive_expect_tx(&full[s], kPieceQ + kMeta13);
                    bulk_load(dst, reinterpret_cast<const uint8_t *>(args.w13_q) + gp * kPieceQ, kPieceQ, &full[s]);
                    bulk_load(dst + kPieceQ, args.w13_meta + gp * kMeta13, kMeta13, &full[s]);
                } else if (tmode) {
                    const int u = i - n13;
                    const int sgrp = u / KP, kp = u - sgrp * KP;
                    const int nseg = min(kTSegsU, A - sgrp * kTSegsU);
                    mbar_arrive_expect_tx(&full[s],
                                          nseg * (kW2KK * 128 + kW2Groups * 32 * MB + hw_planes(MB) * MP * kHwRow));
                    for (int sg = 0; sg < nseg; ++sg) {
                        const int tile = (act[sgrp * kTSegsU + sg] * KP + kp) * kColTiles + b;
                        tma_load_2d(dst + sg * kTQSlot, &t2q1, &full[s], 0, tile * kW2KK);
                        tma_load_2d(dst + kTMeta + sg * kTMetaSlot, &t2m1, &full[s], 0, tile * kW2Groups);
                    }
                } else {
                    const int v = r2b + (i - n13);
                    const int cg = v / per_c, rem = v - cg * per_c;
                    const int a = rem / KP, kp = rem - a * KP;
                    const int tile0 = (act[a] * KP + kp) * kColTiles + cg * kW2Tiles;   // prepared block
                    mbar_arrive_expect_tx(&full[s], kW2Q + kW2Tiles * kW2Groups * 32 * MB + hw_planes(MB) * MP * kHwRow);
                    tma_load_2d(dst, &t2q, &full[s], 0, tile0 * kW2KK);
                    tma_load_2d(dst + kW2Q, &t2m, &full[s], 0, tile0 * kW2Groups);
                }
            }
            __syncwarp();
            if (i >= n13) ++w2_issued;
            live = pump_hw(false);
        }
        while (live && hw_next < n2) live = pump_hw(true);
        return;
    }

    if (warp >= kEpilogueWarp) {
        // ================================ epilogue ================================
        hbuf += (warp - kEpilogueWarp) * 16 * kPieceCols;     // this warp's own buffer
        // Finishes the CTA's W13 pieces in order, one hand-off slot at a time
        // (with two epilogue warps, warp e takes the pieces of slot e).
        int finished = 0;
        int cur_a = -1;
        float wsum = 0.f;                          // lane t < MP: token t's router weight on the segment
        float g13 = 1.f;                           // NVFP4: 2^7 * the expert's W13 global scale
        uint32_t mask = 0;
        const int e0 = warp - kEpilogueWarp;
        int a = (r13b + e0) / PJ, j = r13b + e0 - a * PJ;     // segment and piece of unit r13b + i
        for (int i = e0; i < n13; i += kEpilogueWarps, j += kEpilogueWarps) {
            while (j >= PJ) {
                j -= PJ;
                ++a;
            }
            const int slot = i & 1;
            const int u = r13b + i;
            if (a != cur_a) {
                cur_a = a;
                mask = tm[a];
                const int e = act[a];
                wsum = 0.f;
                if (lane < M && (mask >> lane & 1))
                    for (int q = 0; q < k; ++q)
                        if (s_ids[lane * k + q] == e) wsum += s_w[lane * k + q];
                if constexpr (MB == 2) {
                    g13 = 128.f * args.global_scale[2 * e];
                    wsum *= args.global_scale[2 * e + 1];       // the W2 global, folded into HW
                }
            }
            if (!mbar_wait_bounded(&red_full[slot], (i >> 1) & 1, tmo)) {
                set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                return;
            }
            const float *rs = red + slot * (red_slot_bytes(NT) / 4);
            // fixed-order sum over the warps; lane (g, t) of n-block n holds gate
            // (x: row 8n+2t, y: row 8n+2t+1) and up (z, w) of piece column g
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                float4 sum = *reinterpret_cast<const float4 *>(rs + (n * 32 + lane) * 4);
#pragma unroll
                for (int w = 1; w < kConsumerWarps; ++w) {
                    const float4 v = *reinterpret_cast<const float4 *>(rs + ((w * NT + n) * 32 + lane) * 4);
                    sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
                }
                if constexpr (MB == 2) {
                    sum.x *= g13; sum.y *= g13; sum.z *= g13; sum.w *= g13;
                }
                hbuf[(n * 8 + 2 * t) * kPieceCols + g] = silu_f(sum.x) * sum.z;
                hbuf[(n * 8 + 2 * t + 1) * kPieceCols + g] = silu_f(sum.y) * sum.w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_count(&red_empty[slot], 1);   // slot read out
            // HW[a][token][8j .. 8j+7] as one 16-byte store per token row, scaled
            // by the token's router weight (zero for tokens not routed here)
            if (lane < MP) {
                const bool routed = lane < M && (mask >> lane & 1);
                const int row = __popc(mask & ((1u << lane) - 1u));
                // the octet is stored in MMA fragment order (columns 0,4,1,5,2,6,3,7:
                // the W2 K permutation), so the W2 warps load it as it stands
                uint32_t pk[4], pl[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float v0 = routed ? wsum * hbuf[row * kPieceCols + c] : 0.f;
                    const float v1 = routed ? wsum * hbuf[row * kPieceCols + c + 4] : 0.f;
                    const uint16_t b0 = f2h_bits(v0), b1 = f2h_bits(v1);
                    pk[c] = static_cast<uint32_t>(b0) | (static_cast<uint32_t>(b1) << 16);
                    if constexpr (MB == 2)     // NVFP4: the fp16 residue plane
                        pl[c] = static_cast<uint32_t>(f2h_bits(v0 - __half2float(__ushort_as_half(b0)))) |
                                (static_cast<uint32_t>(f2h_bits(v1 - __half2float(__ushort_as_half(b1)))) << 16);
                }
                const int64_t at = (static_cast<int64_t>(a) * MP + lane) * I + kPieceCols * j;
                *reinterpret_cast<uint4 *>(args.hw + at) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                if constexpr (MB == 2) *reinterpret_cast<uint4 *>(args.hw_lo + at) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
            }
            __syncwarp();                                            // hbuf is reused
            // debug bit 0 withholds the announcement of piece 0
            if (!((args.debug_flags & 1) && u == 0)) ++finished;
        }
        // one announcement for all pieces this CTA finished (release: their HW
        // entries are visible to whoever sees the count)
        if (lane == 0 && finished > 0) red_add_release(done13, finished);
        return;
    }

    // ================================ consumers ================================
    // ok: results valid. dead: a wait for a copy ran out, so later copy waits
    // are skipped (results are then undefined and the status word says so).
    // The W2 phase's waits for other CTAs only clear ok, so the ring is still
    // drained and no copy is in flight when the CTA exits.
    bool ok = true, dead = false;
    // ring position of the next unit (index and phase kept incrementally)
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

    // ---------------- W13 + SwiGLU ----------------
    {
        uint4 xf[kGroupsPerWarp][NT];   // this warp's x fragments of the current segment
        int cur_a = -1, rows = 0;
        int a = r13b / PJ, j = r13b - a * PJ;   // segment and piece of unit r13b + i
        for (int i = 0; i < n13; ++i, ++j) {
            if (j == PJ) {
                j = 0;
                ++a;
            }
            if (a != cur_a) {
                cur_a = a;
                const uint32_t mask = tm[a];
                rows = __popc(mask);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const int tok = nth_token(mask, n * 8 + g);
                    const uint16_t *xr = args.x + static_cast<int64_t>(tok < 0 ? 0 : tok) * kHidden +
                                         warp * kGroupsPerWarp * kGroup + t * 8;
#pragma unroll
                    for (int gi = 0; gi < kGroupsPerWarp; ++gi)
                        xf[gi][n] = tok < 0 ? make_uint4(0, 0, 0, 0) : permute_k8(ld_nc_v4(xr + gi * kGroup));
                }
            }
            wait_stage();
            const uint32_t base = smem_u32(ring + st_idx * kStageBytes);
            float acc[NT][4];
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[n][v] = 0.f;
#pragma unroll
            for (int gi = 0; gi < kGroupsPerWarp; ++gi) {
                const int grp = warp * kGroupsPerWarp + gi;
                const uint2 q = lds_v2(base + ((grp * 4 + t) * kPieceCols + g) * 8);
                if constexpr (MB == 2) {
                    // gate and up records of column g: block (t / 2) scale codes
                    const uint32_t r = lds_u32(base + kPieceQ + (grp * kPieceCols + g) * 4);
                    const uint32_t sg2 = e4m3_scale_pair(r >> (8 * (t >> 1)) & 0xFFu);
                    const uint32_t su2 = e4m3_scale_pair(r >> (16 + 8 * (t >> 1)) & 0xFFu);
#pragma unroll
                    for (int n = 0; n < NT; ++n)
                        if (n == 0 || n * 8 < rows)
                            group_tile_mma_nv(acc[n], q.x, q.y, sg2, su2, xf[gi][n]);
                } else {
                    const MetaPair m = load_meta_pair<MB>(base + kPieceQ + (grp * kPieceCols + g) * 2 * MB);
                    const float sg = half_bits_to_float(m.sg), su = half_bits_to_float(m.su);
#pragma unroll
                    for (int n = 0; n < NT; ++n)
                        if (n == 0 || n * 8 < rows)   // a segment has at least one row
                            group_tile_mma(acc[n], q.x, q.y, m.zg2, m.zu2, sg, su, xf[gi][n]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_count(&empty[st_idx], 1);
            next_stage();
            // hand the warp's tile to the epilogue warp
            const int slot = i & 1;
            if (!dead && !mbar_wait_bounded(&red_empty[slot], ((i >> 1) & 1) ^ 1, tmo)) {
                ok = false;
                dead = true;
                set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
            }
            float *rs = red + slot * (red_slot_bytes(NT) / 4);
#pragma unroll
            for (int n = 0; n < NT; ++n)
                *reinterpret_cast<float4 *>(rs + ((warp * NT + n) * 32 + lane) * 4) =
                    make_float4(acc[n][0], acc[n][1], acc[n][2], acc[n][3]);
            __syncwarp();
            if (lane == 0) mbar_arrive_count(&red_full[slot], 1);
        }
    }

    const int Qg = (g >> 1) | ((g & 1) << 2);      // bank-conflict-free column quad of lane
    // W2 work of this warp: tile w2t (half w2h with 16 warps); idle warps none
    const int w2t = warp % kW2Tiles, w2h = warp / kW2Tiles;
    const bool w2_active = w2h < kW2Split;
    // ---------------- W2 + weighted top-k reduction ----------------
    // Warp w works on tile w % 8 of each unit: both 16-column halves with 10
    // consumer warps (warps 8-9 idle), half w / 8 with 16. A unit's stage
    // holds its weights and, at kHwOff, its activation rows (the producer
    // loads those only once every W13 piece is announced).
    if (tmode) {
        // ---- tile mode: warp w takes segment slot w % 4, column half (w / 4) % 2 and
        // K groups [0, 3) or [3, 5) (w / 8) of every unit of this CTA's tile
        if (n2 > 0) {
            const int ts = warp & 3, th = (warp >> 2) & 1, tq = warp >> 3;
            const int tg0 = tq ? 3 : 0, ng = tq ? kW2Groups - 3 : 3;
            // The units' activations go out together once HW is complete, so the
            // warp waits for all its units first and then expands every group of
            // them in one unrolled pass (no per-unit ramp).
            uint32_t ubase[kTMaxUnits];
            int ustage[kTMaxUnits];
#pragma unroll
            for (int u = 0; u < kTMaxUnits; ++u) {
                ustage[u] = st_idx;
                ubase[u] = smem_u32(ring + st_idx * kStageBytes);
                if (u < n2) {
                    wait_stage();
                    next_stage();
                }
            }
            float tacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int u = 0; u < kTMaxUnits; ++u) {
                if (u < n2 && ts < kTSegsU && (u / KP) * kTSegsU + ts < A) {
                    const uint32_t qb = ubase[u] + ts * kTQSlot;
                    const uint32_t mbase = ubase[u] + kTMeta + ts * kTMetaSlot;
                    const uint32_t hb = ubase[u] + kTHw + ts * MP * kHwRow;
#pragma unroll
                    for (int x = 0; x < 3; ++x) {
                        if (x >= ng) continue;
                        const int gg = tg0 + x;
                        const int L = 4 * gg + t;
                        const uint4 xb = lds_v4(hb + g * kHwRow + L * 16);   // HW octets are in fragment order
                        if constexpr (MB == 4) {
                            // only this warp's half: 8 bytes of the line, 2 of the quad's records
                            const uint2 q = lds_v2(qb + L * 128 + ((Qg ^ (L & 7)) << 4) + th * 8);
                            const uint2 r = lds_v2(mbase + gg * 32 * MB + Qg * 4 * MB + th * 8);
                            group_tile_mma(tacc, q.x, q.y, zero_pair_byte<2>(r.x), zero_pair_byte<2>(r.y),
                                           half_bits_to_float(r.x), half_bits_to_float(r.y), xb);
                        } else if constexpr (MB == 2) {
                            // this warp's half; the two records' block (t / 2) scale codes; HW
                            // and its residue row
                            const uint2 q = lds_v2(qb + L * 128 + ((Qg ^ (L & 7)) << 4) + th * 8);
                            const uint32_t r = lds_u32(mbase + gg * 32 * MB + Qg * 4 * MB + th * 4);
                            const uint4 xl = lds_v4(hb + kTSegsU * MP * kHwRow + g * kHwRow + L * 16);
                            group_tile_mma_nv2(tacc, q.x, q.y, e4m3_scale_pair(r >> (8 * (t >> 1)) & 0xFFu),
                                               e4m3_scale_pair(r >> (16 + 8 * (t >> 1)) & 0xFFu), xb, xl);
                        } else {
                            const uint4 q = lds_v4(qb + L * 128 + ((Qg ^ (L & 7)) << 4));
                            const Meta4<MB> mt = load_meta4<MB>(mbase + gg * 32 * MB + Qg * 4 * MB);
                            group_tile_mma(tacc, th ? q.z : q.x, th ? q.w : q.y, th ? mt.z2[2] : mt.z2[0],
                                           th ? mt.z2[3] : mt.z2[1], half_bits_to_float(th ? mt.s[2] : mt.s[0]),
                                           half_bits_to_float(th ? mt.s[3] : mt.s[1]), xb);
                        }
                    }
                }
            }
            __syncwarp();
#pragma unroll
            for (int u = 0; u < kTMaxUnits; ++u)
                if (u < n2 && lane == 0) mbar_arrive_count(&empty[ustage[u]], 1);
            // the eight warps of each half add their partials in a fixed order (the
            // hand-off slots are idle: every piece of the grid is finished)
            *reinterpret_cast<float4 *>(red + (warp * 32 + lane) * 4) = make_float4(tacc[0], tacc[1], tacc[2], tacc[3]);
            named_barrier_sync(kBarCompute, kConsumerThreads);
            if (warp < 2 && ok) {
                const int hh = warp;
                float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int wq = 0; wq < 2; ++wq)
#pragma unroll
                    for (int ws = 0; ws < kTSegs; ++ws) {
                        const float4 v = *reinterpret_cast<const float4 *>(red + ((ws + 4 * hh + 8 * wq) * 32 + lane) * 4);
                        sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
                    }
                const float osc = MB == 2 ? 128.f : 1.f;    // NVFP4: the weights entered as w 2^-7
                const float vals[4] = {osc * sum.x, osc * sum.y, osc * sum.z, osc * sum.w};
#pragma unroll
                for (int vv = 0; vv < 4; ++vv) {
                    const int tok = 2 * t + (vv & 1);
                    const int col = 32 * b + 4 * Qg + 2 * hh + (vv >> 1);
                    if (tok < M) args.out[static_cast<int64_t>(tok) * kHidden + col] = f2h_bits(vals[vv]);
                }
            }
        }
        return;
    }

    const int cg_first = n2 > 0 ? r2b / per_c : 0;
    float acc0[2][NT][4], acc1[2][NT][4];   // this warp's tile in groups cg_first, cg_first + 1
#pragma unroll
    for (int T = 0; T < 2; ++T)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc0[T][n][v] = acc1[T][n][v] = 0.f;

    int cg = cg_first, cg_rem = r2b - cg_first * per_c;   // column group of unit r2b + i
    for (int i = 0; i < n2; ++i, ++cg_rem) {
        if (cg_rem == per_c) {
            cg_rem = 0;
            ++cg;
        }
        wait_stage();
        const uint32_t base = smem_u32(ring + st_idx * kStageBytes);
        const uint32_t hb = base + kHwOff;
        float part[2][NT][4];
#pragma unroll
        for (int T = 0; T < 2; ++T)
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int vv = 0; vv < 4; ++vv) part[T][n][vv] = 0.f;
        if (kW2Split == 2 && MB == 4) {
            // this warp's 16-column half only: 8 of the line's 16 bytes and 2 of
            // the quad's 4 records (columns 4Qg + 2*w2h + (0, 1)), into part[0]
#pragma unroll
            for (int gg = 0; gg < kW2Groups; ++gg) {
                const int L = w2t * kW2KK + 4 * gg + t;        // line of this warp's tile
                const uint2 q = lds_v2(base + L * 128 + ((Qg ^ (L & 7)) << 4) + w2h * 8);
                const uint2 r = lds_v2(base + kW2Q + (w2t * kW2Groups + gg) * 32 * MB + Qg * 4 * MB + w2h * 8);
                const uint32_t za = zero_pair_byte<2>(r.x), zb = zero_pair_byte<2>(r.y);
                const float sa = half_bits_to_float(r.x), sb = half_bits_to_float(r.y);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const uint4 xb = lds_v4(hb + (n * 8 + g) * kHwRow + (4 * gg + t) * 16);   // fragment order
                    group_tile_mma(part[0][n], q.x, q.y, za, zb, sa, sb, xb);
                }
            }
        } else if (kW2Split == 2 && MB == 2) {
            // NVFP4, this warp's 16-column half: 8 bytes of the line, 2 records
#pragma unroll
            for (int gg = 0; gg < kW2Groups; ++gg) {
                const int L = w2t * kW2KK + 4 * gg + t;
                const uint2 q = lds_v2(base + L * 128 + ((Qg ^ (L & 7)) << 4) + w2h * 8);
                const uint32_t r = lds_u32(base + kW2Q + (w2t * kW2Groups + gg) * 32 * MB + Qg * 4 * MB + w2h * 4);
                const uint32_t sa2 = e4m3_scale_pair(r >> (8 * (t >> 1)) & 0xFFu);
                const uint32_t sb2 = e4m3_scale_pair(r >> (16 + 8 * (t >> 1)) & 0xFFu);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const uint4 xb = lds_v4(hb + (n * 8 + g) * kHwRow + (4 * gg + t) * 16);
                    const uint4 xl = lds_v4(hb + (MP + n * 8 + g) * kHwRow + (4 * gg + t) * 16);   // residue
                    group_tile_mma_nv2(part[0][n], q.x, q.y, sa2, sb2, xb, xl);
                }
            }
        } else if (MB == 2 && w2_active) {
            // NVFP4, both halves of the tile (one warp per tile)
#pragma unroll
            for (int gg = 0; gg < kW2Groups; ++gg) {
                const int L = w2t * kW2KK + 4 * gg + t;
                const uint4 q = lds_v4(base + L * 128 + ((Qg ^ (L & 7)) << 4));
                const uint2 r = lds_v2(base + kW2Q + (w2t * kW2Groups + gg) * 32 * MB + Qg * 4 * MB);
                const int sh = 8 * (t >> 1);
                const uint32_t s0 = e4m3_scale_pair(r.x >> sh & 0xFFu), s1 = e4m3_scale_pair(r.x >> (16 + sh) & 0xFFu);
                const uint32_t s2 = e4m3_scale_pair(r.y >> sh & 0xFFu), s3 = e4m3_scale_pair(r.y >> (16 + sh) & 0xFFu);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const uint4 xb = lds_v4(hb + (n * 8 + g) * kHwRow + (4 * gg + t) * 16);
                    const uint4 xl = lds_v4(hb + (MP + n * 8 + g) * kHwRow + (4 * gg + t) * 16);   // residue
                    group_tile_mma_nv2(part[0][n], q.x, q.y, s0, s1, xb, xl);
                    group_tile_mma_nv2(part[1][n], q.z, q.w, s2, s3, xb, xl);
                }
            }
        } else if (w2_active) {
#pragma unroll
            for (int gg = 0; gg < kW2Groups; ++gg) {
                const int L = w2t * kW2KK + 4 * gg + t;        // line of this warp's tile
                const uint4 q = lds_v4(base + L * 128 + ((Qg ^ (L & 7)) << 4));
                const Meta4<MB> mt = load_meta4<MB>(base + kW2Q + (w2t * kW2Groups + gg) * 32 * MB + Qg * 4 * MB);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const uint4 xb = lds_v4(hb + (n * 8 + g) * kHwRow + (4 * gg + t) * 16);   // fragment order
                    if (kW2Split == 1) {
                        group_tile_mma(part[0][n], q.x, q.y, mt.z2[0], mt.z2[1], half_bits_to_float(mt.s[0]),
                                       half_bits_to_float(mt.s[1]), xb);
                        group_tile_mma(part[1][n], q.z, q.w, mt.z2[2], mt.z2[3], half_bits_to_float(mt.s[2]),
                                       half_bits_to_float(mt.s[3]), xb);
                    } else {
                        // this warp's half only: columns 4Qg + 2*w2h + (0, 1), into part[0]
                        const bool hi = w2h != 0;
                        group_tile_mma(part[0][n], hi ? q.z : q.x, hi ? q.w : q.y, hi ? mt.z2[2] : mt.z2[0],
                                       hi ? mt.z2[3] : mt.z2[1], half_bits_to_float(hi ? mt.s[2] : mt.s[0]),
                                       half_bits_to_float(hi ? mt.s[3] : mt.s[1]), xb);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_count(&empty[st_idx], 1);
        next_stage();
        if (cg == cg_first) {
#pragma unroll
            for (int T = 0; T < 2; ++T)
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int vv = 0; vv < 4; ++vv) acc0[T][n][vv] += part[T][n][vv];
        } else {
#pragma unroll
            for (int T = 0; T < 2; ++T)
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int vv = 0; vv < 4; ++vv) acc1[T][n][vv] += part[T][n][vv];
        }
    }

    if (n2 > 0) {
        // Each active warp holds its part of tile w2t of the column groups it
        // touched: value v of half h, n-block n is (token n*8 + 2t + (v&1),
        // column 32*(8cg + w2t) + 4*Qg + 2h + (v>>1)). A group that lies inside this
        // CTA's share is written out directly. For a group split between CTAs
        // every part publishes its partial; once all parts are in, part q
        // finishes columns [256q/n, 256(q+1)/n) of the group, summing the
        // partials in CTA order. All partials go out before any wait, so no
        // wait depends on another.
        const int cg_last = (r2e - 1) / per_c;
        const int ngroups = cg_last - cg_first + 1;
        for (int ct = 0; ct < ngroups; ++ct) {
            const int cg = cg_first + ct;
            const int V0 = cg * per_c;
            const bool whole = (V0 >= r2b && V0 + per_c <= r2e);
            const int slot = (r2b >= V0) ? 0 : 1;
            float *mine = args.part2 + (static_cast<int64_t>(b) * 2 + slot) * kPartStride;
#pragma unroll
            for (int T = 0; T < 2; ++T)
#pragma unroll
                for (int n = 0; n < NT; ++n)
#pragma unroll
                    for (int vv = 0; vv < 4; ++vv) {
                        const int half = kW2Split == 1 ? T : w2h;     // 16-column half of the tile
                        const int tok = n * 8 + 2 * t + (vv & 1);
                        const int col = 32 * w2t + 4 * Qg + 2 * half + (vv >> 1);
                        const float val = ct == 0 ? acc0[T][n][vv] : acc1[T][n][vv];
                        if (tok < M && w2_active && (kW2Split == 1 || T == 0)) {
                            if (!whole) mine[tok * 256 + col] = val;
                            else if (ok)
                                args.out[static_cast<int64_t>(tok) * kHidden + cg * 256 + col] =
                                    f2h_bits(MB == 2 ? 128.f * val : val);
                        }
                    }
        }
        named_barrier_sync(kBarCompute, kConsumerThreads);
        if (tid == 0) {
            // one fence releases the partials of both groups (a CTA whose share
            // straddles two groups publishes two)
            bool fenced = false;
            for (int ct = 0; ct < ngroups; ++ct) {
                const int V0 = (cg_first + ct) * per_c;
                if (V0 >= r2b && V0 + per_c <= r2e) continue;
                if (!fenced) fence_acq_rel_gpu();
                fenced = true;
                red_add_relaxed(&cnt2[cg_first + ct], 1);
            }
        }
        // Offsets of the split groups' partial blocks, in CTA order (s_ids is
        // free: the epilogue warp is done with it once every piece is in).
        int32_t *s_who = s_ids;                                  // [2][32]
        for (int ct = 0; ct < ngroups; ++ct) {
            const int V0 = (cg_first + ct) * per_c;
            if (V0 >= r2b && V0 + per_c <= r2e) continue;
            if (tid < parts_count(V0, per_c, U2, G))
                s_who[ct * 32 + tid] = part_index(V0, tid, range_owner(V0, U2, G), U2, G) * kPartStride;
        }
        if (tid == 0) {
            bool all_in = true;
            for (int ct = 0; ct < ngroups; ++ct) {
                const int V0 = (cg_first + ct) * per_c;
                if (!(V0 >= r2b && V0 + per_c <= r2e))
                    all_in = wait_counter(&cnt2[cg_first + ct], parts_count(V0, per_c, U2, G), tmo) && all_in;
            }
            s_misc[4] = all_in ? 1 : 0;
        }
        named_barrier_sync(kBarCompute, kConsumerThreads);
        if (!s_misc[4]) {
            ok = false;
            if (tid == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
        }
        // This CTA's column slice of each split group (at most two groups),
        // the items of both in one pass so that their loads are in flight
        // together.
        int n_it[2] = {0, 0}, c0g[2] = {0, 0}, wid[2] = {1, 1}, npg[2] = {0, 0};
#pragma unroll
        for (int ct = 0; ct < 2; ++ct) {
            const int V0 = (cg_first + ct) * per_c;
            if (ct >= ngroups || (V0 >= r2b && V0 + per_c <= r2e)) continue;
            const int nparts = parts_count(V0, per_c, U2, G);
            const int b_first = range_owner(V0, U2, G);
            const int q_me = U2 < G ? r2b - V0 : b - b_first;       // this CTA's part number
            c0g[ct] = (q_me * 256) / nparts;
            wid[ct] = ((q_me + 1) * 256) / nparts - c0g[ct];
            n_it[ct] = M * wid[ct];
            npg[ct] = nparts;
        }
        for (int item = tid; ok && item < n_it[0] + n_it[1]; item += kConsumerThreads) {
            const bool second = item >= n_it[0];
            const int it = second ? item - n_it[0] : item;
            const int width = second ? wid[1] : wid[0], nparts = second ? npg[1] : npg[0];
            const int tk = it / width, col = (second ? c0g[1] : c0g[0]) + (it - tk * width);
            const int32_t *who = s_who + (second ? 32 : 0);
            const float *pb = args.part2 + tk * 256 + col;
            // every part's load in flight at once, then the sum in CTA order
            float v[kMaxParts];
#pragma unroll
            for (int q = 0; q < kMaxParts; ++q) v[q] = q < nparts ? __ldcg(pb + who[q]) : 0.f;
            float sum = 0.f;
#pragma unroll
            for (int q = 0; q < kMaxParts; ++q)
                if (q < nparts) sum += v[q];
            const int cg = cg_first + (second ? 1 : 0);
            args.out[static_cast<int64_t>(tk) * kHidden + cg * 256 + col] = f2h_bits(MB == 2 ? 128.f * sum : sum);
        }
    }
}

awq_status launch_fused(int mb, int sms, cudaStream_t st, const CUtensorMap &t2q,
                        const CUtensorMap &t2m, const CUtensorMap &t2q1, const CUtensorMap &t2m1,
                        const FusedArgs &a)
{
    const int NT = a.M > 8 ? 2 : 1;
    const int smem = fused_layout(NT, mb).total + 1024;
    const int threads = NT == 1 ? fused_threads(1) : fused_threads(2);
    void (*kernel)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, FusedArgs);
    if (mb == 4)
        kernel = NT == 1 ? fused_layer_kernel<4, 1> : fused_layer_kernel<4, 2>;
    else if (mb == 3)
        kernel = NT == 1 ? fused_layer_kernel<3, 1> : fused_layer_kernel<3, 2>;
    else
        kernel = NT == 1 ? fused_layer_kernel<2, 1> : fused_layer_kernel<2, 2>;   // NVFP4
    awq_status r = set_smem(kernel, smem);
    if (r) return r;
    // cooperative: the cross-CTA waits need every CTA resident
    return launch_ex(kernel, dim3(sms), dim3(threads), smem, 1, true, st, t2q, t2m, t2q1, t2m1, a);
}

}  // namespace awq
