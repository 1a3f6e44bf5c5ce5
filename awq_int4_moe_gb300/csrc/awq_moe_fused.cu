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
// sorted slots.
//
// Schedule. One CTA per SM (grid = SM count). Each CTA takes a contiguous,
// equal share of two flat work lists:
//   W13 units  (segment a, 32-column gate|up slab p, 512-row K chunk)        20 KB
//   W2  units  (32-column output tile c, group of 8 segments, 160-row K part) <= 29 KB
// A producer warp streams the units' packed int4 tiles and metadata with TMA
// (one 32-column x 64-row box per gate and up slab, 128-byte swizzled lines)
// and each W13 unit's x rows (cp.async) into a ring of shared-memory stages;
// eight consumer warps dequantise in registers and run m16n8k16 tensor-core
// MMAs with the weights on the M side and tokens on the N side. A tenth warp
// finishes W13 pieces (cross-warp sums, partial publication, SwiGLU) from
// double-buffered hand-off slots while the consumers keep streaming. The W2
// activations are read from L2 one unit ahead.
//
// Reductions are deterministic and need no atomics on data: a (segment, slab)
// piece or output tile that lies inside one CTA's share is finished by that
// CTA; one split between CTAs is finished by the last CTA to publish its
// partial (release/acquire arrival counter), which sums the partials in CTA
// order. W13 finishers apply SwiGLU and store the router-weighted activations
// HW[a][t][:] = (sum of the router weights of token t's slots on segment a) *
// h[a][t][:]; W2 accumulates all segments of a tile with tokens as the MMA N
// dimension. The only cross-CTA wait is the W2 phase waiting for every W13
// piece (bounded by a timeout; the grid is one CTA per SM, all resident).
// Counters reset themselves, so the workspace stays zeroed between calls.
#include <cuda_fp16.h>

#include "awq_dequant.cuh"
#include "awq_launch.cuh"
#include "awq_moe_kernels.cuh"
#include "awq_ptx.cuh"

namespace awq {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kEpilogueWarp = kConsumerWarps + 1;
constexpr int kFusedThreads = (kConsumerWarps + 2) * 32;
constexpr int kMaxSlotsF = kFusedMaxTokens * kMaxTopK;           // 256

// W13 unit: 16 groups (512 k) of one 32-column gate|up slab; warp w takes
// groups 2w and 2w+1. Gate lines at +0, up lines at +8 KB (64 x 128 B each).
constexpr int kFGroups13 = 16;
constexpr int kFKK13 = kFGroups13 * 4;                             // 64 packed rows
constexpr int kFChunks13 = kHidden / (kFGroups13 * kGroup);        // 5 per slab
constexpr int kFHalf13 = kFKK13 * 128;                             // 8 KB
constexpr int kFQ13 = 2 * kFHalf13;                                // 16 KB
// W2 unit: one 32-column tile, 8 segments (warp w <-> segment 8*sg + w), one
// 160-row K part (5 groups). Each segment's q box sits in its own
// 1024-byte-aligned 3 KB slot (the 128-byte swizzle repeats every 1 KB).
constexpr int kW2Seg = 8;
constexpr int kW2KK = 20;
constexpr int kW2Groups = 5;
constexpr int kW2QSlot = 3072;
constexpr int kW2QBytes = kW2KK * 128;                              // 2560 per segment
constexpr int kW2MetaSlot = 640;                                    // 5 groups x 32 x 4
constexpr int kColTiles = kHidden / 32;
constexpr int kBarCompute = 1;
// A W13 stage also holds the unit's x slice: one padded 1088-byte row (512
// fp16 + 64 B, so B-fragment loads are bank-conflict free) per token routed to
// the segment, copied by the producer warp with cp.async.
constexpr int kXSliceOff = kFQ13 + kFGroups13 * 64 * 4;            // 20480
constexpr int kXSliceRow = kFGroups13 * kGroup * 2 + 64;           // 1088

__host__ __device__ constexpr int fused_stage_bytes(int NT)
{
    // max(W2 unit, W13 unit with 8*NT x rows), rounded to 1 KB (swizzle atom)
    return NT == 1 ? 29 * 1024 : 37 * 1024;
}
__host__ __device__ constexpr int fused_stages(int NT) { return NT == 1 ? 6 : 4; }

static_assert(kW2Seg * kW2QSlot + kW2Seg * kW2MetaSlot <= fused_stage_bytes(1), "W2 unit fits");
static_assert(kXSliceOff + 8 * kXSliceRow <= fused_stage_bytes(1), "W13 unit (8 rows) fits");
static_assert(kXSliceOff + 16 * kXSliceRow <= fused_stage_bytes(2), "W13 unit (16 rows) fits");

struct Layout {
    int bars, red, gu, hf, route, total;
};

// One hand-off slot: every consumer warp's W13 accumulators for one piece
// ([warp][tile 4][n NT][lane][4] floats); two slots alternate.
__host__ __device__ constexpr int red_slot_bytes(int NT) { return kConsumerWarps * 4 * NT * 32 * 16; }

__host__ __device__ constexpr int round_up(int v, int a) { return (v + a - 1) / a * a; }

// Shared-memory layout (offsets from the 1024-aligned base). Stage s starts at
// s * kStageBytes, a multiple of 1024.
__host__ __device__ inline Layout fused_layout(int NT)
{
    Layout L;
    const int stages = fused_stages(NT);
    L.bars = round_up(stages * fused_stage_bytes(NT), 1024);
    L.red = round_up(L.bars + (2 * stages + 4) * 8, 128);
    L.gu = L.red + 2 * red_slot_bytes(NT);
    L.hf = L.gu + 16 * 64 * 4;
    L.route = L.hf + 16 * 32 * 4;
    // s_ids[256], s_w[256], act[256], tm[256], bitmap[32], wpre[32], misc[16]
    L.total = L.route + (4 * kMaxSlotsF + 32 + 32 + 16) * 4;
    return L;
}

__device__ __forceinline__ int range_start(int b, int U, int G)
{
    return static_cast<int>((static_cast<int64_t>(b) * U) / G);
}

// CTA whose share contains unit u (largest b with range_start(b) <= u).
__device__ __forceinline__ int range_owner(int u, int U, int G)
{
    return static_cast<int>(((static_cast<int64_t>(u) + 1) * G - 1) / U);
}

__device__ __forceinline__ int atom_add_acq_rel(int32_t *p, int v)
{
    int old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void red_add_release(int32_t *p, int v)
{
    asm volatile("red.add.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
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

// The CTAs whose shares intersect units [U0, U0 + len) of a list of U units
// split over G CTAs, as (CTA, partial slot) pairs in CTA order; a CTA uses
// slot 0 for the first piece of its share and slot 1 for its last. Returns
// the number of parts (at most kMaxParts). Divisions are done once per CTA.
constexpr int kMaxParts = 16;
__device__ __forceinline__ int split_parts(int U0, int len, int U, int G, int (&who)[kMaxParts])
{
    const int b_first = range_owner(U0, U, G), b_last = range_owner(U0 + len - 1, U, G);
    int n = 0;
    int st = range_start(b_first, U, G);
    for (int bb = b_first; bb <= b_last && n < kMaxParts; ++bb) {
        const int nx = range_start(bb + 1, U, G);
        if (st < nx) who[n++] = bb * 2 + (st >= U0 ? 0 : 1);
        st = nx;
    }
    return n;
}

// j-th (0-based) set bit of a token mask, or -1.
__device__ __forceinline__ int nth_token(uint32_t mask, int j)
{
    if (j >= __popc(mask)) return -1;
    return static_cast<int>(__fns(mask, 0, j + 1));
}

}  // namespace

template <int MB, int NT>
__global__ void __launch_bounds__(kFusedThreads, 1)
fused_layer_kernel(const __grid_constant__ CUtensorMap t13q, const __grid_constant__ CUtensorMap t13m,
                   const __grid_constant__ CUtensorMap t2q, const __grid_constant__ CUtensorMap t2m,
                   FusedArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    constexpr int kStages = fused_stages(NT);
    constexpr int kStageBytes = fused_stage_bytes(NT);
    constexpr int MP = 8 * NT;                     // token rows of HW per segment
    const int M = args.M, k = args.top_k, E = args.num_experts, I = args.inter;
    const int P = I / 32, KP = I / 160;            // slabs per expert, W2 K parts
    const Layout Lo = fused_layout(NT);
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lo.bars);
    uint64_t *empty = full + kStages;
    uint64_t *red_full = empty + kStages;          // [2] consumer warps -> epilogue
    uint64_t *red_empty = red_full + 2;            // [2] epilogue -> consumer warps
    float *red = reinterpret_cast<float *>(smem + Lo.red);
    float *gu = reinterpret_cast<float *>(smem + Lo.gu);
    float *hf = reinterpret_cast<float *>(smem + Lo.hf);
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
        prefetch_tmap(&t13q);
        prefetch_tmap(&t13m);
        prefetch_tmap(&t2q);
        prefetch_tmap(&t2m);
    }
    if (tid < 32) bitmap[tid] = 0;
    for (int i = tid; i < kMaxSlotsF; i += kFusedThreads) tm[i] = 0;
    grid_dependency_wait();
    grid_launch_dependents();

    // ---------------- routing in shared memory ----------------
    if (tid < S) {
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

    const int A = s_misc[0];
    const int nsg = (A + kW2Seg - 1) / kW2Seg;
    const int U13 = A * P * kFChunks13;
    const int U2 = kColTiles * nsg * KP;
    const int r13b = range_start(b, U13, G), r13e = range_start(b + 1, U13, G);
    const int r2b = range_start(b, U2, G), r2e = range_start(b + 1, U2, G);
    const int n13 = r13e - r13b, n2 = r2e - r2b;
    const uint64_t tmo = args.timeout_ns;
    const int per_c = nsg * KP;                    // W2 units per output tile

    if (warp == kProducerWarp) {
        // ================================ producer ================================
        for (int i = 0; i < n13 + n2; ++i) {
            const int s = i % kStages;
            const uint32_t ph = (i / kStages) & 1;
            int live = 1;
            if (lane == 0 && !mbar_wait_bounded(&empty[s], ph ^ 1, tmo)) {
                set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                live = 0;
            }
            if (!__shfl_sync(0xffffffffu, live, 0)) break;
            uint8_t *dst = ring + s * kStageBytes;
            if (i < n13) {
                const int u = r13b + i;
                const int piece = u / kFChunks13, ch = u - piece * kFChunks13;
                const int a = piece / P, p = piece - a * P;
                const uint32_t mask = tm[a];
                const int rows = __popc(mask);
                // x[token][512*ch .. +512] of each token of the segment, in token order
                for (int idx = lane; idx < rows * 64; idx += 32) {
                    const int r = idx >> 6, c16 = idx & 63;
                    const int tok = nth_token(mask, r);
                    cp_async_16(dst + kXSliceOff + r * kXSliceRow + c16 * 16,
                                args.x + static_cast<int64_t>(tok) * kHidden + ch * 512 + c16 * 8);
                }
                cp_async_arrive(&full[s]);
                __syncwarp();
                if (lane == 0) {
                    const int e = act[a];
                    mbar_arrive_expect_tx(&full[s], kFQ13 + kFGroups13 * 64 * MB);
                    tma_load_3d(dst, &t13q, &full[s], 32 * p, ch * kFKK13, e);
                    tma_load_3d(dst + kFHalf13, &t13q, &full[s], I + 32 * p, ch * kFKK13, e);
                    tma_load_5d(dst + kFQ13, &t13m, &full[s], 0, p, 0, ch * kFGroups13, e);
                }
            } else if (lane == 0) {
                const int v = r2b + (i - n13);
                const int c = v / per_c, rem = v - c * per_c;
                const int sg = rem / KP, kp = rem - sg * KP;
                const int nseg = min(kW2Seg, A - sg * kW2Seg);
                mbar_arrive_expect_tx(&full[s], nseg * (kW2QBytes + kW2Groups * 32 * MB));
                for (int w = 0; w < nseg; ++w) {
                    const int e = act[sg * kW2Seg + w];
                    tma_load_3d(dst + w * kW2QSlot, &t2q, &full[s], c * 32, kp * kW2KK, e);
                    tma_load_3d(dst + kW2Seg * kW2QSlot + w * kW2MetaSlot, &t2m, &full[s],
                                c * 32 * (MB == 4 ? 1 : 3), kp * kW2Groups, e);
                }
            }
            __syncwarp();
        }
        return;
    }

    if (warp == kEpilogueWarp) {
        // ================================ epilogue ================================
        // Finishes the CTA's W13 pieces in order, one hand-off slot at a time.
        if (n13 == 0) return;
        const int first_piece = r13b / kFChunks13;
        const int n_pieces = (r13e - 1) / kFChunks13 - first_piece + 1;
        for (int ps = 0; ps < n_pieces; ++ps) {
            const int slot = ps & 1;
            if (!mbar_wait_bounded(&red_full[slot], (ps >> 1) & 1, tmo)) {
                set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
                return;
            }
            const int piece = first_piece + ps;
            const int a = piece / P, p = piece - a * P;
            const uint32_t mask = tm[a];
            const int rows = __popc(mask);
            const float *rs = red + slot * (red_slot_bytes(NT) / 4);
            // warp sum (fixed order) -> gu[row][col64]; rows = the segment's tokens in order
            for (int f = lane; f < 4 * NT * 32; f += 32) {
                const int l = f & 31, n = (f >> 5) % NT, T = f / (32 * NT);
                float4 sum = *reinterpret_cast<const float4 *>(rs + (((0 * 4 + T) * NT + n) * 32 + l) * 4);
                for (int w = 1; w < kConsumerWarps; ++w) {
                    const float4 vv = *reinterpret_cast<const float4 *>(rs + (((w * 4 + T) * NT + n) * 32 + l) * 4);
                    sum.x += vv.x; sum.y += vv.y; sum.z += vv.z; sum.w += vv.w;
                }
                const int lg = l >> 2, lt = l & 3;
                const int q4 = (lg >> 1) | ((lg & 1) << 2);
                const int col = (T >> 1) * 32 + 4 * q4 + 2 * (T & 1);
                const int row = n * 8 + 2 * lt;
                gu[row * 64 + col] = sum.x;
                gu[(row + 1) * 64 + col] = sum.y;
                gu[row * 64 + col + 1] = sum.z;
                gu[(row + 1) * 64 + col + 1] = sum.w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_count(&red_empty[slot], 1);   // slot read out

            const int U0 = piece * kFChunks13;
            bool finish = (U0 >= r13b && U0 + kFChunks13 <= r13e);
            if (!finish) {
                // publish this CTA's partial; the last publisher finishes the piece
                const int pslot = (r13b >= U0) ? 0 : 1;
                float *mine = args.part13 + (static_cast<int64_t>(b) * 2 + pslot) * 16 * 64;
                for (int idx = lane; idx < rows * 64; idx += 32) mine[idx] = gu[idx];
                __syncwarp();
                int who[kMaxParts];
                const int nparts = split_parts(U0, kFChunks13, U13, G, who);
                int last = 0;
                if (lane == 0) {
                    const int old = atom_add_acq_rel(&args.cnt13[piece], 1);
                    last = (old == nparts - 1);
                    if (last) args.cnt13[piece] = 0;
                }
                finish = __shfl_sync(0xffffffffu, last, 0) != 0;
                if (finish) {
                    for (int idx = lane; idx < rows * 64; idx += 32) {
                        float sum = 0.f;
                        for (int q = 0; q < nparts; ++q)
                            sum += __ldcg(args.part13 + static_cast<int64_t>(who[q]) * 16 * 64 + idx);
                        gu[idx] = sum;
                    }
                    __syncwarp();
                }
            }
            if (finish) {
                // SwiGLU per token row, scaled by the token's router weight on this
                // expert, into HW[a][token][32p + n] (zero for tokens not routed here)
                const int e = act[a];
                for (int idx = lane; idx < MP * 32; idx += 32) {
                    const int tk = idx >> 5, n = idx & 31;
                    float val = 0.f;
                    if (tk < M && (mask >> tk & 1)) {
                        float wsum = 0.f;
                        for (int j = 0; j < k; ++j)
                            if (s_ids[tk * k + j] == e) wsum += s_w[tk * k + j];
                        const int row = __popc(mask & ((1u << tk) - 1u));
                        val = wsum * (silu_f(gu[row * 64 + n]) * gu[row * 64 + 32 + n]);
                    }
                    args.hw[(static_cast<int64_t>(a) * MP + tk) * I + 32 * p + n] = f2h_bits(val);
                }
                __syncwarp();
                if (lane == 0 && !((args.debug_flags & 1) && piece == 0)) red_add_release(&args.sync[0], 1);
            }
            __syncwarp();
        }
        return;
    }

    // ================================ consumers ================================
    // ok: results valid. dead: a wait for a copy ran out, so later copy waits
    // are skipped (results are then undefined and the status word says so).
    // The W2 phase's wait for other CTAs only clears ok, so the ring is still
    // drained and no copy is in flight when the CTA exits.
    bool ok = true, dead = false;
    auto wait_full = [&](int i) {
        if (!dead && !mbar_wait_bounded(&full[i % kStages], (i / kStages) & 1, tmo)) {
            ok = false;
            dead = true;
            set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
        }
    };

    // ---------------- W13 + SwiGLU ----------------
    float acc[4][NT][4];
#pragma unroll
    for (int T = 0; T < 4; ++T)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[T][n][v] = 0.f;

    const int Qg = (g >> 1) | ((g & 1) << 2);      // bank-conflict-free column quad of lane
    int pseq = 0;                                   // pieces handed to the epilogue warp
    for (int i = 0; i < n13; ++i) {
        const int u = r13b + i;
        const int piece = u / kFChunks13;
        const int a = piece / P;
        const int rows = __popc(tm[a]);
        wait_full(i);
        const uint32_t base = smem_u32(ring + (i % kStages) * kStageBytes);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int lg = 2 * warp + j;                // group inside the unit
            const int kk = 4 * lg + t;
            const uint32_t off = kk * 128 + ((Qg ^ (kk & 7)) << 4);
            const uint4 qg = lds_v4(base + off);
            const uint4 qu = lds_v4(base + kFHalf13 + off);
            const Meta4<MB> mg = load_meta4<MB>(base + kFQ13 + (2 * lg + 0) * 32 * MB + Qg * 4 * MB);
            const Meta4<MB> mu = load_meta4<MB>(base + kFQ13 + (2 * lg + 1) * 32 * MB + Qg * 4 * MB);
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                if (n * 8 < rows) {
                    const int row = n * 8 + g;
                    uint4 xb = make_uint4(0, 0, 0, 0);
                    if (row < rows)
                        xb = permute_k8(lds_v4(base + kXSliceOff + row * kXSliceRow + (4 * lg + t) * 16));
                    group_tile_mma(acc[0][n], qg.x, qg.y, mg.z[0], mg.z[1], half_bits_to_float(mg.s[0]),
                                   half_bits_to_float(mg.s[1]), xb);
                    group_tile_mma(acc[1][n], qg.z, qg.w, mg.z[2], mg.z[3], half_bits_to_float(mg.s[2]),
                                   half_bits_to_float(mg.s[3]), xb);
                    group_tile_mma(acc[2][n], qu.x, qu.y, mu.z[0], mu.z[1], half_bits_to_float(mu.s[0]),
                                   half_bits_to_float(mu.s[1]), xb);
                    group_tile_mma(acc[3][n], qu.z, qu.w, mu.z[2], mu.z[3], half_bits_to_float(mu.s[2]),
                                   half_bits_to_float(mu.s[3]), xb);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_count(&empty[i % kStages], 1);
        if (i + 1 < n13 && (u + 1) / kFChunks13 == piece) continue;

        // ---- the CTA's part of (segment a, slab p) is complete: hand it to the epilogue warp ----
        {
            const int slot = pseq & 1;
            if (!dead && !mbar_wait_bounded(&red_empty[slot], ((pseq >> 1) & 1) ^ 1, tmo)) {
                ok = false;
                dead = true;
                set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
            }
            float *rs = red + slot * (red_slot_bytes(NT) / 4);
#pragma unroll
            for (int T = 0; T < 4; ++T)
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    *reinterpret_cast<float4 *>(rs + (((warp * 4 + T) * NT + n) * 32 + lane) * 4) =
                        make_float4(acc[T][n][0], acc[T][n][1], acc[T][n][2], acc[T][n][3]);
#pragma unroll
                    for (int v = 0; v < 4; ++v) acc[T][n][v] = 0.f;
                }
            __syncwarp();
            if (lane == 0) mbar_arrive_count(&red_full[slot], 1);
            ++pseq;
        }
    }

    // ---------------- W2 + weighted top-k reduction ----------------
    if (n2 > 0) {
        if (tid == 0) s_misc[3] = wait_counter(&args.sync[0], A * P, tmo) ? 1 : 0;
        named_barrier_sync(kBarCompute, kConsumerThreads);
        if (!s_misc[3]) {
            ok = false;
            if (tid == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
        }
    }
    const int c_first = n2 > 0 ? r2b / per_c : 0;
    float acc0[2][NT][4], acc1[2][NT][4];   // tiles c_first, c_first + 1
#pragma unroll
    for (int T = 0; T < 2; ++T)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc0[T][n][v] = acc1[T][n][v] = 0.f;

    // HW fragments of unit i for this warp's segment (zeros past the last segment)
    auto load_hw = [&](int i, uint4 (&hb)[kW2Groups][NT]) {
        const int v = r2b + i;
        const int c = v / per_c, rem = v - c * per_c;
        const int sg = rem / KP, kp = rem - sg * KP;
        const int a = sg * kW2Seg + warp;
#pragma unroll
        for (int gg = 0; gg < kW2Groups; ++gg)
#pragma unroll
            for (int n = 0; n < NT; ++n)
                hb[gg][n] = a < A ? ld_cg_v4(args.hw + (static_cast<int64_t>(a) * MP + n * 8 + g) * I +
                                             kp * 160 + gg * 32 + t * 8)
                                  : make_uint4(0, 0, 0, 0);
    };
    // one W2 unit: this warp's segment of the unit against HW fragments hb
    auto w2_unit = [&](int i, const uint4 (&hb)[kW2Groups][NT]) {
        const int v = r2b + i;
        const int c = v / per_c, rem = v - c * per_c;
        const int sg = rem / KP;
        const int a = sg * kW2Seg + warp;
        wait_full(n13 + i);
        const uint32_t base = smem_u32(ring + ((n13 + i) % kStages) * kStageBytes);
        float part[2][NT][4];
#pragma unroll
        for (int T = 0; T < 2; ++T)
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int vv = 0; vv < 4; ++vv) part[T][n][vv] = 0.f;
        if (a < A) {
            const uint32_t qb = base + warp * kW2QSlot;
            const uint32_t mbase = base + kW2Seg * kW2QSlot + warp * kW2MetaSlot;
#pragma unroll
            for (int gg = 0; gg < kW2Groups; ++gg) {
                const int kk = 4 * gg + t;
                const uint4 q = lds_v4(qb + kk * 128 + ((Qg ^ (kk & 7)) << 4));
                const Meta4<MB> mt = load_meta4<MB>(mbase + gg * 32 * MB + Qg * 4 * MB);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const uint4 xb = permute_k8(hb[gg][n]);
                    group_tile_mma(part[0][n], q.x, q.y, mt.z[0], mt.z[1], half_bits_to_float(mt.s[0]),
                                   half_bits_to_float(mt.s[1]), xb);
                    group_tile_mma(part[1][n], q.z, q.w, mt.z[2], mt.z[3], half_bits_to_float(mt.s[2]),
                                   half_bits_to_float(mt.s[3]), xb);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_count(&empty[(n13 + i) % kStages], 1);
        if (c == c_first) {
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
    };
    {
        // HW fragments are loaded one unit ahead into alternating buffers
        uint4 hb0[kW2Groups][NT], hb1[kW2Groups][NT];
        if (n2 > 0) load_hw(0, hb0);
        for (int i = 0; i < n2; i += 2) {
            if (i + 1 < n2) load_hw(i + 1, hb1);
            w2_unit(i, hb0);
            if (i + 1 >= n2) break;
            if (i + 2 < n2) load_hw(i + 2, hb0);
            w2_unit(i + 1, hb1);
        }
    }

    if (n2 > 0) {
        // warp partials -> red[warp][ct][T][n][lane], then CTA sums per tile
        // The epilogue warp has read every hand-off slot before the last W13
        // piece was announced, so the slots are free once the W2 phase runs.
        float *red2 = red;
#pragma unroll
        for (int T = 0; T < 2; ++T)
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                *reinterpret_cast<float4 *>(red2 + ((((warp * 2 + 0) * 2 + T) * NT + n) * 32 + lane) * 4) =
                    make_float4(acc0[T][n][0], acc0[T][n][1], acc0[T][n][2], acc0[T][n][3]);
                *reinterpret_cast<float4 *>(red2 + ((((warp * 2 + 1) * 2 + T) * NT + n) * 32 + lane) * 4) =
                    make_float4(acc1[T][n][0], acc1[T][n][1], acc1[T][n][2], acc1[T][n][3]);
            }
        named_barrier_sync(kBarCompute, kConsumerThreads);
        // gu reused as tsum[ct][token 0..MP)[32 cols]
        float *tsum = gu;
        for (int f = tid; f < 2 * 2 * NT * 32; f += kConsumerThreads) {
            const int l = f & 31, n = (f >> 5) % NT, T = (f / (32 * NT)) & 1, ct = f / (64 * NT);
            float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float4 vv =
                    *reinterpret_cast<const float4 *>(red2 + ((((w * 2 + ct) * 2 + T) * NT + n) * 32 + l) * 4);
                sum.x += vv.x; sum.y += vv.y; sum.z += vv.z; sum.w += vv.w;
            }
            const int lg = l >> 2, lt = l & 3;
            const int q4 = (lg >> 1) | ((lg & 1) << 2);
            const int col = 4 * q4 + 2 * T;
            const int tok = n * 8 + 2 * lt;
            tsum[(ct * MP + tok) * 32 + col] = sum.x;
            tsum[(ct * MP + tok + 1) * 32 + col] = sum.y;
            tsum[(ct * MP + tok) * 32 + col + 1] = sum.z;
            tsum[(ct * MP + tok + 1) * 32 + col + 1] = sum.w;
        }
        named_barrier_sync(kBarCompute, kConsumerThreads);
        const int c_last = (r2e - 1) / per_c;
        for (int c = c_first; c <= c_last; ++c) {
            const int ct = c - c_first;
            const float *ts = tsum + ct * MP * 32;
            const int V0 = c * per_c;
            bool finish = (V0 >= r2b && V0 + per_c <= r2e);
            const float *src = ts;
            if (!finish) {
                const int slot = (r2b >= V0) ? 0 : 1;
                float *mine = args.part2 + (static_cast<int64_t>(b) * 2 + slot) * 16 * 32;
                for (int idx = tid; idx < M * 32; idx += kConsumerThreads) mine[idx] = ts[idx];
                named_barrier_sync(kBarCompute, kConsumerThreads);
                int who[kMaxParts];
                const int nparts = split_parts(V0, per_c, U2, G, who);
                if (tid == 0) {
                    const int old = atom_add_acq_rel(&args.cnt2[c], 1);
                    s_misc[4] = (old == nparts - 1);
                    if (old == nparts - 1) args.cnt2[c] = 0;
                }
                named_barrier_sync(kBarCompute, kConsumerThreads);
                finish = s_misc[4] != 0;
                if (finish) {
                    float *fin = hf;   // [M][32] scratch
                    for (int idx = tid; idx < M * 32; idx += kConsumerThreads) {
                        float sum = 0.f;
                        for (int q = 0; q < nparts; ++q)
                            sum += __ldcg(args.part2 + static_cast<int64_t>(who[q]) * 16 * 32 + idx);
                        fin[idx] = sum;
                    }
                    named_barrier_sync(kBarCompute, kConsumerThreads);
                    src = fin;
                }
            }
            if (finish && ok) {
                for (int idx = tid; idx < M * 16; idx += kConsumerThreads) {
                    const int tk = idx >> 4, n2c = (idx & 15) * 2;
                    const uint32_t lo = f2h_bits(src[tk * 32 + n2c]);
                    const uint32_t hi = f2h_bits(src[tk * 32 + n2c + 1]);
                    *reinterpret_cast<uint32_t *>(args.out + static_cast<int64_t>(tk) * kHidden + c * 32 + n2c) =
                        lo | (hi << 16);
                }
            }
            named_barrier_sync(kBarCompute, kConsumerThreads);
        }
    }

    // ---- last CTA out resets the grid-wide counters ----
    named_barrier_sync(kBarCompute, kConsumerThreads);
    if (tid == 0) {
        if (atom_add_acq_rel(&args.sync[1], 1) == G - 1) {
            args.sync[0] = 0;
            args.sync[1] = 0;
        }
    }
}

awq_status launch_fused(int mb, int sms, cudaStream_t st, const CUtensorMap &t13q,
                        const CUtensorMap &t13m, const CUtensorMap &t2q, const CUtensorMap &t2m,
                        const FusedArgs &a)
{
    const int NT = a.M > 8 ? 2 : 1;
    const int smem = fused_layout(NT).total + 1024;
    void (*kernel)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                   FusedArgs);
    if (mb == 4)
        kernel = NT == 1 ? fused_layer_kernel<4, 1> : fused_layer_kernel<4, 2>;
    else
        kernel = NT == 1 ? fused_layer_kernel<3, 1> : fused_layer_kernel<3, 2>;
    awq_status r = set_smem(kernel, smem);
    if (r) return r;
    return launch(kernel, dim3(sms), dim3(kFusedThreads), smem, 1, st, t13q, t13m, t2q, t2m, a);
}

}  // namespace awq
