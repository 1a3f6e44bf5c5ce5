// Steps (b) and (c): the grouped W13 + SwiGLU GEMM and the grouped W2 GEMM
// with the router-weighted top-k reduction, each ONE launch over all active
// expert segments (1Cat-vLLM #520 "Narrow Qwen3.8 AWQ active grouped decode",
// Purpose: the active-stage op is called once per stage instead of once per
// segment; Implementation: offsets-based GEMM, grouped-active exact W2
// reduction).
//
// Data path (both stages): one elected thread issues TMA tensor copies of a
// CTA's packed int4 weight tile and its metadata records into shared memory
// (128-byte swizzled lines for the weights, so the fragment loads below are
// bank-conflict free); warps expand nibbles to exact fp16 (q - zero) pairs in
// registers and feed m16n8k16 tensor-core MMAs with the weights on the M side
// (16 output columns) and up to 8 token rows on the N side. Each group of 32
// k is accumulated separately and scaled once by its fp16 scale in fp32, so
// dequantisation is w = (q - zero) * scale with no intermediate rounding.
//
// K-index permutation. Inside one group of 32 k (4 packed words of a column),
// MMA step s (0, 1) of thread (g = lane/4, t = lane%4) takes word t of its two
// columns; fragment halves (lo, hi) of register h (0: k 2t..2t+1, 1: k 2t+8..)
// hold nibbles (2s + h, 2s + h + 4). The B operand (tokens) is laid out with
// the same permutation: k = 8t + {0, 4, 1, 5, 2, 6, 3, 7} within each group.
#include <cuda_fp16.h>

#include "awq_launch.cuh"
#include "awq_moe_kernels.cuh"
#include "awq_ptx.cuh"
#include "awq_dequant.cuh"
#include "awq_nvfp4.cuh"

namespace awq {

// ------------------------------------------------------------------------ W13
//
// grid (I/8, A_max), 256 threads, prepared banks. CTA (j, a) computes the
// piece j of segment a: gate columns [8j, 8j+8) and the matching up columns
// [I+8j, I+8j+8), one 16-row MMA tile (rows 0-7 gate, 8-15 up), over the
// whole K. One bulk copy brings the piece's 20 KB of packed weights and its
// metadata; warp w takes groups 10w .. 10w+9. The segment's rows are done 8
// at a time: each lane loads its x fragments (row g of the block, its
// warp's groups) straight from global memory, the eight warps' partial tiles
// are summed in a fixed order, and SwiGLU is applied in registers (a lane
// holds the gate and up value of the same column and token).
// Four CTAs per multiprocessor (64 registers a thread): each CTA is one
// weight fetch and a short computation, so residency hides the fetches
// (measured 2-4 % faster than three CTAs at 72 registers; five spill).
constexpr int kW13Blocks = 2;     // 8-row blocks that share one expansion of each group

template <int MB>
__global__ void __launch_bounds__(kW13Threads, 4)
w13_swiglu_kernel(StageArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((128 - (smem_u32(smem_raw) & 127)) & 127);
    constexpr int kMeta = piece_meta_bytes(MB);
    uint8_t *sq = smem;
    uint8_t *sm = sq + kPieceQ;
    float *red = reinterpret_cast<float *>(sm + (kMeta + 127) / 128 * 128);   // [block][warp][lane] float4
    uint64_t *bar = reinterpret_cast<uint64_t *>(red + kW13Blocks * kW13RedBytes / 4);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int j = blockIdx.x, a = blockIdx.y;
    const int I = args.inter;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    grid_dependency_wait();
    if (tid == 0) trace_start(args.trace, 0);

    // a < min(M k, E), inside the routing arrays: these loads go out together
    // with the active count's instead of after it
    const int A = *args.num_active;
    const int e = args.active_ids[a];
    const int row0 = args.offsets[a];
    const int rows = args.offsets[a + 1] - row0;
    if (a >= A) return;
    if (e < 0 || e >= args.num_experts) {
        if (tid == 0) set_status(args.status, AWQ_ERR_BAD_EXPERT_ID);
        return;
    }
    if (tid == 0) {
        const int64_t piece = static_cast<int64_t>(e) * (I / kPieceCols) + j;
        mbar_arrive_expect_tx(bar, kPieceQ + kMeta);
        bulk_load(sq, reinterpret_cast<const uint8_t *>(args.w13_q) + piece * kPieceQ, kPieceQ, bar);
        bulk_load(sm, args.w13_meta + piece * kMeta, kMeta, bar);
    }
    grid_launch_dependents();

    const uint32_t sq_base = smem_u32(sq), sm_base = smem_u32(sm);
    bool ok = true;

    // The segment's rows go kW13Blocks blocks of 8 at a time: each group's
    // weights are expanded once per chunk and every block of the chunk runs
    // its MMAs on them (a lane's x fragment of a block: row g of the block);
    // a chunk of one block keeps the one-block loop, whose x loads all go out
    // before the first MMA.
    for (int rt0 = 0; rt0 < rows; rt0 += 8 * kW13Blocks) {
        const bool more = rt0 + 8 < rows;        // a second block in this chunk
        float acc[kW13Blocks][4];
#pragma unroll
        for (int b = 0; b < kW13Blocks; ++b)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[b][v] = 0.f;
        if (!more) {
            // one block: every group's x fragment is loaded first (one load
            // latency for all), and each group is expanded for this block alone
            uint4 xf[kW13GroupsPerWarp];
            {
                const bool live = rt0 + g < rows;
                const int tok = live ? args.sorted_slots[row0 + rt0 + g] / args.top_k : 0;
                const uint16_t *xr = args.x + static_cast<int64_t>(tok) * kHidden +
                                     warp * kW13GroupsPerWarp * kGroup + t * 8;
#pragma unroll
                for (int gi = 0; gi < kW13GroupsPerWarp; ++gi)
                    xf[gi] = live ? ld_nc_v4(xr + gi * kGroup) : make_uint4(0, 0, 0, 0);
            }
            if (rt0 == 0) {
                ok = mbar_wait_bounded(bar, 0, args.timeout_ns);
                if (!ok && tid == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
            }
#pragma unroll
            for (int gi = 0; gi < kW13GroupsPerWarp; ++gi) {
                const int grp = warp * kW13GroupsPerWarp + gi;
                const uint2 q = lds_v2(sq_base + ((grp * 4 + t) * kPieceCols + g) * 8);
                if constexpr (MB == 2) {
                    // NVFP4: the lane's words cover k 8t .. 8t+7 of the group, i.e.
                    // scale block t / 2 of the gate and up records of column g
                    const uint32_t r = lds_u32(sm_base + (grp * kPieceCols + g) * 4);
                    group_tile_mma_nv(acc[0], q.x, q.y, e4m3_scale_pair(r >> (8 * (t >> 1)) & 0xFFu),
                                      e4m3_scale_pair(r >> (16 + 8 * (t >> 1)) & 0xFFu), permute_k8(xf[gi]));
                } else {
                    const MetaPair m = load_meta_pair<MB>(sm_base + (grp * kPieceCols + g) * 2 * MB);
                    group_tile_mma(acc[0], q.x, q.y, m.zg2, m.zu2, half_bits_to_float(m.sg),
                                   half_bits_to_float(m.su), permute_k8(xf[gi]));
                }
            }
        } else {
            // two blocks: each group's weights expanded once, both blocks' MMAs
            // on them (x fragments loaded per group)
            const uint16_t *xr[kW13Blocks];
            bool live[kW13Blocks];
#pragma unroll
            for (int b = 0; b < kW13Blocks; ++b) {
                const int r = rt0 + 8 * b + g;
                live[b] = r < rows;
                const int tok = live[b] ? args.sorted_slots[row0 + r] / args.top_k : 0;
                xr[b] = args.x + static_cast<int64_t>(tok) * kHidden + warp * kW13GroupsPerWarp * kGroup + t * 8;
            }
            if (rt0 == 0) {
                ok = mbar_wait_bounded(bar, 0, args.timeout_ns);
                if (!ok && tid == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
            }
#pragma unroll
            for (int gi = 0; gi < kW13GroupsPerWarp; ++gi) {
                const int grp = warp * kW13GroupsPerWarp + gi;
                uint4 xb[kW13Blocks];
#pragma unroll
                for (int b = 0; b < kW13Blocks; ++b)
                    xb[b] = live[b] ? permute_k8(ld_nc_v4(xr[b] + gi * kGroup)) : make_uint4(0, 0, 0, 0);
                const uint2 q = lds_v2(sq_base + ((grp * 4 + t) * kPieceCols + g) * 8);
                if constexpr (MB == 2) {
                    const uint32_t r = lds_u32(sm_base + (grp * kPieceCols + g) * 4);
                    const NvTile f = nv_tile(q.x, q.y, e4m3_scale_pair(r >> (8 * (t >> 1)) & 0xFFu),
                                             e4m3_scale_pair(r >> (16 + 8 * (t >> 1)) & 0xFFu));
#pragma unroll
                    for (int b = 0; b < kW13Blocks; ++b) {
                        mma_16816(acc[b], f.a[0], f.a[1], f.a[2], f.a[3], xb[b].x, xb[b].y, acc[b]);
                        mma_16816(acc[b], f.a[4], f.a[5], f.a[6], f.a[7], xb[b].z, xb[b].w, acc[b]);
                    }
                } else {
                    const MetaPair m = load_meta_pair<MB>(sm_base + (grp * kPieceCols + g) * 2 * MB);
                    const GroupFrag f = group_frag(q.x, q.y, m.zg2, m.zu2);
                    const float sg = half_bits_to_float(m.sg), su = half_bits_to_float(m.su);
#pragma unroll
                    for (int b = 0; b < kW13Blocks; ++b) frag_mma(acc[b], f, sg, su, xb[b]);
                }
            }
        }
#pragma unroll
        for (int b = 0; b < kW13Blocks; ++b) {
            if (b > 0 && !more) break;
            *reinterpret_cast<float4 *>(red + ((b * (kW13Threads / 32) + warp) * 32 + lane) * 4) =
                make_float4(acc[b][0], acc[b][1], acc[b][2], acc[b][3]);
        }
        __syncthreads();
        if (warp < kW13Blocks && rt0 + 8 * warp < rows) {
            // warp b finishes block b: fixed-order sum over the warps; lane
            // (g, t) holds gate (v0, v1) and up (v2, v3) of column 8j+g for
            // rows rt+2t, rt+2t+1
            const int rt = rt0 + 8 * warp;
            const float *rb = red + warp * (kW13Threads / 32) * 32 * 4;
            float4 sum = *reinterpret_cast<const float4 *>(rb + lane * 4);
#pragma unroll
            for (int w = 1; w < kW13Threads / 32; ++w) {
                const float4 v = *reinterpret_cast<const float4 *>(rb + (w * 32 + lane) * 4);
                sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
            }
            const int n = kPieceCols * j + g;
            if constexpr (MB == 2) {
                // NVFP4: the weights entered as w 2^-7; times 2^7 and the expert's W13 global
                const float g13 = 128.f * args.global_scale[2 * e];
                sum.x *= g13; sum.y *= g13; sum.z *= g13; sum.w *= g13;
            }
            const float h0 = silu_f(sum.x) * sum.z, h1 = silu_f(sum.y) * sum.w;
            const int r0 = rt + 2 * t;
            const uint16_t b0 = f2h_bits(h0), b1 = f2h_bits(h1);
            const int64_t at0 = static_cast<int64_t>(row0 + r0) * I + n, at1 = at0 + I;
            if (ok && r0 < rows) args.h_out[at0] = b0;
            if (ok && r0 + 1 < rows) args.h_out[at1] = b1;
            // the residue plane (fp16 of h - fp16(h)), when the tensor-core W2 follows
            if (args.h_lo && ok && r0 < rows) args.h_lo[at0] = f2h_bits(h0 - __half2float(__ushort_as_half(b0)));
            if (args.h_lo && ok && r0 + 1 < rows) args.h_lo[at1] = f2h_bits(h1 - __half2float(__ushort_as_half(b1)));
        }
        __syncthreads();
    }
    if (!ok) mbar_wait_bounded(bar, 0, args.timeout_ns);
    if (tid == 0) trace_end(args.trace, 0);
}

// ------------------------------------------------------------------------- W2
//
// grid (8, H/32), cluster (8, 1, 1), 128 threads. Cluster = one 32-column
// tile of the output. The work is cut into items of at most 16 rows of one
// segment (a segment's rows in order); item i is handled by CTA i % 8 and,
// inside it, by warp (i / 8) % 4 through that warp's 2-stage TMA ring of
// weight tiles. For each item the warp expands the tile's weights once per
// 160-row K part into registers, streams the item's token blocks through
// them (the 32 x rows product over K = I), weights every row by its router
// weight and adds it into the warp's fp32 accumulator [M][32] of token rows.
// Accumulators are summed warp -> CTA -> cluster in a fixed order and written
// as fp16 (tokens split across the cluster's CTAs).
//
// TMA boxes (2D views of the prepared banks), one per 160-row K part kp:
// q 20 lines -> slot kp [20 rows][32 words], 128 B swizzle; meta 5 rows ->
// meta slot kp [5 groups][32 records].
template <int MB>
__global__ void __launch_bounds__(kW2Threads)
w2_reduce_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tm,
                 StageArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const int I = args.inter, M = args.M, k = args.top_k;
    const int q_stage = w2_q_stage_bytes(I), m_stage = w2_meta_stage_bytes(I, MB);
    uint8_t *sq = smem;                                           // [warp][stage] q
    uint8_t *sm = sq + kW2Warps * kW2Stages * q_stage;            // [warp][stage] meta
    float *acc_all = reinterpret_cast<float *>(sm + kW2Warps * kW2Stages * m_stage);
    int32_t *s_item = reinterpret_cast<int32_t *>(acc_all + kW2Warps * M * kW2ColTile);   // [kW2MaxItems]
    int32_t *s_tok = s_item + kW2MaxItems;                                                // [M * k]
    float *s_wgt = reinterpret_cast<float *>(s_tok + M * k);                              // [M * k]
    uint64_t *bars = reinterpret_cast<uint64_t *>(s_wgt + M * k);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int rank = static_cast<int>(cluster_ctarank());
    const int ctile = blockIdx.y;
    const int Qg = (g >> 1) | ((g & 1) << 2);     // conflict-free column quad
    const int n_groups = I / kGroup;
    const int KP = I / 160;
    const uint32_t q_bytes = (I / 8) * 128, m_bytes = n_groups * 32 * MB;
    constexpr int kMSlot = w2_meta_slot(MB);

    float *acc = acc_all + warp * M * kW2ColTile;
    for (int i = lane; i < M * kW2ColTile; i += 32) acc[i] = 0.f;
    if (lane == 0) {
        for (int s = 0; s < kW2Stages; ++s) mbar_init(&bars[warp * kW2Stages + s], 1);
        fence_barrier_init();
        if (warp == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tm);
        }
    }
    __syncwarp();
    grid_dependency_wait();

    const int A = *args.num_active;
    // Work items: each segment's rows in chunks of kW2ItemRows, numbered
    // segment by segment; item = segment << 15 | (rows - 1) << 11 | first
    // row (in sorted-row order). Item i goes to CTA i % 8 of the cluster and
    // there to warp (i / 8) % 4: a static split (so sums keep a fixed order)
    // whose pieces are bounded, so a long segment is spread over several
    // warps instead of holding one. Every row's token and router weight are
    // staged in shared memory once, off the items' dependency chains.
    __shared__ int32_t s_wsum[kW2Warps];
    int n_items;
    {
        // loads batched so that the prologue costs a few round trips, not one
        // per row or segment
        // Neither the slot nor the offset loads wait for the active count: all
        // S = M k sorted slots are valid slot indices, and the segments are
        // split over the threads by the bound min(S, E) on the count.
        constexpr int kRowsPer = kStagedMaxSlots / kW2Threads;
        constexpr int kSegsPer = kMaxExperts / kW2Threads;
        const int S = M * k;
        const int a_max = min(S, args.num_experts);
        int sl[kRowsPer];
#pragma unroll
        for (int i = 0; i < kRowsPer; ++i) {
            const int r = tid + i * kW2Threads;
            sl[i] = r < S ? args.sorted_slots[r] : 0;
        }
        // this thread's segments [a0, a0 + per) and their row offsets
        const int per = (a_max + kW2Threads - 1) / kW2Threads;
        const int a0 = tid * per;
        int ov[kSegsPer + 1];
#pragma unroll
        for (int i = 0; i <= kSegsPer; ++i)
            ov[i] = (i <= per && a0 + i <= a_max) ? args.offsets[a0 + i] : 0;
        float wv[kRowsPer];
#pragma unroll
        for (int i = 0; i < kRowsPer; ++i) {
            const int r = tid + i * kW2Threads;
            wv[i] = r < S ? args.topk_weights[sl[i]] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kRowsPer; ++i) {
            const int r = tid + i * kW2Threads;
            if (r < S) {
                s_tok[r] = sl[i] / k;
                s_wgt[r] = wv[i];
            }
        }
        int cnt = 0;
#pragma unroll
        for (int i = 0; i < kSegsPer; ++i)
            if (i < per && a0 + i < A) cnt += (ov[i + 1] - ov[i] + kW2ItemRows - 1) / kW2ItemRows;
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) s_wsum[warp] = incl;
        __syncthreads();
        int pos = incl - cnt;
        n_items = 0;
        for (int w = 0; w < kW2Warps; ++w) {
            if (w < warp) pos += s_wsum[w];
            n_items += s_wsum[w];
        }
#pragma unroll
        for (int i = 0; i < kSegsPer; ++i) {
            const int a = a0 + i;
            if (i < per && a < A) {
                const int rows = ov[i + 1] - ov[i];
                for (int r = 0; r < rows; r += kW2ItemRows)
                    s_item[pos++] = (a << 15) | ((min(kW2ItemRows, rows - r) - 1) << 11) | (ov[i] + r);
            }
        }
        __syncthreads();
    }
    // m-th item of this warp
    auto item_of = [&](int m) { return rank + kW2Cluster * (warp + kW2Warps * m); };
    auto expert_ok = [&](int e) { return e >= 0 && e < args.num_experts; };
    // Issue item m's weights into its stage (lane 0); every lane returns
    // whether a copy is now in flight for it.
    auto issue = [&](int m) {
        const int a = s_item[item_of(m)] >> 15;
        const int e = args.active_ids[a];
        if (!expert_ok(e)) {
            if (lane == 0) set_status(args.status, AWQ_ERR_BAD_EXPERT_ID);
            return false;
        }
        const int st = m % kW2Stages;
        uint64_t *bar = &bars[warp * kW2Stages + st];
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, q_bytes + m_bytes);
            for (int kp = 0; kp < KP; ++kp) {
                const int tile = (e * KP + kp) * kColTiles + ctile;
                tma_load_2d(sq + (warp * kW2Stages + st) * q_stage + kp * kW2PartSlot, &tq, bar, 0,
                            tile * kW2TileKK);
                tma_load_2d(sm + (warp * kW2Stages + st) * m_stage + kp * kMSlot, &tm, bar, 0, tile * 5);
            }
        }
        return true;
    };
    // in_flight[st]: a copy issued into stage st and not yet waited for
    // issued_m[st]: the segment index whose copy went into stage st last
    bool in_flight[kW2Stages];
    int issued_m[kW2Stages];
#pragma unroll
    for (int s = 0; s < kW2Stages; ++s) {
        in_flight[s] = false;
        issued_m[s] = s;
    }
    bool ok = true;
    for (int m = 0; m < kW2Stages && item_of(m) < n_items; ++m) in_flight[m] = issue(m);
    grid_launch_dependents();

    // Activation fragments of an item's first token block in K part 0 (row
    // first + g): the next item's go out while the current item computes.
    auto load_first = [&](int mm, uint4 (&hb)[5]) {
        const int it2 = s_item[item_of(mm)];
        const int rb = it2 & 2047, re = rb + ((it2 >> 11) & 15) + 1;
        const bool hrow = rb + g < re;
        const uint16_t *hp = args.h_in + static_cast<int64_t>(rb + (hrow ? g : 0)) * I + t * 8;
#pragma unroll
        for (int c5 = 0; c5 < 5; ++c5) hb[c5] = hrow ? ld_v4(hp + c5 * kGroup) : make_uint4(0, 0, 0, 0);
    };
    uint4 hpre[5];
    if (item_of(0) < n_items) load_first(0, hpre);

    for (int m = 0; item_of(m) < n_items; ++m) {
        const int item = s_item[item_of(m)];
        // sorted rows [r_begin, rows) of segment item >> 15
        const int r_begin = item & 2047, rows = r_begin + ((item >> 11) & 15) + 1;
        uint4 hfirst[5];
#pragma unroll
        for (int c5 = 0; c5 < 5; ++c5) hfirst[c5] = hpre[c5];
        if (item_of(m + 1) < n_items) load_first(m + 1, hpre);
        const int st = m % kW2Stages;
        const uint32_t parity = (m / kW2Stages) & 1;
        if (!in_flight[st]) break;                       // bad expert id, reported at issue
        if (!mbar_wait_bounded(&bars[warp * kW2Stages + st], parity, args.timeout_ns)) {
            if (lane == 0) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
            ok = false;
            break;
        }
        in_flight[st] = false;
        const uint32_t sq_base = smem_u32(sq + (warp * kW2Stages + st) * q_stage);
        const uint32_t sm_base = smem_u32(sm + (warp * kW2Stages + st) * m_stage);
        // Per 160-row K part: the tile's 5 groups x 2 column halves expanded
        // once into registers, then the segment's token blocks streamed
        // through them (activation fragments of the next block in flight
        // while the current one is multiplied).
        for (int kp = 0; kp < KP; ++kp) {
            GroupFrag fr[5][2];
            float sc[5][2][2];
#pragma unroll
            for (int c5 = 0; c5 < 5; ++c5) {
                const int kk = 4 * c5 + t;              // row inside the K part's 20
                const uint4 q = lds_v4(sq_base + kp * kW2PartSlot + kk * 128 + ((Qg ^ (kk & 7)) << 4));
                const Meta4<MB> mt = load_meta4<MB>(sm_base + kp * kMSlot + c5 * 32 * MB + Qg * 4 * MB);
                fr[c5][0] = group_frag(q.x, q.y, mt.z2[0], mt.z2[1]);
                fr[c5][1] = group_frag(q.z, q.w, mt.z2[2], mt.z2[3]);
#pragma unroll
                for (int T = 0; T < 2; ++T) {
                    sc[c5][T][0] = half_bits_to_float(mt.s[2 * T]);
                    sc[c5][T][1] = half_bits_to_float(mt.s[2 * T + 1]);
                }
            }
            // activation fragments of block rt: row rt + g, this K part
            auto load_h = [&](int rt, uint4 (&hb)[5]) {
                const bool hrow = rt + g < rows;
                const uint16_t *hp = args.h_in + static_cast<int64_t>(rt + (hrow ? g : 0)) * I + kp * 160 + t * 8;
#pragma unroll
                for (int c5 = 0; c5 < 5; ++c5)
                    hb[c5] = hrow ? ld_v4(hp + c5 * kGroup) : make_uint4(0, 0, 0, 0);
            };
            uint4 hcur[5], hnext[5];
            if (kp == 0) {
#pragma unroll
                for (int c5 = 0; c5 < 5; ++c5) hcur[c5] = hfirst[c5];
            } else {
                load_h(r_begin, hcur);
            }
            for (int rt = r_begin; rt < rows; rt += 8) {
                if (rt + 8 < rows) load_h(rt + 8, hnext);
                // router weight and token of the two rows this lane accumulates
                int tok[2];
                float wgt[2];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int j = rt + 2 * t + c;
                    tok[c] = -1;
                    wgt[c] = 0.f;
                    if (j < rows) {
                        tok[c] = s_tok[j];
                        wgt[c] = s_wgt[j];
                    }
                }
                float accs[2][4];
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) accs[i][j] = 0.f;
#pragma unroll
                for (int c5 = 0; c5 < 5; ++c5) {
                    const uint4 xb = permute_k8(hcur[c5]);
                    frag_mma(accs[0], fr[c5][0], sc[c5][0][0], sc[c5][0][1], xb);
                    frag_mma(accs[1], fr[c5][1], sc[c5][1][0], sc[c5][1][1], xb);
                }
#pragma unroll
                for (int T = 0; T < 2; ++T)
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int c = v & 1;
                        if (tok[c] >= 0) {
                            const int n = 4 * Qg + 2 * T + (v >> 1);
                            red_shared_add_f32(acc + tok[c] * kW2ColTile + n, wgt[c] * accs[T][v]);
                        }
                    }
#pragma unroll
                for (int c5 = 0; c5 < 5; ++c5) hcur[c5] = hnext[c5];
            }
        }
        __syncwarp();
        if (item_of(m + kW2Stages) < n_items) {
            if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            in_flight[st] = issue(m + kW2Stages);
            issued_m[st] = m + kW2Stages;
        }
    }
    // Let any copy still in flight land before this CTA's memory is released.
    for (int s = 0; s < kW2Stages; ++s)
        if (in_flight[s])
            mbar_wait_bounded(&bars[warp * kW2Stages + s], (issued_m[s] / kW2Stages) & 1,
                              args.timeout_ns);
    __syncthreads();
    // warp partials -> CTA sum (fixed order) in warp 0's buffer
    for (int i = tid; i < M * kW2ColTile; i += kW2Threads) {
        float s = acc_all[i];
#pragma unroll
        for (int w = 1; w < kW2Warps; ++w) s += acc_all[w * M * kW2ColTile + i];
        acc_all[i] = s;
    }
    cluster_sync();
    // CTA sums -> cluster sum (fixed order); CTA r writes float4 chunks f = r mod 8
    const int n_chunks = M * (kW2ColTile / 4);
    for (int f = rank + kW2Cluster * tid; f < n_chunks; f += kW2Cluster * kW2Threads) {
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < kW2Cluster; ++r) {
            const float4 v = ld_shared_cluster_f4(map_shared_rank(acc_all + 4 * f, r));
            s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
        }
        const int tok = f / (kW2ColTile / 4), c4 = f - tok * (kW2ColTile / 4);
        uint2 o;
        o.x = static_cast<uint32_t>(f2h_bits(s.x)) | (static_cast<uint32_t>(f2h_bits(s.y)) << 16);
        o.y = static_cast<uint32_t>(f2h_bits(s.z)) | (static_cast<uint32_t>(f2h_bits(s.w)) << 16);
        if (ok)
            *reinterpret_cast<uint2 *>(args.out + static_cast<int64_t>(tok) * kHidden +
                                       ctile * kW2ColTile + 4 * c4) = o;
    }
    cluster_sync();
}

awq_status launch_w13(int mb, dim3 grid, cudaStream_t st, const StageArgs &a)
{
    const int smem = w13_smem_bytes(mb) + (kW13Blocks - 1) * kW13RedBytes;   // one hand-off slot per block
    auto kernel = mb == 4 ? w13_swiglu_kernel<4> : mb == 3 ? w13_swiglu_kernel<3> : w13_swiglu_kernel<2>;
    awq_status r = set_smem(kernel, smem);
    if (r) return r;
    return launch(kernel, grid, dim3(kW13Threads), smem, 1, st, a);
}

awq_status launch_w2(int mb, dim3 grid, cudaStream_t st, const CUtensorMap &tq,
                     const CUtensorMap &tm, const StageArgs &a)
{
    const int smem = w2_smem_bytes(a.inter, mb, a.M, a.top_k);
    auto kernel = mb == 4 ? w2_reduce_kernel<4> : w2_reduce_kernel<3>;
    awq_status r = set_smem(kernel, smem);
    if (r) return r;
    return launch(kernel, grid, dim3(kW2Threads), smem, kW2Cluster, st, tq, tm, a);
}

}  // namespace awq
