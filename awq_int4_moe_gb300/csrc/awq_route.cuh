// Routing metadata as a block-level device function, shared by the
// standalone routing kernel and the fused layer kernel (which recomputes it
// in every CTA's prologue from the <= 256 slots of a decode batch).
#pragma once

#include <cstdint>

#include "awq_moe_kernels.cuh"
#include "awq_ptx.cuh"

namespace awq {

// In-place exclusive scan of data[0..n) by one block of NT threads; returns
// the total. Deterministic (integer adds in a fixed order).
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int32_t *data, int n, int32_t *warp_sums)
{
    const int per = (n + NT - 1) / NT;
    const int beg = min(n, static_cast<int>(threadIdx.x) * per);
    const int end = min(n, beg + per);
    int local = 0;
    for (int i = beg; i < end; ++i) local += data[i];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int v = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = lane < NT / 32 ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < NT / 32) warp_sums[lane] = w;
    }
    __syncthreads();
    int prefix = (warp > 0 ? warp_sums[warp - 1] : 0) + v - local;
    const int total = warp_sums[NT / 32 - 1];
    for (int i = beg; i < end; ++i) {
        const int c = data[i];
        data[i] = prefix;
        prefix += c;
    }
    __syncthreads();
    return total;
}


// Groups the S slots (slot s = t*k + j) by expert id with one block of NT
// threads. Writes active_ids[0..A) ascending (rest of [0, S) = -1),
// offsets[0..S] (CSR; entries past A = number of valid slots) and
// sorted_slots[0..S) (stable: slots of a segment in ascending order).
// Ids outside [0, E) are reported in `status` and go to an extra bucket E
// after every segment. Shared scratch: s_id[S], s_wcnt[NT/32][E+1],
// s_start[E+1], s_fidx[E+1], s_warp[NT/32]. Returns A in every thread;
// outputs are complete after the caller's next __syncthreads().
//
// Stable placement in parallel: warp w owns the slots [w C, (w+1) C); it
// counts its slots per expert, the counts are turned into per-(warp,
// expert) starting rows (expert start + the counts of the warps before),
// and each warp then places its own slots in order, 32 at a time.
template <int NT>
__device__ int route_block(const int32_t *topk_ids, int S, int E, int32_t *s_id, int32_t *s_wcnt,
                           int32_t *s_start, int32_t *s_fidx, int32_t *s_warp, int32_t *active_ids,
                           int32_t *offsets, int32_t *sorted_slots, int32_t *status)
{
    constexpr int NW = NT / 32;
    constexpr int kPer = kMaxSlots / NT;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t lt = (1u << lane) - 1u;
    for (int i = tid; i < NW * (E + 1); i += NT) s_wcnt[i] = 0;
    // all loads of the ids in flight at once
    int idv[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int s = tid + i * NT;
        idv[i] = s < S ? topk_ids[s] : 0;
    }
    bool bad = false;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int s = tid + i * NT;
        if (s < S) {
            int e = idv[i];
            if (e < 0 || e >= E) {
                bad = true;
                e = E;
            }
            s_id[s] = e;
        }
    }
    if (bad) set_status(status, AWQ_ERR_BAD_EXPERT_ID);
    __syncthreads();
    // per-warp counts over the warp's own slots
    const int C = ((S + NW - 1) / NW + 31) / 32 * 32;
    const int wbeg = min(S, warp * C), wend = min(S, wbeg + C);
    int32_t *mine = s_wcnt + warp * (E + 1);
    for (int b = wbeg; b < wend; b += 32) {
        const int s = b + lane;
        const int e = s < wend ? s_id[s] : -1;
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && (same & lt) == 0) mine[e] += __popc(same);
        __syncwarp();
    }
    __syncthreads();
    for (int e = tid; e <= E; e += NT) {
        int tot = 0;
        for (int w = 0; w < NW; ++w) tot += s_wcnt[w * (E + 1) + e];
        s_start[e] = tot;
        s_fidx[e] = (e < E && tot > 0) ? 1 : 0;
    }
    __syncthreads();
    block_exclusive_scan<NT>(s_start, E + 1, s_warp);
    const int A = block_exclusive_scan<NT>(s_fidx, E + 1, s_warp);
    // per-(warp, expert) starting rows
    for (int e = tid; e <= E; e += NT) {
        int run = s_start[e];
        for (int w = 0; w < NW; ++w) {
            const int c = s_wcnt[w * (E + 1) + e];
            s_wcnt[w * (E + 1) + e] = run;
            run += c;
        }
    }
    __syncthreads();
    for (int b = wbeg; b < wend; b += 32) {
        const int s = b + lane;
        const int e = s < wend ? s_id[s] : -1;
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        const int base = e >= 0 ? mine[e] : 0;
        __syncwarp();
        if (e >= 0) {
            sorted_slots[base + __popc(same & lt)] = s;
            if ((same & lt) == 0) mine[e] = base + __popc(same);
        }
        __syncwarp();
    }
    const int n_valid = s_start[E];
    for (int e = tid; e < E; e += NT) {
        if (s_start[e + 1] > s_start[e]) {
            active_ids[s_fidx[e]] = e;
            offsets[s_fidx[e]] = s_start[e];
        }
    }
    for (int i = A + tid; i < S; i += NT) active_ids[i] = -1;
    for (int i = A + tid; i <= S; i += NT) offsets[i] = n_valid;
    return A;
}

}  // namespace awq
