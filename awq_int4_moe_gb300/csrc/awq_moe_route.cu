// Step (a): routing metadata, and the load-time 4-byte -> 3-byte metadata
// conversion.
//
// Routing follows 1Cat-vLLM #520 "Narrow Qwen3.8 AWQ active grouped decode",
// Purpose and Implementation: the (token, top-k slot) pairs are grouped into
// multi-row segments, one per distinct active expert, described by
// active_expert_ids (ascending) and CSR active_expert_offsets; the slots of a
// segment keep their original order (slot s = t*k + j).
//
// The compact conversion follows 1Cat-vLLM #522 "Coalesce AWQ QPN W13 compact
// metadata loads and enable compact metadata by default", Default switch: a
// {fp16 scale, u8 zero, pad} record becomes {fp16 scale, u8 zero}.
#include "awq_launch.cuh"
#include "awq_moe_kernels.cuh"
#include "awq_ptx.cuh"

namespace awq {

namespace {

constexpr int kRouteThreads = 256;

// In-place exclusive scan of data[0..n) by one block of NT threads; returns
// the total. Deterministic (integer adds in a fixed order).
template <int NT>
__device__ int block_exclusive_scan(int32_t *data, int n, int32_t *warp_sums)
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

}  // namespace

// One block. Slots whose id is outside [0, E) are reported in `status` and
// placed in an extra bucket E after every active segment, so no segment ever
// refers to them.
__global__ void __launch_bounds__(kRouteThreads)
route_kernel(const int32_t *topk_ids, int32_t S, int32_t num_experts, int32_t *active_ids,
             int32_t *offsets, int32_t *sorted_slots, int32_t *num_active, int32_t *status)
{
    __shared__ int32_t s_id[kMaxSlots];
    __shared__ int32_t s_cnt[kMaxExperts + 1];
    __shared__ int32_t s_start[kMaxExperts + 1];
    __shared__ int32_t s_run[kMaxExperts + 1];
    __shared__ int32_t s_fidx[kMaxExperts + 1];
    __shared__ int32_t s_warp[kRouteThreads / 32];

    const int tid = threadIdx.x;
    const int E = num_experts;
    for (int e = tid; e <= E; e += kRouteThreads) {
        s_cnt[e] = 0;
        s_run[e] = 0;
    }
    grid_dependency_wait();
    bool bad = false;
    for (int s = tid; s < S; s += kRouteThreads) {
        int e = topk_ids[s];
        if (e < 0 || e >= E) {
            bad = true;
            e = E;
        }
        s_id[s] = e;
    }
    if (bad) set_status(status, AWQ_ERR_BAD_EXPERT_ID);
    __syncthreads();
    grid_launch_dependents();
    for (int s = tid; s < S; s += kRouteThreads) atomicAdd(&s_cnt[s_id[s]], 1);
    __syncthreads();
    for (int e = tid; e <= E; e += kRouteThreads) {
        s_start[e] = s_cnt[e];
        s_fidx[e] = (e < E && s_cnt[e] > 0) ? 1 : 0;
    }
    __syncthreads();
    block_exclusive_scan<kRouteThreads>(s_start, E + 1, s_warp);
    const int A = block_exclusive_scan<kRouteThreads>(s_fidx, E + 1, s_warp);

    // Stable placement: one warp walks the slots in order, 32 at a time; lanes
    // holding the same expert are ranked by lane order.
    if (tid < 32) {
        const int lane = tid;
        const uint32_t lt = (1u << lane) - 1u;
        for (int b = 0; b < S; b += 32) {
            const int s = b + lane;
            const int e = s < S ? s_id[s] : -1;
            const uint32_t same = __match_any_sync(0xffffffffu, e);
            const int rank = __popc(same & lt);
            const int base = s < S ? s_run[e] : 0;
            __syncwarp();
            if (s < S) {
                sorted_slots[s_start[e] + base + rank] = s;
                if (rank == 0) s_run[e] = base + __popc(same);
            }
            __syncwarp();
        }
    }
    const int n_valid = s_start[E];
    for (int e = tid; e < E; e += kRouteThreads) {
        if (s_cnt[e] > 0) {
            active_ids[s_fidx[e]] = e;
            offsets[s_fidx[e]] = s_start[e];
        }
    }
    for (int i = A + tid; i < S; i += kRouteThreads) active_ids[i] = -1;
    for (int i = A + tid; i <= S; i += kRouteThreads) offsets[i] = n_valid;
    if (tid == 0) *num_active = A;
}

// Four records per thread: 16 bytes in, 12 bytes out (vectorised when both
// banks are suitably aligned), else byte by byte.
__global__ void prepare_compact_kernel(const uint8_t *meta4, uint8_t *meta3, int64_t n_records,
                                       int32_t vectorised)
{
    grid_dependency_wait();
    const int64_t n_quads = n_records / 4;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (vectorised) {
        for (int64_t q = i; q < n_quads; q += stride) {
            const uint4 w = ld_nc_v4(meta4 + 16 * q);
            uint32_t *o = reinterpret_cast<uint32_t *>(meta3 + 12 * q);
            o[0] = (w.x & 0x00FFFFFFu) | (w.y << 24);
            o[1] = ((w.y >> 8) & 0x0000FFFFu) | (w.z << 16);
            o[2] = ((w.z >> 16) & 0x000000FFu) | (w.w << 8);
        }
        for (int64_t r = 4 * n_quads + i; r < n_records; r += stride) {
            meta3[3 * r + 0] = meta4[4 * r + 0];
            meta3[3 * r + 1] = meta4[4 * r + 1];
            meta3[3 * r + 2] = meta4[4 * r + 2];
        }
    } else {
        for (int64_t r = i; r < n_records; r += stride) {
            meta3[3 * r + 0] = meta4[4 * r + 0];
            meta3[3 * r + 1] = meta4[4 * r + 1];
            meta3[3 * r + 2] = meta4[4 * r + 2];
        }
    }
}

}  // namespace awq
