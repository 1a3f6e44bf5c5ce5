// Step (a): routing metadata, the router from logits that produces its
// inputs, and the load-time 4-byte -> 3-byte metadata conversion.
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
#include "awq_route.cuh"
#include "awq_router.cuh"

namespace awq {



// One block (standalone routing call).
__global__ void __launch_bounds__(kRouteThreads)
route_kernel(const int32_t *topk_ids, int32_t S, int32_t num_experts, int32_t *active_ids,
             int32_t *offsets, int32_t *sorted_slots, int32_t *num_active, int32_t *status)
{
    // dynamic shared memory: s_id[S], s_wcnt[8][E+1], s_start[E+1], s_fidx[E+1]
    extern __shared__ int32_t s_route[];
    __shared__ int32_t s_warp[kRouteThreads / 32];
    const int E1 = num_experts + 1;
    int32_t *s_id = s_route;
    int32_t *s_wcnt = s_id + S;
    int32_t *s_start = s_wcnt + (kRouteThreads / 32) * E1;
    int32_t *s_fidx = s_start + E1;
    grid_dependency_wait();
    grid_launch_dependents();
    const int A = route_block<kRouteThreads>(topk_ids, S, num_experts, s_id, s_wcnt, s_start, s_fidx, s_warp,
                                             active_ids, offsets, sorted_slots, status);
    if (threadIdx.x == 0) *num_active = A;
}

// Router from logits (standalone call): warp w of block b routes token 8b + w.
__global__ void __launch_bounds__(kRouterWarps * 32)
router_topk_kernel(const float *logits, int32_t M, int32_t top_k, int32_t *topk_ids,
                   float *topk_weights)
{
    grid_dependency_wait();
    grid_launch_dependents();
    const int tok = blockIdx.x * kRouterWarps + (threadIdx.x >> 5);
    if (tok >= M) return;
    warp_router_topk<kRouterExperts / 32>(logits + static_cast<int64_t>(tok) * kRouterExperts, top_k,
                                          threadIdx.x & 31, topk_ids + static_cast<int64_t>(tok) * top_k,
                                          topk_weights + static_cast<int64_t>(tok) * top_k);
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
