// Kernel-side declarations shared by the translation units of the CUDA
// library: launch constants, argument block and kernel prototypes.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/awq_moe.h"

namespace awq {

// ----------------------------------------------------------- fixed geometry
constexpr int kHidden = 2560;           // W13 K, W2 N
constexpr int kGroup = 32;              // quantisation group along K
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 16;
constexpr int kMaxSlots = AWQ_MAX_TOKENS * kMaxTopK;

// W13: a cluster of 4 CTAs shares one (segment, 32-column gate/up slab);
// CTA r of the cluster covers K rows [r*640, (r+1)*640).
constexpr int kW13Cluster = 4;
constexpr int kW13Threads = 128;                               // 4 warps
constexpr int kW13KRows = kHidden / kW13Cluster;               // 640 k per CTA
constexpr int kW13KK = kW13KRows / 8;                          // 80 packed rows
constexpr int kW13Groups = kW13KRows / kGroup;                 // 20 groups
constexpr int kW13GroupsPerWarp = kW13Groups / (kW13Threads / 32);  // 5
constexpr int kW13QBytes = kW13KK * 2 * 128;                   // gate+up, 128 B lines
constexpr int kW13XRowBytes = (kW13KK + 4) * 16;               // padded x row
constexpr int kW13XBytes = 8 * kW13XRowBytes;
constexpr int kW13RedBytes = 4 * 4 * 32 * 16;                  // warps x tiles x lanes x float4
constexpr int kW13CsumBytes = 4 * 32 * 16;

__host__ __device__ constexpr int w13_meta_bytes(int mb) { return kW13Groups * 2 * 32 * mb; }
__host__ __device__ constexpr int w13_smem_bytes(int mb)
{
    return 1024 /*align slack*/ + kW13QBytes + ((w13_meta_bytes(mb) + 127) / 128) * 128 +
           kW13XBytes + kW13RedBytes + kW13CsumBytes + 64;
}

// W2: a cluster of 8 CTAs shares one 32-column output tile; segment a goes
// to CTA a % 8, and within it to warp (a / 8) % 4, each warp with its own
// 2-stage TMA ring.
constexpr int kW2Cluster = 8;
constexpr int kW2Threads = 128;
constexpr int kW2Warps = kW2Threads / 32;
constexpr int kW2Stages = 2;
constexpr int kW2ColTile = 32;

__host__ __device__ constexpr int w2_q_stage_bytes(int inter)
{
    return ((inter / 8) * 128 + 1023) / 1024 * 1024;
}
__host__ __device__ constexpr int w2_meta_stage_bytes(int inter, int mb)
{
    return ((inter / kGroup) * 32 * mb + 127) / 128 * 128;
}
__host__ __device__ constexpr int w2_smem_bytes(int inter, int mb, int M)
{
    return 1024 + kW2Warps * kW2Stages * (w2_q_stage_bytes(inter) + w2_meta_stage_bytes(inter, mb)) +
           kW2Warps * M * kW2ColTile * 4 + 128;
}

struct StageArgs {
    const uint16_t *x;             // fp16[M][H]
    const uint16_t *h_in;          // fp16[S][I] (W2)
    uint16_t *h_out;               // fp16[S][I] (W13)
    const float *topk_weights;     // f32[M][k]
    uint16_t *out;                 // fp16[M][H]
    const int32_t *active_ids;
    const int32_t *offsets;
    const int32_t *sorted_slots;
    const int32_t *num_active;
    int32_t *status;
    int32_t M, top_k, num_experts, inter;
    uint64_t timeout_ns;
};

// Arguments of the fused (single-launch) decode layer kernel. Workspace
// buffers are carved by the host from the caller's workspace.
struct FusedArgs {
    const uint16_t *x;            // fp16[M][H]
    const int32_t *topk_ids;      // i32[M][k]
    const float *topk_weights;    // f32[M][k]
    uint16_t *out;                // fp16[M][H]
    uint16_t *hw;                 // fp16[A_max][8*NT][I]  weighted activations per (segment, token)
    float *part13;                // f32[kMaxGrid][2][16][64] W13 partials of split pieces
    float *part2;                 // f32[kMaxGrid][2][16][32] W2 partials of split tiles
    int32_t *cnt13;               // arrival counters per (segment, slab), zero between calls
    int32_t *cnt2;                // arrival counters per output tile, zero between calls
    int32_t *sync;                // [0] finished (segment, slab) pieces, [1] CTAs done
    int32_t *status;
    int32_t M, top_k, num_experts, inter;
    uint64_t timeout_ns;
    int32_t debug_flags;          // bit 0: piece 0 is never announced (exercises the timeout)
};

constexpr int kMaxGrid = 256;            // upper bound on the fused kernel's grid (SM count)
constexpr int kFusedMaxTokens = 16;
constexpr int kFusedMinSms = 80;         // a W2 share must span at most two output tiles

// ------------------------------------------------------------------ kernels
__global__ void route_kernel(const int32_t *topk_ids, int32_t S, int32_t num_experts,
                             int32_t *active_ids, int32_t *offsets, int32_t *sorted_slots,
                             int32_t *num_active, int32_t *status);

__global__ void prepare_compact_kernel(const uint8_t *meta4, uint8_t *meta3, int64_t n_records,
                                       int32_t vectorised);

// Host launchers of the templated GEMM kernels (defined next to them).
awq_status launch_w13(int meta_bytes, dim3 grid, cudaStream_t stream, const CUtensorMap &tq,
                      const CUtensorMap &tm, const StageArgs &args);
awq_status launch_w2(int meta_bytes, dim3 grid, cudaStream_t stream, const CUtensorMap &tq,
                     const CUtensorMap &tm, const StageArgs &args);
awq_status launch_fused(int meta_bytes, int sms, cudaStream_t stream, const CUtensorMap &t13q,
                        const CUtensorMap &t13m, const CUtensorMap &t2q, const CUtensorMap &t2m,
                        const FusedArgs &args);

}  // namespace awq
