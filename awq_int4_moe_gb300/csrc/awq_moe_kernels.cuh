// Kernel-side declarations shared by the translation units of the CUDA
// library: launch constants, argument block and kernel prototypes.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/awq_moe.h"
#include "awq_ptx.cuh"

namespace awq {

// ----------------------------------------------------------- fixed geometry
constexpr int kHidden = 2560;           // W13 K, W2 N
constexpr int kGroup = 32;              // quantisation group along K
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 16;
constexpr int kMaxSlots = AWQ_MAX_TOKENS * kMaxTopK;
// the warp-level MMA W2 kernel of the three-launch path keeps every token's
// output tile in shared memory: it takes at most this many tokens
constexpr int kStagedMaxTokens = AWQ_W2_STAGE_MAX_TOKENS;
constexpr int kStagedMaxSlots = kStagedMaxTokens * kMaxTopK;

// Prepared-layout geometry (see awq_moe_prepare.cu).
// W13 piece: 8 gate columns and the 8 matching up columns over the whole K
// (80 groups), i.e. one 16-row MMA tile: q as 80 x [t 4][g 8][gate, up]
// words (20 KB), metadata as 80 x [g 8][gate, up] records.
constexpr int kGroups13 = kHidden / kGroup;                        // 80
constexpr int kPieceCols = 8;
constexpr int kPieceQ = kGroups13 * 4 * kPieceCols * 2 * 4;        // 20480
__host__ __device__ constexpr int piece_meta_bytes(int mb) { return kGroups13 * kPieceCols * 2 * mb; }
// W2 tile: 20 packed rows (160 k, 5 groups) of 32 columns, 20 contiguous
// 128-byte lines; its metadata is 5 rows of 32 records.
constexpr int kW2TileKK = 20;
constexpr int kColTiles = kHidden / 32;                            // 80

// W13 stage call: one CTA per (segment, piece); warp w takes groups
// 10w .. 10w+9 of K for 8 segment rows at a time.
constexpr int kW13Threads = 256;                                   // 8 warps
constexpr int kW13GroupsPerWarp = kGroups13 / (kW13Threads / 32);  // 10
constexpr int kW13RedBytes = (kW13Threads / 32) * 32 * 16;         // warps x lanes x float4

__host__ __device__ constexpr int w13_smem_bytes(int mb)
{
    return 128 /*align slack*/ + kPieceQ + (piece_meta_bytes(mb) + 127) / 128 * 128 + kW13RedBytes + 64;
}

// W2 stage call: a cluster of 8 CTAs shares one 32-column output tile;
// segment a goes to CTA a % 8, and within it to warp (a / 8) % 4, each warp
// with its own 2-stage TMA ring. A stage holds the I/160 K parts of the tile,
// each 20 lines in its own 1 KB-aligned 3 KB slot (the swizzle atom is 1 KB).
constexpr int kW2Cluster = 8;
constexpr int kW2Threads = 128;
constexpr int kW2Warps = kW2Threads / 32;
constexpr int kW2Stages = 2;
constexpr int kW2ColTile = 32;
constexpr int kW2PartSlot = 3072;
// W2 work items: up to 16 rows (two token blocks) of one segment.
constexpr int kW2ItemRows = 16;
constexpr int kW2MaxItems = kMaxExperts + kStagedMaxSlots / kW2ItemRows;

__host__ __device__ constexpr int w2_meta_slot(int mb) { return ((5 * 32 * mb) + 127) / 128 * 128; }
__host__ __device__ constexpr int w2_q_stage_bytes(int inter) { return (inter / 160) * kW2PartSlot; }
__host__ __device__ constexpr int w2_meta_stage_bytes(int inter, int mb)
{
    return (inter / 160) * w2_meta_slot(mb);
}
// ring stages, per-warp accumulators, the work-item list, each sorted row's
// token and router weight (S = M * top_k rows), barriers
__host__ __device__ constexpr int w2_smem_bytes(int inter, int mb, int M, int top_k)
{
    return 1024 + kW2Warps * kW2Stages * (w2_q_stage_bytes(inter) + w2_meta_stage_bytes(inter, mb)) +
           kW2Warps * M * kW2ColTile * 4 + kW2MaxItems * 4 + 2 * M * top_k * 4 + 128;
}

struct StageArgs {
    const uint32_t *w13_q;         // prepared W13 bank (W13)
    const uint8_t *w13_meta;
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
    // tensor-core W2 (prefill-sized batches): prepared W2 bank and the
    // weighted per-slot products y f32[S][H] (slot order)
    const uint32_t *w2_q;
    const uint8_t *w2_meta;
    float *y;
    // prefill path: W13 also writes the rounding residue h - fp16(h) as a
    // second fp16 plane h_lo[S][I] (h_out + S * I), which W2 reads as well
    uint16_t *h_lo;
    // NVFP4 banks: per-expert global scales f32[E][2] (W13, W2); null for int4
    const float *global_scale;
    // prefill path tracing (null in normal use): launch k (0 W13, 1 W2,
    // 2 combine) takes the earliest CTA start past its dependency wait into
    // trace[2k] (atomic min) and the latest CTA end into trace[2k+1] (max)
    uint64_t *trace;
};

__device__ __forceinline__ void trace_start(uint64_t *trace, int k)
{
    if (trace) atomicMin(reinterpret_cast<unsigned long long *>(trace + 2 * k), global_timer_ns());
}
__device__ __forceinline__ void trace_end(uint64_t *trace, int k)
{
    if (trace) atomicMax(reinterpret_cast<unsigned long long *>(trace + 2 * k + 1), global_timer_ns());
}

// Arguments of the fused (single-launch) decode layer kernel. Workspace
// buffers are carved by the host from the caller's workspace.
struct FusedArgs {
    const uint16_t *x;            // fp16[M][H]
    const int32_t *topk_ids;      // i32[M][k]
    const float *topk_weights;    // f32[M][k]
    uint16_t *out;                // fp16[M][H]
    const uint32_t *w13_q;        // prepared W13 bank
    const uint8_t *w13_meta;
    uint16_t *hw;                 // fp16[A_max][8*NT][I]  weighted activations per (segment, token)
    float *part2;                 // f32[kMaxGrid][2][kPartStride] W2 partials of split column groups
    int32_t *cnt2;                // [2][10] published W2 partials per 256-column group, per sense
    int32_t *sync;                // [2] finished W13 pieces, per sense
    int32_t *sense;               // [kMaxGrid] per-CTA call parity (selects the counter set)
    int32_t *status;
    int32_t M, top_k, num_experts, inter;
    uint64_t timeout_ns;
    int32_t debug_flags;          // bit 0: piece 0 is never announced (exercises the timeout)
    // Routing from logits instead of topk_ids / topk_weights when non-null:
    // f32[M][E]; every CTA routes in its prologue, CTA 0 writes the choice.
    const float *logits;
    int32_t *topk_ids_out;        // i32[M][k]
    float *topk_weights_out;      // f32[M][k]
    // NVFP4 banks only: f32[E][2] per-expert global scales (W13, W2) and the
    // fp16 residue plane of hw (same shape), hw + hw_lo being HW to ~22 bits.
    const float *global_scale;
    uint16_t *hw_lo;
};

// Arguments of the sliced decode layer kernel (W2 sliced along K with W13,
// up to kSlicedMaxTokens tokens); workspace buffers carved by the host.
constexpr int kSlicedMaxTokens = 8;
struct SlicedArgs {
    const uint16_t *x;            // fp16[M][H]
    const int32_t *topk_ids;      // i32[M][k]
    const float *topk_weights;    // f32[M][k]
    uint16_t *out;                // fp16[M][H]
    const uint32_t *w13_q;        // prepared W13 bank
    const uint8_t *w13_meta;
    float *part;                  // f32[grid][M][H] partial outputs per CTA; in tile mode
                                  // fp16 HW[A][8][I] (weighted activations)
    uint64_t *gbar;               // grid barrier: arrivals over all calls on the workspace (G per call)
    int32_t *status;
    int32_t M, top_k, num_experts, inter;
    uint64_t timeout_ns;
    int32_t debug_flags;          // bit 0: CTA 0 reaches the grid barrier only after the others' wait ran out
    uint64_t *trace;              // [grid][AWQ_TRACE_POINTS] phase timestamps, or null
    const float *logits;          // as FusedArgs
    int32_t *topk_ids_out;
    float *topk_weights_out;
};

constexpr int kMaxGrid = 256;            // upper bound on the persistent kernels' grid (SM count)
constexpr int kFusedMaxTokens = 16;
constexpr int kFusedMinSms = 80;         // a W2 share must span at most two column groups
constexpr int kFusedW2Tiles = 8;         // 32-column tiles per fused W2 unit (one per consumer warp)
// One W2 partial block: 16 tokens x 256 columns of fp32, padded by 192 bytes so
// that the same element of consecutive blocks falls in different L2 slices
// (the finishing CTA reads it from every part at once).
constexpr int kPartStride = 16 * 256 + 48;

// ------------------------------------------------------------------ kernels
constexpr int kRouteThreads = 256;
// dynamic shared memory of route_kernel for S slots and E experts
__host__ __device__ constexpr int route_smem_bytes(int S, int E)
{
    return (S + (kRouteThreads / 32 + 2) * (E + 1)) * 4;
}
__global__ void route_kernel(const int32_t *topk_ids, int32_t S, int32_t num_experts,
                             int32_t *active_ids, int32_t *offsets, int32_t *sorted_slots,
                             int32_t *num_active, int32_t *status);

// Router from logits (E = 512): one warp per token, 8 tokens per block.
constexpr int kRouterExperts = 512;
constexpr int kRouterWarps = 8;
__global__ void router_topk_kernel(const float *logits, int32_t M, int32_t top_k, int32_t *topk_ids,
                                   float *topk_weights);
__global__ void prepare_compact_kernel(const uint8_t *meta4, uint8_t *meta3, int64_t n_records,
                                       int32_t vectorised);

// Host launchers of the templated GEMM kernels (defined next to them).
awq_status launch_w13(int meta_bytes, dim3 grid, cudaStream_t stream, const StageArgs &a);
awq_status launch_w2(int meta_bytes, dim3 grid, cudaStream_t stream, const CUtensorMap &tq,
                     const CUtensorMap &tm, const StageArgs &args);
awq_status launch_fused(int meta_bytes, int sms, cudaStream_t stream, const CUtensorMap &t2q,
                        const CUtensorMap &t2m, const CUtensorMap &t2q1, const CUtensorMap &t2m1,
                        const FusedArgs &args);
awq_status launch_sliced(int meta_bytes, int sms, cudaStream_t stream, const CUtensorMap &tq,
                         const CUtensorMap &tm, const CUtensorMap &t1q, const CUtensorMap &t1m,
                         const SlicedArgs &args);
int sliced_smem_bytes(int inter);
// Tensor-core (tcgen05) grouped GEMMs for prefill-sized batches: W13 + SwiGLU
// (x rows gathered by the kernel), W2 into per-slot products y, and the
// per-token combine of y into out. th: tensor maps of the two h planes
// f16[2 S][I] (fp16(h) rows, then the residue rows) with boxes of
// 64 x {16, 32, 64, 128} rows, 128-byte swizzle.
constexpr int kTcRows13 = 32;                        // W13 rows (tokens) per work item
constexpr int kTcKbPerStage13 = 2;                   // W13 K blocks of 64 per ring stage (one TMA box)
__host__ __device__ constexpr int tc_rows2(int inter) { return inter == 160 ? 64 : 16; }   // W2
// Persistent launches, one CTA per multiprocessor (`sms`).
// tq13 / tm13: 3D views of the prepared W13 bank, [piece][K block of 64][512 B
// of words] and [piece][K block][32 mb bytes of records], boxes of 8 pieces.
awq_status launch_w13_tc(int meta_bytes, int S, int sms, cudaStream_t stream, const CUtensorMap &tq13,
                         const CUtensorMap &tm13, const StageArgs &a);
awq_status launch_w2_tc(int meta_bytes, int S, int sms, cudaStream_t stream, const CUtensorMap (&th)[4],
                        const StageArgs &a);
awq_status launch_combine(int M, int top_k, const float *y, uint16_t *out, uint64_t *trace, cudaStream_t stream);
awq_status launch_prepare(const awq_moe_shape &s, const awq_moe_weights &canon,
                          const awq_moe_weights &prep, cudaStream_t stream);

}  // namespace awq
