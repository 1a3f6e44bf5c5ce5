// Measurement helper: the latency floor of a decode-sized layer call.
//
// One cooperative persistent launch (one CTA per multiprocessor) that walks
// the dependency chain of the persistent layer kernels with none of their
// arithmetic: wait for the previous launch; load the top-k ids and build the
// distinct active experts in shared memory; read every byte of those
// experts' prepared banks once (the algorithmic bytes of the call: W13 and
// W2 words and records), as bulk copies of up to 16 KB dealt round-robin
// over the CTAs into a discarded shared-memory ring; one grid barrier (the
// hand-off from the weight phase to the output phase); write the output rows
// (zeros). Its time per call, in the same graph of layer calls as the real
// kernel, is what a kernel with this chain cannot beat: the real kernels'
// time above it is arithmetic, hand-offs and imbalance.
//
// The grid barrier is the same monotonic 64-bit arrival counter the sliced
// layer kernel keeps in the workspace (G arrivals per call; the epoch is read
// after the wait for the previous launch). Every wait is bounded.
#include <cstdint>

#include "awq_dequant.cuh"
#include "awq_launch.cuh"
#include "awq_moe_kernels.cuh"
#include "awq_ptx.cuh"

namespace awq {

namespace {

constexpr int kFloorThreads = 256;
constexpr int kFloorSlots = 8;
constexpr int kFloorChunk = 16384;
constexpr int kFloorMaxSlots = kFusedMaxTokens * kMaxTopK;   // 256 slots

struct FloorArgs {
    const int32_t *topk_ids;
    const uint8_t *bank[4];        // prepared W13 q, W13 meta, W2 q, W2 meta
    int64_t region[4];             // bytes per expert of each bank
    int32_t chunks_per_expert;     // sum over banks of ceil(region / kFloorChunk)
    uint16_t *out;
    uint64_t *gbar;
    int32_t *status;
    int32_t S, num_experts, M;
    uint64_t timeout_ns;
};

__device__ __forceinline__ void red_add_release(uint64_t *p, uint64_t v)
{
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

}  // namespace

__global__ void __launch_bounds__(kFloorThreads, 1) floor_kernel(FloorArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = align1024(smem_raw);
    __shared__ uint64_t bars[kFloorSlots];
    __shared__ uint32_t bitmap[kMaxExperts / 32];
    __shared__ int32_t act[kFloorMaxSlots];
    __shared__ int32_t s_count;
    __shared__ const uint8_t *s_bank[4];
    __shared__ int64_t s_region[4];
    const int tid = threadIdx.x, G = gridDim.x, b = blockIdx.x;

    if (tid < kMaxExperts / 32) bitmap[tid] = 0;
    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s_bank[i] = args.bank[i];
            s_region[i] = args.region[i];
        }
    }
    if (tid == 0) {
        for (int s = 0; s < kFloorSlots; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    grid_dependency_wait();
    grid_launch_dependents();
    uint64_t epoch = 0;
    if (tid == 0) epoch = ld_relaxed_u64(args.gbar) / static_cast<uint64_t>(G);
    __syncthreads();
    // distinct active experts, ascending
    for (int s = tid; s < args.S; s += kFloorThreads) {
        const int e = args.topk_ids[s];
        if (e >= 0 && e < args.num_experts) atomicOr(&bitmap[e >> 5], 1u << (e & 31));
        else set_status(args.status, AWQ_ERR_BAD_EXPERT_ID);
    }
    __syncthreads();
    if (tid < 32) {
        const int c = __popc(bitmap[tid]);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (tid >= o) incl += y;
        }
        if (tid == 31) s_count = incl;
        uint32_t bits = bitmap[tid];
        int pos = incl - c;
        while (bits) {
            act[pos++] = 32 * tid + __ffs(bits) - 1;
            bits &= bits - 1;
        }
    }
    __syncthreads();
    const int A = s_count;

    // this CTA's chunks of the active experts' banks (chunk j -> CTA j mod G)
    bool fine = true;
    if (tid == 0) {
        const int total = A * args.chunks_per_expert;
        int issued = 0;
        for (int j = b; j < total; j += G, ++issued) {
            const int a = j / args.chunks_per_expert;
            int c = j - a * args.chunks_per_expert;
            int bank = 0;
            int64_t n = (s_region[0] + kFloorChunk - 1) / kFloorChunk;
            while (c >= n && bank < 3) {
                c -= static_cast<int>(n);
                ++bank;
                n = (s_region[bank] + kFloorChunk - 1) / kFloorChunk;
            }
            const int64_t off = static_cast<int64_t>(c) * kFloorChunk;
            const int64_t len = s_region[bank] - off < kFloorChunk ? s_region[bank] - off : kFloorChunk;
            const int s = issued % kFloorSlots;
            if (issued >= kFloorSlots && !mbar_wait_bounded(&bars[s], ((issued / kFloorSlots) - 1) & 1, args.timeout_ns)) {
                fine = false;
                break;
            }
            mbar_arrive_expect_tx(&bars[s], static_cast<uint32_t>(len));
            bulk_load(ring + s * kFloorChunk, s_bank[bank] + static_cast<int64_t>(act[a]) * s_region[bank] + off,
                      static_cast<uint32_t>(len), &bars[s]);
        }
        // every copy has landed before the barrier (and before the CTA exits)
        for (int j = issued - kFloorSlots < 0 ? 0 : issued - kFloorSlots; j < issued; ++j)
            if (!mbar_wait_bounded(&bars[j % kFloorSlots], (j / kFloorSlots) & 1, args.timeout_ns)) fine = false;
        // grid barrier: the weight phase of every CTA is done
        red_add_release(args.gbar, 1ull);
        const uint64_t target = (epoch + 1) * static_cast<uint64_t>(G);
        const uint64_t t0 = global_timer_ns();
        while (ld_acquire_u64(args.gbar) < target) {
            if (global_timer_ns() - t0 > args.timeout_ns) {
                fine = false;
                break;
            }
            sleep_ns(20);
        }
        if (!fine) set_status(args.status, AWQ_ERR_DEVICE_TIMEOUT);
    }
    __syncthreads();
    // output phase: the M x H fp16 rows, 16 bytes per store
    const int64_t n16 = static_cast<int64_t>(args.M) * kHidden / 8;
    for (int64_t i = static_cast<int64_t>(b) * kFloorThreads + tid; i < n16; i += static_cast<int64_t>(G) * kFloorThreads)
        reinterpret_cast<uint4 *>(args.out)[i] = make_uint4(0, 0, 0, 0);
}

awq_status launch_floor(const int32_t *topk_ids, int32_t M, const awq_moe_shape &s, const awq_moe_weights &w,
                        uint16_t *out, uint64_t *gbar, int32_t *status, uint64_t timeout_ns, int sms, cudaStream_t st)
{
    FloorArgs a = {};
    a.topk_ids = topk_ids;
    a.bank[0] = reinterpret_cast<const uint8_t *>(w.w13_q);
    a.bank[1] = w.w13_meta;
    a.bank[2] = reinterpret_cast<const uint8_t *>(w.w2_q);
    a.bank[3] = w.w2_meta;
    const int64_t H = kHidden, I = s.inter, G = s.group, mb = s.meta_bytes;
    a.region[0] = (H / 8) * 2 * I * 4;
    a.region[1] = (H / G) * 2 * I * mb;
    a.region[2] = (I / 8) * H * 4;
    a.region[3] = (I / G) * H * mb;
    a.chunks_per_expert = 0;
    for (int i = 0; i < 4; ++i) a.chunks_per_expert += static_cast<int32_t>((a.region[i] + kFloorChunk - 1) / kFloorChunk);
    a.out = out;
    a.gbar = gbar;
    a.status = status;
    a.S = M * s.top_k;
    a.num_experts = s.num_experts;
    a.M = M;
    a.timeout_ns = timeout_ns;
    const int smem = kFloorSlots * kFloorChunk + 1024;
    awq_status r = set_smem(floor_kernel, smem);
    if (r) return r;
    return launch_ex(floor_kernel, dim3(sms), dim3(kFloorThreads), smem, 1, true, st, a);
}

}  // namespace awq
