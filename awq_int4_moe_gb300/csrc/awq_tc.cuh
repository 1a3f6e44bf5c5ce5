// 5th-generation tensor-core building blocks (tcgen05) shared by the
// prefill-sized grouped GEMM kernels: shared-memory matrix descriptors for
// the K-major 128-byte-swizzled operand layout, the f16 MMA with an fp32
// accumulator in tensor memory, commit-to-mbarrier, TMEM allocation and
// loads, cp.async row gathers, and the (segment, row chunk) work-item search.
#pragma once

#include <cstdint>

#include "awq_moe_kernels.cuh"
#include "awq_ptx.cuh"

namespace awq {

// Offset of 16-byte chunk c of row r in a K-major tile of 128-byte rows with
// the 128-byte swizzle: 8-row atoms of 1 KB, chunk index XOR (row mod 8).
// TMA writes this layout for a box of 64 fp16 x rows with
// CU_TENSOR_MAP_SWIZZLE_128B into a 1024-byte-aligned destination.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int r, int c)
{
    return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// Shared memory matrix descriptor: start address >> 4 in bits [0,14),
// leading byte offset >> 4 in [16,30) (16 B: unused by a swizzled K-major
// operand), stride byte offset >> 4 in [32,46) (1024 B between 8-row atoms),
// the fixed 0b001 at bit 46 and the 128-byte swizzle (2) in [61,64). A K16
// step inside the 128-byte row advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t addr)
{
    uint64_t d = static_cast<uint64_t>((addr & 0x3FFFF) >> 4);
    d |= static_cast<uint64_t>(16 >> 4) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// Instruction descriptor of kind::f16 with f16 A and B (both K-major) and
// an fp32 accumulator: D format 1 in bits [4,6), N >> 3 in [17,23), M >> 4
// in [24,29).
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N)
{
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[adesc] * B[bdesc]^T, issued by one thread.
__device__ __forceinline__ void tc_mma_f16(uint32_t tmem, uint64_t ad, uint64_t bd, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
        "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[a_tmem] * B[bdesc]^T with A in tensor memory: row m in
// lane m, two fp16 of consecutive k per 32-bit column (even k in the low
// half), a K16 step = 8 columns.
__device__ __forceinline__ void tc_mma_f16_tmem_a(uint32_t tmem, uint32_t a_tmem, uint64_t bd, uint32_t idesc,
                                                  uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem),
        "r"(a_tmem), "l"(bd), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The warp's 32 lanes each store 16 consecutive 32-bit columns of their own
// TMEM lane (lane base + lane index); tc_wait_st() waits for the stores.
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 3D TMA tile load (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *m, uint64_t *bar, int c0, int c1, int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// One arrival on `bar` once every tcgen05 operation this thread issued
// before has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// Warp-collective TMEM allocation of `cols` columns (a power of two >= 32);
// the base address goes to *slot.
__device__ __forceinline__ void tc_alloc(uint32_t *slot, uint32_t cols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_dealloc(uint32_t tmem, uint32_t cols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(cols) : "memory");
}

// 16 consecutive fp32 columns of the warp's 32 TMEM lanes (lane i of the warp
// gets lane base + i); waits for the load.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16-byte global -> shared copy (L2 only), tracked by commit groups.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// One arrival on `bar` once every cp.async this thread issued before has
// completed; the barrier's expected count includes it (no pending-count
// increment). The waiting side still issues fence.proxy.async before the
// tensor core (async proxy) reads what the copies wrote.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) { mbar_arrive_count(bar, 1); }

// Barrier `id` over `n` threads that also ANDs a predicate across them: every
// participant gets true only when all passed true.
__device__ __forceinline__ bool named_barrier_and(int id, int n, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Work items of the grouped GEMMs: each active segment's rows in chunks of C,
// numbered segment by segment. Every thread of the NT-thread block calls
// this; item -> (segment, chunk) lands in s_res[0..1] (segment -1 when the
// item is past the last one). Scratch s_warp[NT / 32]. Ends with a
// __syncthreads().
template <int NT>
__device__ void find_work_item(int item, int A, const int32_t *offsets, int C, int32_t *s_warp, int32_t *s_res)
{
    constexpr int kPer = (kMaxExperts + NT - 1) / NT;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (A + NT - 1) / NT;
    const int a0 = tid * per;
    int ov[kPer + 1];
#pragma unroll
    for (int i = 0; i <= kPer; ++i) ov[i] = (i <= per && a0 + i <= A) ? offsets[a0 + i] : 0;
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        if (i < per && a0 + i < A) cnt += (ov[i + 1] - ov[i] + C - 1) / C;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    if (tid == 0) s_res[0] = -1;
    __syncthreads();
    int pos = incl - cnt;
    for (int w = 0; w < warp; ++w) pos += s_warp[w];
    if (item >= pos && item < pos + cnt) {
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            if (i < per && a0 + i < A) {
                const int n = (ov[i + 1] - ov[i] + C - 1) / C;
                if (item < pos + n) {
                    s_res[0] = a0 + i;
                    s_res[1] = item - pos;
                    break;
                }
                pos += n;
            }
        }
    }
    __syncthreads();
}

// Units of a persistent grouped GEMM: work items (each active segment's rows
// in chunks of C, numbered segment by segment) x `tiles` column tiles, unit
// u = item * tiles + tile, dealt round-robin: CTA c of G takes u = c, c + G,
// ... Every thread of the NT-thread block calls this; the CTA's k-th unit
// lands in table[k] as (segment, chunk, tile, 0). Returns the CTA's unit
// count (at most max_units are written; the caller sizes the grid so that
// none is dropped). Scratch s_warp[NT / 32 + 1]. Ends with __syncthreads().
template <int NT>
__device__ int build_unit_table(int A, const int32_t *offsets, int C, int tiles, int G, int c, int4 *table,
                                int max_units, int32_t *s_warp)
{
    constexpr int kPer = (kMaxExperts + NT - 1) / NT;
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (A + NT - 1) / NT;
    const int a0 = tid * per;
    int ov[kPer + 1];
#pragma unroll
    for (int i = 0; i <= kPer; ++i) ov[i] = (i <= per && a0 + i <= A) ? offsets[a0 + i] : 0;
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        if (i < per && a0 + i < A) cnt += (ov[i + 1] - ov[i] + C - 1) / C;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int item = incl - cnt, total = 0;
    for (int w = 0; w < NW; ++w) {
        if (w < warp) item += s_warp[w];
        total += s_warp[w];
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        if (i < per && a0 + i < A) {
            const int n = (ov[i + 1] - ov[i] + C - 1) / C;
            for (int z = 0; z < n; ++z, ++item)
                for (int t = 0; t < tiles; ++t) {
                    const int u = item * tiles + t;
                    if (u % G == c && u / G < max_units) table[u / G] = make_int4(a0 + i, z, t, 0);
                }
        }
    }
    const int U = total * tiles;
    __syncthreads();
    return U > c ? min(max_units, (U - c + G - 1) / G) : 0;
}

// Upper bound on the number of work items: sum over segments of
// ceil(rows / C) <= A + S / C, A <= min(S, E).
__host__ __device__ inline int max_work_items(int S, int E, int C) { return (S < E ? S : E) + S / C; }

}  // namespace awq
