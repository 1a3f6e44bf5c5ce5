// Load-time preparation of an expert bank: the canonical row-major layout
// (q [E][K/8][N], records [E][K/32][N]) is permuted, 16 bytes at a time, into
// the layout the kernels stream. Every work unit of the kernels then reads one
// contiguous block, which keeps DRAM rows fully used (a 32-column slab of the
// canonical layout touches 128 bytes of every 1280-byte row).
//
// The pages keep prepared, interleaved weight banks for the same reason
// (Leonccaa/1Cat-vLLM #12 "Add opt-in native-g32 AWQ QPN M1 dispatch", Purpose
// and stack: prepared g32 batched banks with W13 interleaving). The
// permutation moves whole packed words and whole metadata records, so the
// prepared bank decodes to exactly the same weights.
//
// Prepared layout (PJ = I/8 pieces per expert, KP = I/160):
//   W13 q     piece (e, j), 20 KB: word (group 0..79, t 0..3, g 0..7, half)
//             is packed row 4*group + t, column half*I + 8j + g
//   W13 meta  piece (e, j): record (group, g, half) of column half*I + 8j + g
//   W2 q      line (e, kp, tile 0..79, r 0..19): the 32 words of packed
//             row 20*kp + r, columns 32*tile .. +32
//   W2 meta   row  (e, kp, tile, group 0..4): the 32 records of group
//             5*kp + group, columns 32*tile .. +32
// The W13 pieces interleave gate and up columns word by word, so they are
// gathered one word / one record at a time; the W2 banks move in 16-byte
// chunks.
#include <algorithm>

#include "awq_launch.cuh"
#include "awq_moe_kernels.cuh"
#include "awq_ptx.cuh"

namespace awq {

namespace {

// W13 banks, one element (a 4-byte word for kind 0, an mb-byte record for
// kind 1) per thread iteration.
__global__ void prepare_w13_kernel(const uint8_t *src, uint8_t *dst, int64_t n_elems, int kind,
                                   int I, int mb)
{
    grid_dependency_wait();
    const int PJ = I / kPieceCols;
    const int64_t N13 = 2 * I;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n_elems;
         idx += stride) {
        if (kind == 0) {
            const int64_t piece = idx / (kGroups13 * 64);
            const int w = static_cast<int>(idx - piece * (kGroups13 * 64));
            const int grp = w >> 6, t = (w >> 4) & 3, g = (w >> 1) & 7, half = w & 1;
            const int64_t e = piece / PJ, j = piece - e * PJ;
            const int64_t word = (e * (kHidden / 8) + 4 * grp + t) * N13 + half * I + 8 * j + g;
            reinterpret_cast<uint32_t *>(dst)[idx] = __ldg(reinterpret_cast<const uint32_t *>(src) + word);
        } else {
            const int64_t piece = idx / (kGroups13 * 16);
            const int r = static_cast<int>(idx - piece * (kGroups13 * 16));
            const int grp = r >> 4, g = (r >> 1) & 7, half = r & 1;
            const int64_t e = piece / PJ, j = piece - e * PJ;
            const int64_t rec = (e * kGroups13 + grp) * N13 + half * I + 8 * j + g;
            for (int c = 0; c < mb; ++c) dst[idx * mb + c] = __ldg(src + rec * mb + c);
        }
    }
}

// W2 banks, one 16-byte chunk per thread iteration (kind 2: q, 3: meta).
__global__ void prepare_w2_kernel(const uint8_t *src, uint8_t *dst, int64_t n_chunks, int kind, int I,
                                  int mb)
{
    grid_dependency_wait();
    const int KP = I / 160;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n_chunks;
         idx += stride) {
        int64_t off;   // canonical byte offset of this 16-byte chunk
        if (kind == 2) {                                     // W2 q
            const int64_t L = idx >> 3;
            const int c16 = static_cast<int>(idx & 7);
            const int64_t r = L % 20, t1 = L / 20;
            const int64_t c = t1 % kColTiles, t2 = t1 / kColTiles;
            const int64_t kp = t2 % KP, e = t2 / KP;
            off = 4 * ((e * (I / 8) + kp * 20 + r) * kHidden + 32 * c + 4 * c16);
        } else {                                             // W2 meta
            const int per = 2 * mb;                          // chunks per 32-record row
            const int64_t R = idx / per;
            const int c16 = static_cast<int>(idx % per);
            const int64_t g5 = R % 5, t1 = R / 5;
            const int64_t c = t1 % kColTiles, t2 = t1 / kColTiles;
            const int64_t kp = t2 % KP, e = t2 / KP;
            off = ((e * (I / kGroup) + kp * 5 + g5) * kHidden + 32 * c) * mb + 16 * c16;
        }
        *reinterpret_cast<uint4 *>(dst + 16 * idx) = ld_nc_v4(src + off);
    }
}

// NVFP4 block scales (canonical u8[E][K/16][N], one E4M3 code per 16 K of a
// column) -> prepared 2-byte records per (group of 32, column): the codes of
// blocks 2 group and 2 group + 1, in the int4 record orders (which 0: W13
// pieces, record (group, g, half); which 1: W2 rows (e, kp, tile, group) of
// 32 records). One prepared record per thread iteration.
__global__ void prepare_nvfp4_scales_kernel(const uint8_t *src, uint8_t *dst, int64_t n_records, int which, int I)
{
    grid_dependency_wait();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n_records;
         idx += stride) {
        int64_t row0, N;   // canonical row of block 2 * group, columns per row
        int64_t col;
        if (which == 0) {
            const int PJ = I / kPieceCols;
            const int64_t piece = idx / (kGroups13 * 16);
            const int r = static_cast<int>(idx - piece * (kGroups13 * 16));
            const int grp = r >> 4, g = (r >> 1) & 7, half = r & 1;
            const int64_t e = piece / PJ, j = piece - e * PJ;
            N = 2 * I;
            col = half * I + 8 * j + g;
            row0 = e * (kHidden / 16) + 2 * grp;
        } else {
            const int KP = I / 160;
            const int c = static_cast<int>(idx & 31);
            const int64_t R = idx >> 5;
            const int64_t g5 = R % 5, t1 = R / 5;
            const int64_t tile = t1 % kColTiles, t2 = t1 / kColTiles;
            const int64_t kp = t2 % KP, e = t2 / KP;
            N = kHidden;
            col = 32 * tile + c;
            row0 = e * (I / 16) + 2 * (5 * kp + g5);
        }
        dst[2 * idx] = __ldg(src + row0 * N + col);
        dst[2 * idx + 1] = __ldg(src + (row0 + 1) * N + col);
    }
}

}  // namespace

awq_status launch_prepare(const awq_moe_shape &s, const awq_moe_weights &canon,
                          const awq_moe_weights &prep, cudaStream_t st)
{
    const int E = s.num_experts, I = s.inter, mb = s.meta_bytes;
    if (s.group == 16) {
        // NVFP4: words as int4 banks, block scales regrouped into 2-byte records
        const int64_t w13_q = static_cast<int64_t>(E) * (kHidden / 8) * 2 * I;       // words
        const int64_t w2_q16 = static_cast<int64_t>(E) * (I / 8) * kHidden * 4 / 16;  // 16-byte chunks
        const int64_t r13 = static_cast<int64_t>(E) * (kHidden / 32) * 2 * I;         // prepared records
        const int64_t r2 = static_cast<int64_t>(E) * (I / 32) * kHidden;
        auto blocks = [](int64_t n) { return static_cast<int>(std::min<int64_t>((n + 255) / 256, 152 * 32)); };
        awq_status r = launch(prepare_w13_kernel, dim3(blocks(w13_q)), dim3(256), 0, 1, st,
                              reinterpret_cast<const uint8_t *>(canon.w13_q),
                              const_cast<uint8_t *>(reinterpret_cast<const uint8_t *>(prep.w13_q)), w13_q, 0, I, 4);
        if (!r)
            r = launch(prepare_w2_kernel, dim3(blocks(w2_q16)), dim3(256), 0, 1, st,
                       reinterpret_cast<const uint8_t *>(canon.w2_q),
                       const_cast<uint8_t *>(reinterpret_cast<const uint8_t *>(prep.w2_q)), w2_q16, 2, I, 4);
        if (!r)
            r = launch(prepare_nvfp4_scales_kernel, dim3(blocks(r13)), dim3(256), 0, 1, st, canon.w13_meta,
                       const_cast<uint8_t *>(prep.w13_meta), r13, 0, I);
        if (!r)
            r = launch(prepare_nvfp4_scales_kernel, dim3(blocks(r2)), dim3(256), 0, 1, st, canon.w2_meta,
                       const_cast<uint8_t *>(prep.w2_meta), r2, 1, I);
        return r;
    }
    const int64_t w13_q = static_cast<int64_t>(E) * (kHidden / 8) * 2 * I * 4;
    const int64_t w13_m = static_cast<int64_t>(E) * (kHidden / kGroup) * 2 * I * mb;
    const int64_t w2_q = static_cast<int64_t>(E) * (I / 8) * kHidden * 4;
    const int64_t w2_m = static_cast<int64_t>(E) * (I / kGroup) * kHidden * mb;
    const void *srcs[4] = {canon.w13_q, canon.w13_meta, canon.w2_q, canon.w2_meta};
    const void *dsts[4] = {prep.w13_q, prep.w13_meta, prep.w2_q, prep.w2_meta};
    const int64_t elems[4] = {w13_q / 4, w13_m / mb, w2_q / 16, w2_m / 16};
    for (int kind = 0; kind < 4; ++kind) {
        const int blocks = static_cast<int>(std::min<int64_t>((elems[kind] + 255) / 256, 152 * 32));
        const uint8_t *src = static_cast<const uint8_t *>(srcs[kind]);
        uint8_t *dst = const_cast<uint8_t *>(static_cast<const uint8_t *>(dsts[kind]));
        awq_status r = kind < 2 ? launch(prepare_w13_kernel, dim3(blocks), dim3(256), 0, 1, st, src, dst,
                                         elems[kind], kind, I, mb)
                                : launch(prepare_w2_kernel, dim3(blocks), dim3(256), 0, 1, st, src, dst,
                                         elems[kind], kind, I, mb);
        if (r) return r;
    }
    return AWQ_OK;
}

}  // namespace awq
