// Host side of the C ABI declared in include/awq_moe.h: argument validation
// (fail closed, nothing launched on a host-visible error), TMA tensor-map
// construction and the launches.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include "awq_launch.cuh"
#include "awq_moe_kernels.cuh"

namespace awq {

// measurement helper (awq_moe_floor.cu)
awq_status launch_floor(const int32_t *topk_ids, int32_t M, const awq_moe_shape &s, const awq_moe_weights &w,
                        uint16_t *out, uint64_t *gbar, int32_t *status, uint64_t timeout_ns, int sms, cudaStream_t st);

namespace {

constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;   // 1 s per device wait
// AWQ_PATH_AUTO takes the hybrid path (stage W13, tensor-core W2) for the
// calls the persistent decode kernels do not take, up to kHybridMaxTokens
// tokens: measured faster on GB300 than the three stage launches (M =
// 17..128: 48 vs 53 us at 17, 138 vs 168 us at 128) and than the
// tensor-core W13 of the prefill path, for int4 and NVFP4 banks alike
// (Zipf routing: int4 276 vs 318 us at 512; NVFP4 168 vs 203 us at 256,
// 253 vs 258 us at 512)
constexpr int kHybridMaxTokens = AWQ_MAX_TOKENS;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

awq_status check_shape(const awq_moe_shape *s)
{
    if (!s) return AWQ_ERR_INVALID_ARG;
    if (s->num_experts < 1 || s->num_experts > kMaxExperts) return AWQ_ERR_UNSUPPORTED_SHAPE;
    if (s->top_k < 1 || s->top_k > kMaxTopK) return AWQ_ERR_UNSUPPORTED_SHAPE;
    if (s->hidden != kHidden) return AWQ_ERR_UNSUPPORTED_SHAPE;
    if (s->inter != 160 && s->inter != 640) return AWQ_ERR_UNSUPPORTED_SHAPE;
    // int4: group 32 with 3- or 4-byte records; NVFP4: 16-element blocks with
    // one E4M3 scale byte
    const bool int4 = s->group == kGroup && (s->meta_bytes == 3 || s->meta_bytes == 4);
    const bool nvfp4 = s->group == 16 && s->meta_bytes == 1;
    if (!int4 && !nvfp4) return AWQ_ERR_UNSUPPORTED_SHAPE;
    return AWQ_OK;
}

bool is_nvfp4(const awq_moe_shape &s) { return s.group == 16; }

// Bytes of one prepared metadata record per (group of 32, column): the int4
// record, or NVFP4's two block-scale codes.
int prepared_record_bytes(const awq_moe_shape &s) { return is_nvfp4(s) ? 2 : s.meta_bytes; }

// NVFP4 banks also need their global scales.
awq_status check_global(const awq_moe_shape &s, const awq_moe_weights &w)
{
    if (!is_nvfp4(s)) return AWQ_OK;
    if (!w.global_scale) return AWQ_ERR_INVALID_ARG;
    return aligned(w.global_scale, 4) ? AWQ_OK : AWQ_ERR_MISALIGNED;
}

awq_status check_banks(const awq_moe_weights *w)
{
    if (!w || !w->w13_q || !w->w13_meta || !w->w2_q || !w->w2_meta) return AWQ_ERR_INVALID_ARG;
    if (!aligned(w->w13_q, 16) || !aligned(w->w13_meta, 16) || !aligned(w->w2_q, 16) ||
        !aligned(w->w2_meta, 16))
        return AWQ_ERR_MISALIGNED;
    return AWQ_OK;
}

// Weights of a compute call: valid banks in the prepared layout.
awq_status check_weights(const awq_moe_weights *w)
{
    awq_status r = check_banks(w);
    if (r) return r;
    return w->layout == AWQ_LAYOUT_PREPARED ? AWQ_OK : AWQ_ERR_LAYOUT;
}

// Multiprocessor count of the current device, looked up once per device
// (atomic entries: host threads may call concurrently).
int current_sm_count()
{
    static std::atomic<int> cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cache[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

awq_status check_m(int32_t M)
{
    return (M < 0 || M > AWQ_MAX_TOKENS) ? AWQ_ERR_INVALID_ARG : AWQ_OK;
}

// ------------------------------------------------------------- tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool encode(CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *base,
            const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box,
            CUtensorMapSwizzle swz, CUtensorMapL2promotion l2 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(m, dt, rank, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Prepared W2 banks are viewed as 2D arrays of 128-byte q lines and 32-record
// metadata rows; every unit of work is one box of consecutive lines / rows.
// q boxes are 128-byte swizzled (the consumers undo it); metadata is not.
// (W13 pieces are fetched with plain bulk copies and need no tensor map.)
bool make_line_map(CUtensorMap *m, const void *base, uint64_t lines, uint32_t box_lines)
{
    cuuint64_t dims[2] = {32, lines};
    cuuint64_t str[1] = {128};
    cuuint32_t box[2] = {32, box_lines};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, base, dims, str, box,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_row_map(CUtensorMap *m, const void *base, uint64_t rows, int mb, uint32_t box_rows)
{
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(32 * mb), rows};
    cuuint64_t str[1] = {static_cast<cuuint64_t>(32 * mb)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(32 * mb), box_rows};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, str, box,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
}

// W2: `tiles` consecutive 32-column tiles of one (expert, 160-row K part) per
// box: 20 lines and 5 rows each (1 tile for the three-launch path, 8 for the
// fused kernel).
//
// A map is a pure function of the bank addresses, the shape and the box, so
// the pairs are kept in a small direct-mapped table: a caller that does not
// capture its calls in a graph does not pay the driver's encoding (up to
// four maps per layer call) every time.
struct W2MapEntry {
    const void *q = nullptr, *meta = nullptr;
    int32_t num_experts = 0, inter = 0, meta_bytes = 0, tiles = 0;
    CUtensorMap tq, tm;
};

bool make_w2_maps(const awq_moe_shape &s, const awq_moe_weights &w, int tiles, CUtensorMap *tq,
                  CUtensorMap *tm)
{
    constexpr uint64_t kEntries = 512;
    static W2MapEntry table[kEntries];
    static std::mutex mu;
    uint64_t hsh = reinterpret_cast<uintptr_t>(w.w2_q) ^ (reinterpret_cast<uintptr_t>(w.w2_meta) << 7) ^
                   (static_cast<uint64_t>(tiles) << 3) ^ (static_cast<uint64_t>(s.inter) << 11) ^
                   static_cast<uint64_t>(s.meta_bytes);
    hsh ^= hsh >> 29;
    hsh *= 0xbf58476d1ce4e5b9ull;
    hsh ^= hsh >> 32;
    W2MapEntry &e = table[hsh % kEntries];
    {
        std::lock_guard<std::mutex> lock(mu);
        if (e.q == w.w2_q && e.meta == w.w2_meta && e.num_experts == s.num_experts && e.inter == s.inter &&
            e.meta_bytes == s.meta_bytes && e.tiles == tiles) {
            *tq = e.tq;
            *tm = e.tm;
            return true;
        }
    }
    const uint64_t all = static_cast<uint64_t>(s.num_experts) * (s.inter / 160) * kColTiles;
    if (!make_line_map(tq, w.w2_q, all * kW2TileKK, tiles * kW2TileKK) ||
        !make_row_map(tm, w.w2_meta, all * 5, s.meta_bytes, tiles * 5))
        return false;
    std::lock_guard<std::mutex> lock(mu);
    e.q = w.w2_q;
    e.meta = w.w2_meta;
    e.num_experts = s.num_experts;
    e.inter = s.inter;
    e.meta_bytes = s.meta_bytes;
    e.tiles = tiles;
    e.tq = *tq;
    e.tm = *tm;
    return true;
}

// The sliced decode kernel views the same prepared W2 banks in 3D: q as
// [tile (e, kp, 32-column tile)][20 word rows][32 words], one word row of 40
// consecutive tiles per box; metadata as [tile][5 groups][32 records], one
// group row of 40 tiles per box. Neither is swizzled.
bool make_w2_maps3(const awq_moe_shape &s, const awq_moe_weights &w, CUtensorMap *tq, CUtensorMap *tm)
{
    constexpr uint64_t kEntries = 256;
    static W2MapEntry table[kEntries];
    static std::mutex mu;
    uint64_t hsh = reinterpret_cast<uintptr_t>(w.w2_q) ^ (reinterpret_cast<uintptr_t>(w.w2_meta) << 5) ^
                   (static_cast<uint64_t>(s.inter) << 9) ^ static_cast<uint64_t>(s.meta_bytes);
    hsh ^= hsh >> 31;
    hsh *= 0x94d049bb133111ebull;
    hsh ^= hsh >> 29;
    W2MapEntry &e = table[hsh % kEntries];
    {
        std::lock_guard<std::mutex> lock(mu);
        if (e.q == w.w2_q && e.meta == w.w2_meta && e.num_experts == s.num_experts && e.inter == s.inter &&
            e.meta_bytes == s.meta_bytes) {
            *tq = e.tq;
            *tm = e.tm;
            return true;
        }
    }
    const uint64_t tiles = static_cast<uint64_t>(s.num_experts) * (s.inter / 160) * kColTiles;
    const uint64_t mb = s.meta_bytes;
    {
        cuuint64_t dims[3] = {32, kW2TileKK, tiles};
        cuuint64_t str[2] = {128, 128 * kW2TileKK};
        cuuint32_t box[3] = {32, 1, 40};
        // each box row is one 128-byte line: promoting it to 256 bytes would
        // fetch the next word row, which another box (or CTA) reads
        if (!encode(tq, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, w.w2_q, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B))
            return false;
    }
    {
        cuuint64_t dims[3] = {32 * mb, 5, tiles};
        cuuint64_t str[2] = {32 * mb, 160 * mb};
        cuuint32_t box[3] = {static_cast<cuuint32_t>(32 * mb), 1, 40};
        if (!encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, w.w2_meta, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B))
            return false;
    }
    std::lock_guard<std::mutex> lock(mu);
    e.q = w.w2_q;
    e.meta = w.w2_meta;
    e.num_experts = s.num_experts;
    e.inter = s.inter;
    e.meta_bytes = s.meta_bytes;
    e.tiles = -1;
    e.tq = *tq;
    e.tm = *tm;
    return true;
}

// The prefill path's W13 reads the prepared W13 bank through two 3D views:
// words [piece][K block of 64][128 words] and records [piece][K block][32 mb
// bytes], boxes of 8 pieces x kTcKbPerStage13 K blocks (one copy per ring
// stage for a column tile of 8 pieces). Kept in a small table like the W2 maps.
bool make_w13_maps(const awq_moe_shape &s, const awq_moe_weights &w, CUtensorMap *tq, CUtensorMap *tm)
{
    constexpr uint64_t kEntries = 256;
    static W2MapEntry table[kEntries];
    static std::mutex mu;
    uint64_t hsh = reinterpret_cast<uintptr_t>(w.w13_q) ^ (reinterpret_cast<uintptr_t>(w.w13_meta) << 5) ^
                   (static_cast<uint64_t>(s.inter) << 9) ^ static_cast<uint64_t>(s.meta_bytes);
    hsh ^= hsh >> 31;
    hsh *= 0xd6e8feb86659fd93ull;
    hsh ^= hsh >> 29;
    W2MapEntry &e = table[hsh % kEntries];
    {
        std::lock_guard<std::mutex> lock(mu);
        if (e.q == w.w13_q && e.meta == w.w13_meta && e.num_experts == s.num_experts && e.inter == s.inter &&
            e.meta_bytes == s.meta_bytes) {
            *tq = e.tq;
            *tm = e.tm;
            return true;
        }
    }
    const uint64_t pieces = static_cast<uint64_t>(s.num_experts) * (s.inter / kPieceCols);
    const uint64_t mb = prepared_record_bytes(s);
    {
        cuuint64_t dims[3] = {128, kHidden / 64, pieces};
        cuuint64_t str[2] = {512, kPieceQ};
        cuuint32_t box[3] = {128, kTcKbPerStage13, 8};
        if (!encode(tq, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, w.w13_q, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return false;
    }
    {
        cuuint64_t dims[3] = {32 * mb, kHidden / 64, pieces};
        cuuint64_t str[2] = {32 * mb, static_cast<cuuint64_t>(piece_meta_bytes(static_cast<int>(mb)))};
        cuuint32_t box[3] = {static_cast<cuuint32_t>(32 * mb), kTcKbPerStage13, 8};
        if (!encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, w.w13_meta, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return false;
    }
    std::lock_guard<std::mutex> lock(mu);
    e.q = w.w13_q;
    e.meta = w.w13_meta;
    e.num_experts = s.num_experts;
    e.inter = s.inter;
    e.meta_bytes = s.meta_bytes;
    e.tiles = -2;
    e.tq = *tq;
    e.tm = *tm;
    return true;
}

// The prefill path's W2 reads its B operand (h rows of a work item, K-major)
// with TMA: the two planes h f16[2 S][I] (fp16(h), then the residue)
// viewed 2D, boxes of 64 K x {16, 32, 64, 128} rows,
// 128-byte swizzle (the tensor core's operand layout). Built per call: h
// lives in the caller's workspace.
bool make_h_maps(const awq_moe_shape &s, const uint16_t *h, int S, CUtensorMap (&th)[4])
{
    for (int i = 0; i < 4; ++i) {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(s.inter), static_cast<cuuint64_t>(2 * S)};
        cuuint64_t str[1] = {static_cast<cuuint64_t>(2 * s.inter)};
        cuuint32_t box[2] = {64, 16u << i};
        if (!encode(&th[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, h, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return false;
    }
    return true;
}

// ----------------------------------------------------------------- launches

StageArgs base_args(int32_t M, const awq_moe_shape &s, const int32_t *ids, const int32_t *off,
                    const int32_t *slots, const int32_t *na, int32_t *status)
{
    StageArgs a = {};
    a.active_ids = ids;
    a.offsets = off;
    a.sorted_slots = slots;
    a.num_active = na;
    a.status = status;
    a.M = M;
    a.top_k = s.top_k;
    a.num_experts = s.num_experts;
    a.inter = s.inter;
    a.timeout_ns = kDefaultTimeoutNs;
    return a;
}

awq_status run_route(const int32_t *topk_ids, int32_t M, const awq_moe_shape &s, int32_t *ids,
                     int32_t *off, int32_t *slots, int32_t *na, int32_t *status, cudaStream_t st)
{
    const int smem = route_smem_bytes(M * s.top_k, s.num_experts);
    awq_status r = set_smem(route_kernel, smem);
    if (r) return r;
    return launch(route_kernel, dim3(1), dim3(kRouteThreads), smem, 1, st, topk_ids, M * s.top_k,
                  static_cast<int32_t>(s.num_experts), ids, off, slots, na, status);
}

awq_status run_w13(const awq_moe_weights &w, const uint16_t *x, int32_t M, const awq_moe_shape &s,
                   const int32_t *ids, const int32_t *off, const int32_t *slots, const int32_t *na,
                   uint16_t *h, int32_t *status, cudaStream_t st, uint16_t *h_lo = nullptr,
                   uint64_t *trace = nullptr, bool stage_kernel = false)
{
    StageArgs a = base_args(M, s, ids, off, slots, na, status);
    a.trace = trace;
    a.w13_q = w.w13_q;
    a.w13_meta = w.w13_meta;
    a.global_scale = w.global_scale;
    a.x = x;
    a.h_out = h;
    a.h_lo = h_lo;
    if (M > kStagedMaxTokens && !stage_kernel) {
        CUtensorMap tq13, tm13;
        if (!make_w13_maps(s, w, &tq13, &tm13)) return AWQ_ERR_CUDA;
        return launch_w13_tc(prepared_record_bytes(s), M * s.top_k, current_sm_count(), st, tq13, tm13, a);
    }
    const int a_max = std::min(M * s.top_k, s.num_experts);
    return launch_w13(prepared_record_bytes(s), dim3(s.inter / kPieceCols, a_max), st, a);
}

awq_status run_w2(const CUtensorMap &tq, const CUtensorMap &tm, const uint16_t *h, const float *wts,
                  int32_t M, const awq_moe_shape &s, const int32_t *ids, const int32_t *off,
                  const int32_t *slots, const int32_t *na, uint16_t *out, int32_t *status,
                  cudaStream_t st)
{
    StageArgs a = base_args(M, s, ids, off, slots, na, status);
    a.h_in = h;
    a.topk_weights = wts;
    a.out = out;
    return launch_w2(s.meta_bytes, dim3(kW2Cluster, kHidden / kW2ColTile), st, tq, tm, a);
}

// Workspace: a counter region first (zero between calls; only the fused
// kernel touches it), then one region shared by the two paths.
struct WorkspaceLayout {
    size_t sync, cnt2, sense, gbar, region;           // counters
    size_t ids, off, slots, na, h;                    // three-launch and prefill paths
    size_t y;                                         // prefill path: f32[S][H] products
    size_t part2, hw, hw_lo;                          // fused path (hw_lo: NVFP4 banks)
    size_t part3;                                     // sliced path
    size_t total;
};

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

WorkspaceLayout workspace_layout(const awq_moe_shape &s, int32_t M)
{
    const size_t S = static_cast<size_t>(M) * s.top_k;
    const size_t a_max = std::min<size_t>(S, s.num_experts);
    WorkspaceLayout L;
    // The counter region must not move with M: a workspace sized for M_max
    // serves calls of every M <= M_max, and its counters carry over between
    // calls. It is a fixed 2 KB.
    L.sync = 0;
    L.cnt2 = 64;
    L.sense = 256;
    L.gbar = 1536;
    L.region = 2048;
    static_assert(256 + 4 * kMaxGrid <= 1536, "sense words fit below the grid barrier words");
    // three launches
    L.ids = L.region;
    L.off = up256(L.ids + 4 * S);
    L.slots = up256(L.off + 4 * (S + 1));
    L.na = up256(L.slots + 4 * S);
    L.h = up256(L.na + 4);
    const size_t end3 = up256(L.h + 2 * S * s.inter);
    // the prefill path keeps a second fp16 plane of h (the residue) after the first
    L.y = up256(L.h + 2 * 2 * S * s.inter);
    const size_t endp = up256(L.y + sizeof(float) * S * kHidden);
    // fused (only for M <= kFusedMaxTokens)
    L.part2 = L.region;
    L.hw = up256(L.part2 + sizeof(float) * kMaxGrid * 2 * kPartStride);
    const size_t mp = M > 8 ? 16 : 8;
    // NVFP4 banks: the fp16 residue plane of hw after it
    L.hw_lo = up256(L.hw + 2 * a_max * mp * s.inter);
    const size_t endf = M <= kFusedMaxTokens ? (is_nvfp4(s) ? up256(L.hw_lo + 2 * a_max * mp * s.inter) : L.hw_lo) : 0;
    // sliced (only for M <= kSlicedMaxTokens): per-CTA fp32 partial outputs
    L.part3 = L.region;
    const size_t ends = M <= kSlicedMaxTokens
                            ? up256(L.part3 + sizeof(float) * kMaxGrid * M * kHidden)
                            : 0;
    L.total = std::max(std::max(endp, endf), ends);
    return L;
}

}  // namespace
}  // namespace awq

using namespace awq;

extern "C" {

const char *awq_status_string(awq_status st)
{
    switch (st) {
    case AWQ_OK: return "ok";
    case AWQ_ERR_INVALID_ARG: return "invalid argument (null pointer or value out of range)";
    case AWQ_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case AWQ_ERR_MISALIGNED: return "misaligned pointer";
    case AWQ_ERR_CUDA: return "CUDA runtime or driver call failed";
    case AWQ_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case AWQ_ERR_BAD_EXPERT_ID: return "expert id outside [0, num_experts)";
    case AWQ_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than awq_moe_workspace_bytes()";
    case AWQ_ERR_LAYOUT: return "weight banks are not in the layout the call needs";
    }
    return "unknown status";
}

size_t awq_moe_workspace_bytes(const awq_moe_shape *shape, int32_t M_max)
{
    if (check_shape(shape) != AWQ_OK || M_max < 1 || M_max > AWQ_MAX_TOKENS) return 0;
    // The need is not monotone in M: calls of up to kFusedMaxTokens tokens
    // take the fused path, whose per-CTA partial blocks outweigh the three
    // launches' arrays of a larger M. The largest need over 1..M_max serves
    // every call of at most M_max tokens.
    size_t total = 0;
    for (int32_t M = 1; M <= M_max; ++M) total = std::max(total, workspace_layout(*shape, M).total);
    return total;
}

awq_status awq_moe_prepare_weights(const awq_moe_shape *shape, const awq_moe_weights *src,
                                   awq_moe_weights *dst, void *stream)
{
    awq_status r = check_shape(shape);
    if (r) return r;
    if ((r = check_banks(src))) return r;
    if (!dst) return AWQ_ERR_INVALID_ARG;
    awq_moe_weights d = *dst;
    d.layout = AWQ_LAYOUT_PREPARED;
    if ((r = check_banks(&d))) return r;
    if (src->layout != AWQ_LAYOUT_CANONICAL) return AWQ_ERR_LAYOUT;
    const uint64_t E = shape->num_experts, I = shape->inter, H = kHidden, mb = shape->meta_bytes;
    const uint64_t G = shape->group;
    const uint64_t bytes[4] = {E * (H / 8) * 2 * I * 4, E * (H / G) * 2 * I * mb, E * (I / 8) * H * 4,
                               E * (I / G) * H * mb};
    const void *sp[4] = {src->w13_q, src->w13_meta, src->w2_q, src->w2_meta};
    const void *dp[4] = {d.w13_q, d.w13_meta, d.w2_q, d.w2_meta};
    for (int i = 0; i < 4; ++i)
        for (int j = 0; j < 4; ++j) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(sp[i]), b = reinterpret_cast<uintptr_t>(dp[j]);
            if (a < b + bytes[j] && b < a + bytes[i]) return AWQ_ERR_INVALID_ARG;   // overlap
        }
    if ((r = launch_prepare(*shape, *src, d, static_cast<cudaStream_t>(stream)))) return r;
    dst->layout = AWQ_LAYOUT_PREPARED;
    return AWQ_OK;
}

awq_status awq_prepare_compact(const uint8_t *meta4, uint8_t *meta3, int64_t n_records, void *stream)
{
    if (n_records < 0) return AWQ_ERR_INVALID_ARG;
    if (n_records == 0) return AWQ_OK;
    if (!meta4 || !meta3) return AWQ_ERR_INVALID_ARG;
    const uintptr_t a4 = reinterpret_cast<uintptr_t>(meta4), a3 = reinterpret_cast<uintptr_t>(meta3);
    if (a3 < a4 + 4 * static_cast<uintptr_t>(n_records) && a4 < a3 + 3 * static_cast<uintptr_t>(n_records))
        return AWQ_ERR_INVALID_ARG;   // overlapping buffers
    const int32_t vec = (aligned(meta4, 16) && aligned(meta3, 4)) ? 1 : 0;
    const int64_t work = (n_records + 3) / 4;
    const int blocks = static_cast<int>(std::min<int64_t>((work + 255) / 256, 152 * 16));
    return launch(prepare_compact_kernel, dim3(blocks), dim3(256), 0, 1,
                  static_cast<cudaStream_t>(stream), meta4, meta3, n_records, vec);
}

awq_status awq_moe_route(const int32_t *topk_ids, int32_t M, const awq_moe_shape *shape,
                         int32_t *active_expert_ids, int32_t *active_expert_offsets,
                         int32_t *sorted_slots, int32_t *num_active, int32_t *dev_status,
                         void *stream)
{
    awq_status r = check_shape(shape);
    if (r) return r;
    if ((r = check_m(M))) return r;
    if (!active_expert_offsets || !num_active || !dev_status) return AWQ_ERR_INVALID_ARG;
    if (M > 0 && (!topk_ids || !active_expert_ids || !sorted_slots)) return AWQ_ERR_INVALID_ARG;
    return run_route(topk_ids, M, *shape, active_expert_ids, active_expert_offsets, sorted_slots,
                     num_active, dev_status, static_cast<cudaStream_t>(stream));
}

awq_status awq_moe_w13_swiglu(const uint16_t *x, int32_t M, const awq_moe_shape *shape,
                              const awq_moe_weights *weights, const int32_t *active_expert_ids,
                              const int32_t *active_expert_offsets, const int32_t *sorted_slots,
                              const int32_t *num_active, uint16_t *h, int32_t *dev_status,
                              void *stream)
{
    awq_status r = check_shape(shape);
    if (r) return r;
    if ((r = check_m(M))) return r;
    if ((r = check_weights(weights))) return r;
    if (is_nvfp4(*shape)) return AWQ_ERR_UNSUPPORTED_SHAPE;   // NVFP4: the layer calls only
    if (M == 0) return AWQ_OK;
    if (!x || !active_expert_ids || !active_expert_offsets || !sorted_slots || !num_active || !h ||
        !dev_status)
        return AWQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(h, 16)) return AWQ_ERR_MISALIGNED;
    return run_w13(*weights, x, M, *shape, active_expert_ids, active_expert_offsets, sorted_slots,
                   num_active, h, dev_status, static_cast<cudaStream_t>(stream));
}

awq_status awq_moe_w2_reduce(const uint16_t *h, const float *topk_weights, int32_t M,
                             const awq_moe_shape *shape, const awq_moe_weights *weights,
                             const int32_t *active_expert_ids, const int32_t *active_expert_offsets,
                             const int32_t *sorted_slots, const int32_t *num_active, uint16_t *out,
                             int32_t *dev_status, void *stream)
{
    awq_status r = check_shape(shape);
    if (r) return r;
    if ((r = check_m(M))) return r;
    if ((r = check_weights(weights))) return r;
    if (is_nvfp4(*shape)) return AWQ_ERR_UNSUPPORTED_SHAPE;   // NVFP4: the layer calls only
    if (M == 0) return AWQ_OK;
    if (!h || !topk_weights || !active_expert_ids || !active_expert_offsets || !sorted_slots ||
        !num_active || !out || !dev_status)
        return AWQ_ERR_INVALID_ARG;
    if (!aligned(h, 16) || !aligned(out, 16) || !aligned(topk_weights, 4)) return AWQ_ERR_MISALIGNED;
    if (M > kStagedMaxTokens) return AWQ_ERR_UNSUPPORTED_SHAPE;
    CUtensorMap tq, tm;
    if (!make_w2_maps(*shape, *weights, 1, &tq, &tm)) return AWQ_ERR_CUDA;
    return run_w2(tq, tm, h, topk_weights, M, *shape, active_expert_ids, active_expert_offsets,
                  sorted_slots, num_active, out, dev_status, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace awq {
namespace {

awq_status run_router(const float *logits, int32_t M, const awq_moe_shape &s, int32_t *ids, float *w,
                      cudaStream_t st)
{
    return launch(router_topk_kernel, dim3((M + kRouterWarps - 1) / kRouterWarps), dim3(kRouterWarps * 32), 0,
                  1, st, logits, M, static_cast<int32_t>(s.top_k), ids, w);
}

// The layer call, from topk_ids / topk_weights or (logits non-null) from
// router logits, whose choice goes to ids_out / w_out.
awq_status layer_impl(const uint16_t *x, const int32_t *topk_ids, const float *topk_weights,
                      const float *logits, int32_t *ids_out, float *w_out, int32_t M,
                      const awq_moe_shape *shape, const awq_moe_weights *weights, uint16_t *out,
                      void *workspace, size_t ws_bytes, int32_t *dev_status, const awq_moe_options *opts,
                      void *stream)
{
    awq_status r = check_shape(shape);
    if (r) return r;
    if ((r = check_m(M))) return r;
    if ((r = check_weights(weights))) return r;
    if ((r = check_global(*shape, *weights))) return r;
    const int path = opts ? opts->path : AWQ_PATH_AUTO;
    if (path < AWQ_PATH_AUTO || path > AWQ_PATH_HYBRID) return AWQ_ERR_INVALID_ARG;
    if (M == 0) return AWQ_OK;
    if (!x || !out || !workspace || !dev_status) return AWQ_ERR_INVALID_ARG;
    if (logits ? (!ids_out || !w_out) : (!topk_ids || !topk_weights)) return AWQ_ERR_INVALID_ARG;
    if (logits && (shape->num_experts != kRouterExperts || shape->top_k > 32)) return AWQ_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(x, 16) || !aligned(out, 16) || !aligned(workspace, 256)) return AWQ_ERR_MISALIGNED;
    if (logits ? (!aligned(logits, 4) || !aligned(ids_out, 4) || !aligned(w_out, 4)) : !aligned(topk_weights, 4))
        return AWQ_ERR_MISALIGNED;
    const WorkspaceLayout L = workspace_layout(*shape, M);
    if (ws_bytes < L.total) return AWQ_ERR_WORKSPACE_TOO_SMALL;
    const int sms = current_sm_count();
    const bool fused_ok = M <= kFusedMaxTokens && sms >= kFusedMinSms && sms <= kMaxGrid;
    // the sliced kernel: a CTA's share spans at most two segments when
    // M * top_k <= grid (at most M * top_k active experts)
    const bool sliced_ok = M <= kSlicedMaxTokens && M * shape->top_k <= sms && sms >= kFusedMinSms &&
                           sms <= kMaxGrid;
    if (path == AWQ_PATH_FUSED && !fused_ok) return AWQ_ERR_UNSUPPORTED_SHAPE;
    if (path == AWQ_PATH_SLICED && !sliced_ok) return AWQ_ERR_UNSUPPORTED_SHAPE;
    if (path == AWQ_PATH_STAGED && M > kStagedMaxTokens) return AWQ_ERR_UNSUPPORTED_SHAPE;
    // NVFP4 banks run on the fused decode kernel, the hybrid path and the
    // tensor-core prefill path; all three carry the fp16 residue of the
    // (weighted) activations into W2. (A single fp16 rounding of them put
    // about one output in 20,000-40,000 of NVFP4 layers outside the stage's
    // tolerance.)
    const bool nv = is_nvfp4(*shape);
    if (nv && path != AWQ_PATH_AUTO && path != AWQ_PATH_PREFILL && path != AWQ_PATH_HYBRID &&
        path != AWQ_PATH_FUSED)
        return AWQ_ERR_UNSUPPORTED_SHAPE;
    // AWQ_PATH_AUTO takes, per call shape, whichever persistent kernel measured
    // faster on GB300 (both within the same tolerance): the sliced kernel at
    // M = 2, and at M = 1 with intermediate 160 (its tile mode covers up to 24
    // active experts, where the fused kernel's W2 needs its split-group
    // exchange; at these sizes the host knows tile mode is certain and
    // launches the build without the flat-mode code), the fused kernel
    // otherwise.
    const bool sliced_auto = sliced_ok && (M == 2 || (M == 1 && shape->inter == 160));
    const bool sliced = !nv && (path == AWQ_PATH_SLICED || (path == AWQ_PATH_AUTO && sliced_auto));
    const bool fused = !sliced && (path == AWQ_PATH_FUSED || (path == AWQ_PATH_AUTO && fused_ok));
    const uint64_t timeout = (opts && opts->timeout_ns) ? opts->timeout_ns : kDefaultTimeoutNs;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    if (sliced) {
        CUtensorMap tq, tm, t1q, t1m;
        if (!make_w2_maps3(*shape, *weights, &tq, &tm) || !make_w2_maps(*shape, *weights, 1, &t1q, &t1m))
            return AWQ_ERR_CUDA;
        SlicedArgs a = {};
        a.x = x;
        a.topk_ids = topk_ids;
        a.topk_weights = topk_weights;
        a.logits = logits;
        a.topk_ids_out = ids_out;
        a.topk_weights_out = w_out;
        a.out = out;
        a.w13_q = weights->w13_q;
        a.w13_meta = weights->w13_meta;
        a.part = reinterpret_cast<float *>(ws + L.part3);
        a.gbar = reinterpret_cast<uint64_t *>(ws + L.gbar);
        a.status = dev_status;
        a.M = M;
        a.top_k = shape->top_k;
        a.num_experts = shape->num_experts;
        a.inter = shape->inter;
        a.timeout_ns = timeout;
        a.debug_flags = opts ? opts->debug_flags : 0;
        a.trace = opts ? opts->trace : nullptr;
        return launch_sliced(shape->meta_bytes, sms, st, tq, tm, t1q, t1m, a);
    }

    if (fused) {
        CUtensorMap t2q, t2m;
        CUtensorMap t2q1, t2m1;   // one-tile boxes (the kernel's tile mode for few experts)
        awq_moe_shape ps = *shape;              // the prepared records' size (2 bytes for NVFP4)
        ps.meta_bytes = prepared_record_bytes(*shape);
        if (!make_w2_maps(ps, *weights, kFusedW2Tiles, &t2q, &t2m) || !make_w2_maps(ps, *weights, 1, &t2q1, &t2m1))
            return AWQ_ERR_CUDA;
        FusedArgs a = {};
        a.x = x;
        a.topk_ids = topk_ids;
        a.topk_weights = topk_weights;
        a.logits = logits;
        a.topk_ids_out = ids_out;
        a.topk_weights_out = w_out;
        a.out = out;
        a.w13_q = weights->w13_q;
        a.w13_meta = weights->w13_meta;
        a.hw = reinterpret_cast<uint16_t *>(ws + L.hw);
        a.part2 = reinterpret_cast<float *>(ws + L.part2);
        a.cnt2 = reinterpret_cast<int32_t *>(ws + L.cnt2);
        a.sync = reinterpret_cast<int32_t *>(ws + L.sync);
        a.sense = reinterpret_cast<int32_t *>(ws + L.sense);
        a.status = dev_status;
        a.M = M;
        a.top_k = shape->top_k;
        a.num_experts = shape->num_experts;
        a.inter = shape->inter;
        a.timeout_ns = timeout;
        a.debug_flags = opts ? opts->debug_flags : 0;
        a.global_scale = weights->global_scale;
        a.hw_lo = nv ? reinterpret_cast<uint16_t *>(ws + L.hw_lo) : nullptr;
        return launch_fused(ps.meta_bytes, sms, st, t2q, t2m, t2q1, t2m1, a);
    }

    int32_t *ids = reinterpret_cast<int32_t *>(ws + L.ids);
    int32_t *off = reinterpret_cast<int32_t *>(ws + L.off);
    int32_t *slots = reinterpret_cast<int32_t *>(ws + L.slots);
    int32_t *na = reinterpret_cast<int32_t *>(ws + L.na);
    uint16_t *h = reinterpret_cast<uint16_t *>(ws + L.h);
    const bool prefill = path == AWQ_PATH_PREFILL ||
                         (path == AWQ_PATH_AUTO && M > kHybridMaxTokens);
    // (AUTO reaches here below 17 tokens only on a grid the fused kernel does not take)
    const bool hybrid = !prefill && (path == AWQ_PATH_HYBRID || path == AWQ_PATH_AUTO);
    if (hybrid) {
        // W13 + SwiGLU by the stage kernel (h and its residue plane), then the
        // tensor-core W2 into per-slot products and the per-token sum
        CUtensorMap th[4];
        if (!make_h_maps(*shape, h, M * shape->top_k, th)) return AWQ_ERR_CUDA;
        if (logits) {
            if ((r = run_router(logits, M, *shape, ids_out, w_out, st))) return r;
            topk_ids = ids_out;
            topk_weights = w_out;
        }
        if ((r = run_route(topk_ids, M, *shape, ids, off, slots, na, dev_status, st))) return r;
        uint16_t *h_lo = h + static_cast<size_t>(M) * shape->top_k * shape->inter;
        if ((r = run_w13(*weights, x, M, *shape, ids, off, slots, na, h, dev_status, st, h_lo,
                         opts ? opts->trace : nullptr, true)))
            return r;
        StageArgs a = base_args(M, *shape, ids, off, slots, na, dev_status);
        a.timeout_ns = timeout;
        a.trace = opts ? opts->trace : nullptr;
        a.h_in = h;
        a.w2_q = weights->w2_q;
        a.w2_meta = weights->w2_meta;
        a.global_scale = weights->global_scale;
        a.topk_weights = topk_weights;
        float *y = reinterpret_cast<float *>(ws + L.y);
        a.y = y;
        if ((r = launch_w2_tc(prepared_record_bytes(*shape), M * shape->top_k, sms, st, th, a))) return r;
        return launch_combine(M, shape->top_k, y, out, a.trace, st);
    }
    if (prefill) {
        // every host-side step that can fail comes before the first launch
        CUtensorMap th[4], tq13, tm13;
        if (!make_h_maps(*shape, h, M * shape->top_k, th) || !make_w13_maps(*shape, *weights, &tq13, &tm13))
            return AWQ_ERR_CUDA;
        if (logits) {
            if ((r = run_router(logits, M, *shape, ids_out, w_out, st))) return r;
            topk_ids = ids_out;
            topk_weights = w_out;
        }
        if ((r = run_route(topk_ids, M, *shape, ids, off, slots, na, dev_status, st))) return r;
        StageArgs a = base_args(M, *shape, ids, off, slots, na, dev_status);
        a.timeout_ns = timeout;
        a.trace = opts ? opts->trace : nullptr;
        a.w13_q = weights->w13_q;
        a.w13_meta = weights->w13_meta;
        a.global_scale = weights->global_scale;
        a.x = x;
        a.h_out = h;
        a.h_lo = h + static_cast<size_t>(M) * shape->top_k * shape->inter;
        const int rb = prepared_record_bytes(*shape);
        if ((r = launch_w13_tc(rb, M * shape->top_k, sms, st, tq13, tm13, a))) return r;
        a.h_in = h;
        a.w2_q = weights->w2_q;
        a.w2_meta = weights->w2_meta;
        a.topk_weights = topk_weights;
        float *y = reinterpret_cast<float *>(ws + L.y);
        a.y = y;
        if ((r = launch_w2_tc(rb, M * shape->top_k, sms, st, th, a))) return r;
        return launch_combine(M, shape->top_k, y, out, a.trace, st);
    }
    // every host-side step that can fail comes before the first launch
    CUtensorMap t2q, t2m;
    if (!make_w2_maps(*shape, *weights, 1, &t2q, &t2m)) return AWQ_ERR_CUDA;
    if (logits) {
        if ((r = run_router(logits, M, *shape, ids_out, w_out, st))) return r;
        topk_ids = ids_out;
        topk_weights = w_out;
    }
    if ((r = run_route(topk_ids, M, *shape, ids, off, slots, na, dev_status, st))) return r;
    if ((r = run_w13(*weights, x, M, *shape, ids, off, slots, na, h, dev_status, st))) return r;
    return run_w2(t2q, t2m, h, topk_weights, M, *shape, ids, off, slots, na, out, dev_status, st);
}

}  // namespace
}  // namespace awq

extern "C" {

awq_status awq_moe_layer_ex(const uint16_t *x, const int32_t *topk_ids, const float *topk_weights,
                            int32_t M, const awq_moe_shape *shape, const awq_moe_weights *weights,
                            uint16_t *out, void *workspace, size_t ws_bytes, int32_t *dev_status,
                            const awq_moe_options *opts, void *stream)
{
    return layer_impl(x, topk_ids, topk_weights, nullptr, nullptr, nullptr, M, shape, weights, out, workspace,
                      ws_bytes, dev_status, opts, stream);
}

awq_status awq_moe_layer_logits(const uint16_t *x, const float *logits, int32_t M,
                                const awq_moe_shape *shape, const awq_moe_weights *weights,
                                uint16_t *out, int32_t *topk_ids, float *topk_weights, void *workspace,
                                size_t ws_bytes, int32_t *dev_status, const awq_moe_options *opts,
                                void *stream)
{
    if (M > 0 && !logits) return AWQ_ERR_INVALID_ARG;
    return layer_impl(x, nullptr, nullptr, logits, topk_ids, topk_weights, M, shape, weights, out, workspace,
                      ws_bytes, dev_status, opts, stream);
}

awq_status awq_moe_router_topk(const float *logits, int32_t M, const awq_moe_shape *shape,
                               int32_t *topk_ids, float *topk_weights, void *stream)
{
    awq_status r = check_shape(shape);
    if (r) return r;
    if (shape->num_experts != kRouterExperts || shape->top_k > 32) return AWQ_ERR_UNSUPPORTED_SHAPE;
    if ((r = check_m(M))) return r;
    if (M == 0) return AWQ_OK;
    if (!logits || !topk_ids || !topk_weights) return AWQ_ERR_INVALID_ARG;
    if (!aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(topk_weights, 4)) return AWQ_ERR_MISALIGNED;
    return run_router(logits, M, *shape, topk_ids, topk_weights, static_cast<cudaStream_t>(stream));
}

awq_status awq_moe_layer(const uint16_t *x, const int32_t *topk_ids, const float *topk_weights,
                         int32_t M, const awq_moe_shape *shape, const awq_moe_weights *weights,
                         uint16_t *out, void *workspace, size_t ws_bytes, int32_t *dev_status,
                         void *stream)
{
    return awq_moe_layer_ex(x, topk_ids, topk_weights, M, shape, weights, out, workspace, ws_bytes,
                            dev_status, nullptr, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Layer call without a caller-provided workspace.
//
// Some callers cannot hand the library device scratch: a plain C host or a
// plugin that owns no device allocator, or a serving process whose device
// memory is planned up front and that forbids allocation on the request
// path. awq_moe_layer_static serves them from one fixed array in the
// library's own device memory, created with the module (zero-filled, never
// freed), so neither the library nor the caller allocates anything per call.
// Its device address is looked up with cudaGetSymbolAddress, with the device
// current, on every call.
//
// It runs the three-launch path (route, W13 + SwiGLU, W2 + reduction): those
// kernels fully rewrite every scratch byte they read, so nothing in the array
// has to start at zero and an earlier failed call leaves nothing behind. The
// array is shared by every call on a device: two calls that can overlap in
// time (different streams, or different host threads without ordering) race
// on it and give undefined results.
namespace awq {
namespace {

__device__ __align__(256) uint8_t g_static_scratch[AWQ_STATIC_SCRATCH_BYTES];

// Device address of g_static_scratch in the current device's context, looked
// up on every call. The lookup is cheap once the module is loaded (the first
// call on a device loads it: that is the set-up), and it is never stale: a
// context torn down and created again (cudaDeviceReset) reloads the module,
// possibly at another address, which a cached pointer would not follow.
void *static_scratch()
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
    return p;
}

}  // namespace
}  // namespace awq

extern "C" awq_status awq_moe_latency_floor(const int32_t *topk_ids, int32_t M, const awq_moe_shape *shape,
                                            const awq_moe_weights *weights, uint16_t *out, void *workspace,
                                            size_t ws_bytes, int32_t *dev_status, void *stream)
{
    awq_status r = check_shape(shape);
    if (r) return r;
    if ((r = check_weights(weights))) return r;
    if (M < 0 || M > kFusedMaxTokens) return AWQ_ERR_INVALID_ARG;
    if (M == 0) return AWQ_OK;
    if (!topk_ids || !out || !workspace || !dev_status) return AWQ_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(workspace, 256)) return AWQ_ERR_MISALIGNED;
    const WorkspaceLayout L = workspace_layout(*shape, M);
    if (ws_bytes < L.region) return AWQ_ERR_WORKSPACE_TOO_SMALL;
    const int sms = current_sm_count();
    if (sms < 1 || sms > kMaxGrid) return AWQ_ERR_UNSUPPORTED_SHAPE;
    return launch_floor(topk_ids, M, *shape, *weights, out,
                        reinterpret_cast<uint64_t *>(static_cast<uint8_t *>(workspace) + L.gbar), dev_status,
                        kDefaultTimeoutNs, sms, static_cast<cudaStream_t>(stream));
}

extern "C" awq_status awq_moe_layer_static(const uint16_t *x, const int32_t *topk_ids,
                                           const float *topk_weights, int32_t M,
                                           const awq_moe_shape *shape,
                                           const awq_moe_weights *weights, uint16_t *out,
                                           int32_t *dev_status, void *stream)
{
    awq_status r = check_shape(shape);
    if (r) return r;
    if ((r = check_m(M))) return r;
    if ((r = check_weights(weights))) return r;
    if (is_nvfp4(*shape)) return AWQ_ERR_UNSUPPORTED_SHAPE;   // the three launches take int4 banks only
    if (M == 0) return AWQ_OK;
    if (!x || !topk_ids || !topk_weights || !out || !dev_status) return AWQ_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(out, 16) || !aligned(topk_weights, 4)) return AWQ_ERR_MISALIGNED;
    if (M > kStagedMaxTokens) return AWQ_ERR_UNSUPPORTED_SHAPE;
    // the three-launch path's part of the workspace layout must fit the array
    const WorkspaceLayout L = workspace_layout(*shape, M);
    const size_t need = up256(L.h + 2 * static_cast<size_t>(M) * shape->top_k * shape->inter);
    if (need > AWQ_STATIC_SCRATCH_BYTES) return AWQ_ERR_WORKSPACE_TOO_SMALL;
    CUtensorMap t2q, t2m;
    if (!make_w2_maps(*shape, *weights, 1, &t2q, &t2m)) return AWQ_ERR_CUDA;
    uint8_t *ws = static_cast<uint8_t *>(static_scratch());
    if (!ws) return AWQ_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t *ids = reinterpret_cast<int32_t *>(ws + L.ids);
    int32_t *off = reinterpret_cast<int32_t *>(ws + L.off);
    int32_t *slots = reinterpret_cast<int32_t *>(ws + L.slots);
    int32_t *na = reinterpret_cast<int32_t *>(ws + L.na);
    uint16_t *h = reinterpret_cast<uint16_t *>(ws + L.h);
    if ((r = run_route(topk_ids, M, *shape, ids, off, slots, na, dev_status, st))) return r;
    if ((r = run_w13(*weights, x, M, *shape, ids, off, slots, na, h, dev_status, st))) return r;
    return run_w2(t2q, t2m, h, topk_weights, M, *shape, ids, off, slots, na, out, dev_status, st);
}
