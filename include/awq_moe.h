/*
 * awq_moe.h -- C ABI of the GB300 (sm_103a) AWQ int4 mixture-of-experts
 * expert stage for decode and small prefill batches.
 *
 * The stage, as the pages define it (1Cat-vLLM #520 "Narrow Qwen3.8 AWQ
 * active grouped decode", Purpose and Implementation; 1Cat-vLLM #522
 * "Coalesce AWQ QPN W13 compact metadata loads and enable compact metadata by
 * default", Purpose and Default switch; Leonccaa/1Cat-vLLM #12 "Add opt-in
 * native-g32 AWQ QPN M1 dispatch", Purpose and stack):
 *
 *   (a) routing metadata: the per-token top-k expert ids become the ascending
 *       list of distinct active experts and CSR offsets of their row segments
 *       (active_expert_ids / active_expert_offsets, mutated outputs);
 *   (b) one offsets-scheduled grouped W13 GEMM (K = hidden -> N = 2*inter,
 *       gate columns 0..inter-1, up columns inter..2*inter-1) with SwiGLU;
 *   (c) one grouped W2 GEMM (K = inter -> N = hidden) with the router-weighted
 *       top-k reduction into the token output.
 *
 * Weights are AWQ int4, group 32 along K, with one metadata record per
 * (group, output column): {fp16 scale, u8 zero} (+ 1 pad byte in the 4-byte
 * layout). Dequantisation: w[k][n] = (q[k][n] - zero[k/32][n]) * scale[k/32][n].
 *
 * Canonical bank layouts (all row-major, last index fastest; E = num_experts,
 * H = hidden, I = inter, mb = meta_bytes):
 *   w13_q    u32[E][H/8][2I]     nibble j (bits 4j..4j+3) of word (i, n) is row 8i+j
 *   w13_meta u8 [E][H/32][2I][mb] bytes 0-1 fp16 scale (little-endian), byte 2 zero
 *   w2_q     u32[E][I/8][H]
 *   w2_meta  u8 [E][I/32][H][mb]
 *   x        fp16[M][H]           (fp16 values passed as uint16_t bit patterns)
 *   topk_ids i32[M][k], topk_weights f32[M][k]; slot s = t*k + j
 *   h        fp16[M*k][I]         rows in sorted-slot order (row r is slot sorted_slots[r])
 *   out      fp16[M][H]
 * The compute calls read PREPARED banks (awq_moe_prepare_weights): the same
 * bytes, permuted in 16-byte pieces so that each unit of work is one
 * contiguous block. Sizes are unchanged.
 *
 * Conventions common to every call:
 *   - every pointer argument is a DEVICE pointer unless stated otherwise;
 *     shape and weights structs are read on the host during the call and may
 *     be freed afterwards;
 *   - all memory is owned by the caller; the library allocates nothing and
 *     keeps no state between calls except the looked-up address of the
 *     driver's tensor-map encoder, each device's multiprocessor count and
 *     occupancy of the persistent kernel, and a table of encoded W2 tensor
 *     maps (a pure function of bank addresses, shape and box);
 *   - work is enqueued asynchronously on `stream` (a cudaStream_t; NULL means
 *     the legacy default stream); the call never synchronises the device and
 *     may be captured in a CUDA graph;
 *   - problems the host can see (null pointers, unsupported shapes, sizes out
 *     of range, misaligned pointers, a too-small workspace) are rejected
 *     synchronously with a non-zero awq_status and NOTHING is launched
 *     (fail closed: there is no fallback path);
 *   - problems only the data can show are reported through `dev_status`, a
 *     device int32 the caller zeroes beforehand and reads after the stream
 *     has synchronised: the first error code raised is kept. An expert id
 *     outside [0, E) gives AWQ_ERR_BAD_EXPERT_ID (outputs then undefined); a
 *     device-side wait that exceeds its time limit gives
 *     AWQ_ERR_DEVICE_TIMEOUT.
 *
 * NVFP4 weights (the second weight format; shape group 16, meta_bytes 1): the
 * same packed words hold FP4 E2M1 codes (sign, 2 exponent bits with bias 1, 1
 * mantissa bit), the metadata banks hold one FP8 E4M3 scale code per block of
 * 16 consecutive K elements of a column (u8[E][K/16][N], the record formula
 * above with group 16 and mb 1), and awq_moe_weights.global_scale holds one
 * fp32 scale per expert and matrix: w[k][n] = e2m1(q) * e4m3(scale[k/16][n]) *
 * global. The pages name a native NVFP4 kernel only as a comparison column
 * (#520 Results, #522 Operator results); the format is the published NVFP4
 * definition. NVFP4 banks run on the fused decode kernel, the hybrid path and
 * the tensor-core prefill path, each of which carries the fp16 residue of the
 * activations that enter W2 (the stage calls, the sliced path and
 * awq_moe_layer_static return AWQ_ERR_UNSUPPORTED_SHAPE); E4M3 NaN scale
 * codes are not supported.
 *
 * Supported shapes: num_experts 1..1024, top_k 1..16, hidden 2560,
 * inter 160 or 640, (group 32, meta_bytes 3 or 4) for int4 or (group 16,
 * meta_bytes 1) for NVFP4, M (tokens) 0..AWQ_MAX_TOKENS.
 * Alignment: weight banks, x, h and out 16-byte aligned; workspace 256-byte
 * aligned. Weight banks given to the compute calls must be prepared
 * (layout AWQ_LAYOUT_PREPARED), else AWQ_ERR_LAYOUT.
 */
#ifndef AWQ_MOE_H
#define AWQ_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define AWQ_MAX_TOKENS 512
/* awq_moe_w2_reduce and awq_moe_layer_static take at most this many tokens
 * (their W2 kernel keeps every token's output tile in shared memory); the
 * layer calls reach AWQ_MAX_TOKENS through the workspace. */
#define AWQ_W2_STAGE_MAX_TOKENS 128

#if defined(__GNUC__)
#define AWQ_API __attribute__((visibility("default")))
#else
#define AWQ_API
#endif

typedef enum {
    AWQ_OK = 0,
    AWQ_ERR_INVALID_ARG = 1,        /* null pointer or value out of range       */
    AWQ_ERR_UNSUPPORTED_SHAPE = 2,  /* shape outside the supported set          */
    AWQ_ERR_MISALIGNED = 3,         /* a pointer breaks its alignment rule      */
    AWQ_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed        */
    AWQ_ERR_DEVICE_TIMEOUT = 5,     /* a bounded device wait ran out (dev_status) */
    AWQ_ERR_BAD_EXPERT_ID = 6,      /* expert id outside [0, E) (dev_status)    */
    AWQ_ERR_WORKSPACE_TOO_SMALL = 7, /* ws_bytes below awq_moe_workspace_bytes  */
    AWQ_ERR_LAYOUT = 8              /* weight banks in the wrong layout         */
} awq_status;

/* Layout of a weight bank set. */
typedef enum {
    AWQ_LAYOUT_CANONICAL = 0,  /* the row-major layouts above */
    AWQ_LAYOUT_PREPARED = 1    /* written by awq_moe_prepare_weights */
} awq_layout;

typedef struct {
    int32_t num_experts;  /* E */
    int32_t top_k;        /* k */
    int32_t hidden;       /* H: W13 K and W2 N */
    int32_t inter;        /* I: W13 N is 2I (gate | up), W2 K */
    int32_t group;        /* quantisation group along K: 32 (int4), 16 (NVFP4 block) */
    int32_t meta_bytes;   /* 4: {scale, zero, pad}; 3: {scale, zero} packed;
                             1: NVFP4 E4M3 block scale */
} awq_moe_shape;

typedef struct {
    const uint32_t *w13_q;    /* u32[E][H/8][2I]      device (canonical shape/size) */
    const uint8_t *w13_meta;  /* u8 [E][H/32][2I][mb] device */
    const uint32_t *w2_q;     /* u32[E][I/8][H]       device */
    const uint8_t *w2_meta;   /* u8 [E][I/32][H][mb]  device */
    int32_t layout;           /* awq_layout of all four banks */
    const float *global_scale; /* NVFP4: f32[E][2] (W13, W2) device, 4-byte aligned,
                                  not permuted by preparation; NULL for int4 */
} awq_moe_weights;

/*
 * awq_moe_prepare_weights -- load-time permutation of canonical banks into
 * the prepared layout the compute calls stream.
 * Source: Leonccaa/1Cat-vLLM #12 "Add opt-in native-g32 AWQ QPN M1 dispatch",
 * Purpose and stack (prepared g32 batched banks, W13 interleaving, built once
 * at load time). The permutation moves whole packed words and whole metadata
 * records: a prepared bank decodes to exactly the weights of its source.
 * Prepared order (PJ = I/8 W13 pieces per expert, KP = I/160):
 *   w13_q    pieces (e, j 0..PJ-1) of 20480 bytes; word (group 0..79, t 0..3,
 *            g 0..7, half 0..1) of a piece is packed row 4*group + t, column
 *            half*I + 8j + g (gate and up columns interleaved)
 *   w13_meta pieces (e, j) of 1280*mb bytes; record (group, g, half) is the
 *            record of column half*I + 8j + g
 *   w2_q     128-byte lines (e, kp, tile 0..79, r 0..19): packed row
 *            20kp + r, columns 32*tile .. 32*tile+31
 *   w2_meta  rows of 32 records (e, kp, tile, g 0..4): group 5kp + g,
 *            columns 32*tile .. 32*tile+31
 * For NVFP4 banks the words move the same way and the prepared records are
 * 2 bytes per (group of 32, column): the scale codes of blocks 2*group and
 * 2*group + 1 of that column (records of 2 bytes in the orders above).
 * src: canonical banks (layout AWQ_LAYOUT_CANONICAL, device). dst: four
 * caller-allocated device buffers of the same sizes, not overlapping src;
 * dst->layout is ignored on entry and set to AWQ_LAYOUT_PREPARED once the
 * work is enqueued. Asynchronous on `stream`; bit-exact.
 */
AWQ_API awq_status awq_moe_prepare_weights(const awq_moe_shape *shape, const awq_moe_weights *src,
                                           awq_moe_weights *dst, void *stream);

/*
 * awq_prepare_compact -- 4-byte metadata records -> 3-byte records.
 * Source: #522, Default switch (the load-time preparation op that converts a
 * bank to the compact layout; both layouts decode to identical weights) and
 * Addendum, Layout-level capacity (1 byte saved per record).
 * meta4: u8[n_records][4] (device), meta3: u8[n_records][3] (device, written);
 * record r of meta3 is bytes 0..2 of record r of meta4. The buffers must not
 * overlap. n_records >= 0 (0 launches nothing). Bit-exact.
 */
AWQ_API awq_status awq_prepare_compact(const uint8_t *meta4, uint8_t *meta3, int64_t n_records,
                               void *stream);

/*
 * awq_moe_route -- routing metadata of one layer call (step a).
 * Source: #520, Purpose (multi-row active-expert segments, offsets-based
 * scheduling) and Implementation (active_expert_offsets and
 * active_expert_ids are mutated outputs of the op).
 * Inputs:  topk_ids i32[M][k] (device).
 * Outputs (device, S = M*k entries each, caller-allocated):
 *   active_expert_ids     i32[S]   distinct experts ascending; entries >= A are -1
 *   active_expert_offsets i32[S+1] row segment a is [off[a], off[a+1]); entries > A are S
 *   sorted_slots          i32[S]   slots sorted by (expert, slot)
 *   num_active            i32[1]   A
 * Bit-exact and deterministic. An id outside [0, E) sets AWQ_ERR_BAD_EXPERT_ID
 * in dev_status; such slots are left out of every segment.
 */
AWQ_API awq_status awq_moe_route(const int32_t *topk_ids, int32_t M, const awq_moe_shape *shape,
                         int32_t *active_expert_ids, int32_t *active_expert_offsets,
                         int32_t *sorted_slots, int32_t *num_active, int32_t *dev_status,
                         void *stream);

/*
 * awq_moe_w13_swiglu -- grouped W13 GEMM with fused SwiGLU (step b), one launch
 * over all active-expert segments.
 * Source: #520, Purpose (W13 K2560/N320, active-stage op called once per stage
 * instead of once per segment) and Implementation (offsets fast path);
 * #522, Operator results ("W13 + SwiGLU").
 * For every segment a (expert e = active_expert_ids[a]) and row r of it
 * (slot s = sorted_slots[r], token t = s / k):
 *   g = x[t] W13_e[:, 0:I], u = x[t] W13_e[:, I:2I], h[r] = silu(g) * u,
 * accumulated in fp32 and rounded once to fp16. Routing arrays are the outputs
 * of awq_moe_route (device). h: fp16[M*k][I] (device, written; rows past the
 * last segment untouched). Deterministic run to run.
 * Up to AWQ_W2_STAGE_MAX_TOKENS tokens the warp-level MMA kernel runs (exact
 * (q - zero) products, the scale applied in fp32 per group); above it the
 * tcgen05 kernel of the prefill path, whose tensor-core operands are the
 * weights (q - zero) * scale rounded once to fp16 (same tolerance).
 */
AWQ_API awq_status awq_moe_w13_swiglu(const uint16_t *x, int32_t M, const awq_moe_shape *shape,
                              const awq_moe_weights *weights,
                              const int32_t *active_expert_ids,
                              const int32_t *active_expert_offsets,
                              const int32_t *sorted_slots, const int32_t *num_active,
                              uint16_t *h, int32_t *dev_status, void *stream);

/*
 * awq_moe_w2_reduce -- grouped W2 GEMM with the router-weighted top-k
 * reduction (step c), one launch over all active-expert segments.
 * Source: #520, Purpose (W2 K160/N2560) and Implementation (grouped-active
 * exact W2 reduction).
 *   out[t][c] = sum over slots s of token t of topk_weights[s] * (h[row(s)] W2_{e(s)})[c]
 * h: fp16[M*k][I] in sorted-slot order (as written by awq_moe_w13_swiglu),
 * topk_weights f32[M][k]; out fp16[M][H] (written; every element of the M
 * rows is written, tokens with no valid slot get 0). fp32 accumulation,
 * one rounding to fp16. Deterministic run to run. M <= AWQ_W2_STAGE_MAX_TOKENS
 * (else AWQ_ERR_UNSUPPORTED_SHAPE): larger batches go through the layer call,
 * whose workspace holds the per-slot products of the tensor-core W2.
 */
AWQ_API awq_status awq_moe_w2_reduce(const uint16_t *h, const float *topk_weights, int32_t M,
                             const awq_moe_shape *shape, const awq_moe_weights *weights,
                             const int32_t *active_expert_ids,
                             const int32_t *active_expert_offsets,
                             const int32_t *sorted_slots, const int32_t *num_active,
                             uint16_t *out, int32_t *dev_status, void *stream);

/* Execution path of awq_moe_layer_ex. */
typedef enum {
    AWQ_PATH_AUTO = 0,    /* per call shape, the path measured faster on GB300:
                             sliced at M = 2 and at M = 1 with intermediate 160,
                             fused at other M <= 16, hybrid above (NVFP4 banks:
                             fused up to 16 tokens, hybrid above) */
    AWQ_PATH_FUSED = 1,   /* one persistent launch, W2 after a grid-wide hand-over of
                             the W13 results (M <= 16; 80..256 multiprocessors;
                             int4 and NVFP4 banks) */
    AWQ_PATH_STAGED = 2,  /* route, W13 + SwiGLU and W2 launches
                             (M <= AWQ_W2_STAGE_MAX_TOKENS) */
    AWQ_PATH_SLICED = 3,  /* one persistent launch, W2 sliced along K with each CTA's
                             own W13 columns, one grid-wide sum of partial outputs
                             (M <= 8, M * top_k <= multiprocessors, 80..256 of them) */
    AWQ_PATH_PREFILL = 4, /* tensor-core grouped GEMMs (tcgen05): route, W13 + SwiGLU,
                             W2 into per-slot fp32 products in the workspace, and a
                             per-token sum of the products in slot order (any M) */
    AWQ_PATH_HYBRID = 5   /* route, the W13 + SwiGLU stage kernel (h and its residue
                             plane), then the prefill path's tensor-core W2 and
                             per-token sum (any M; int4 and NVFP4 banks) */
} awq_path;

typedef struct {
    uint64_t timeout_ns;  /* limit of each device-side wait; 0 = default (1 s) */
    int32_t path;         /* awq_path */
    int32_t debug_flags;  /* 0 in normal use; bit 0 makes one bounded wait run out
                             (a test of the AWQ_ERR_DEVICE_TIMEOUT path): on the fused
                             path one finished W13 piece is never announced, on the
                             sliced path CTA 0 reaches the grid barrier only after
                             twice the wait limit */
    uint64_t *trace;      /* NULL in normal use (tracing/profiling). Sliced path: a
                             device buffer of grid x AWQ_TRACE_POINTS uint64; CTA c
                             writes the %globaltimer (ns) of each phase point p of
                             the call at trace[c * AWQ_TRACE_POINTS + p]. Prefill
                             path: 6 uint64 that the caller sets to (UINT64_MAX, 0)
                             pairs; launch k (0 W13, 1 W2, 2 per-token sum) lowers
                             trace[2k] to its earliest CTA start (after its wait
                             for the previous launch) and raises trace[2k+1] to
                             its latest CTA end. Other paths ignore it. */
} awq_moe_options;

/* Phase points of awq_moe_options.trace (sliced path): 0 kernel start,
 * 1 predecessor done (programmatic-dependency wait passed), 2 routing and
 * work list ready, 3 first W13 piece in shared memory, 4 last W13 piece
 * consumed, 5 last W2 unit consumed, 6 partial output written, 7 grid
 * barrier passed, 8 output written, 9 last epilogue finished. */
#define AWQ_TRACE_POINTS 16

/*
 * awq_moe_layer -- the whole expert stage of one layer call: route, W13 +
 * SwiGLU, W2 + weighted reduction.
 * Source: #520, Purpose and Implementation; #12, Purpose and stack (physical
 * M=1: fp16 (1, 2560) hidden state, int32 (1, 10) ids, fp32 router weights).
 * x fp16[M][H], topk_ids i32[M][k], topk_weights f32[M][k], out fp16[M][H]
 * (all device). workspace: device scratch of at least
 * awq_moe_workspace_bytes(shape, M) bytes, 256-byte aligned, owned by the
 * caller. It holds the routing arrays, intermediate activations, cross-CTA
 * partial sums and arrival counters. It must be zero-filled once before its
 * first use; after that every call, one that reported AWQ_ERR_DEVICE_TIMEOUT
 * included, leaves it ready for the next call on the same device, so it is
 * reused without clearing (its counter region does not return to zero: two
 * counter sets alternate from call to call). It must not be used by two calls
 * that can run at the same time. For M <= 16 the stage runs as ONE
 * persistent launch (one CTA per multiprocessor); above that as the hybrid
 * path (route, the W13 + SwiGLU stage kernel, tensor-core W2 products, a
 * per-token sum), up to AWQ_MAX_TOKENS. awq_moe_layer_ex selects any other
 * path (AWQ_PATH_*). All give results within the same tolerance.
 * The persistent launches are cooperative: every CTA (one per multiprocessor)
 * must be resident at once, because CTAs wait on each other (bounded waits).
 * If other work on the device keeps multiprocessors busy, the launch waits
 * for them or fails with AWQ_ERR_CUDA; it never runs partly resident.
 */
AWQ_API awq_status awq_moe_layer(const uint16_t *x, const int32_t *topk_ids, const float *topk_weights,
                         int32_t M, const awq_moe_shape *shape, const awq_moe_weights *weights,
                         uint16_t *out, void *workspace, size_t ws_bytes, int32_t *dev_status,
                         void *stream);

/*
 * awq_moe_layer_ex -- awq_moe_layer with explicit options (opts may be NULL:
 * same as awq_moe_layer). AWQ_PATH_FUSED with M > 16 or an unsuitable device
 * returns AWQ_ERR_UNSUPPORTED_SHAPE.
 */
AWQ_API awq_status awq_moe_layer_ex(const uint16_t *x, const int32_t *topk_ids,
                                    const float *topk_weights, int32_t M,
                                    const awq_moe_shape *shape, const awq_moe_weights *weights,
                                    uint16_t *out, void *workspace, size_t ws_bytes,
                                    int32_t *dev_status, const awq_moe_options *opts,
                                    void *stream);

/*
 * awq_moe_router_topk -- the stage's routing inputs from router logits.
 * Source: #12, Purpose and stack (the stage takes int32 top-10 ids and fp32
 * router weights) and its quality section (expert membership follows the
 * router scores); the router is softmax, top-k, renormalised.
 * For every token t: softmax of logits[t][0..E), the top_k experts by
 * probability with ties to the lower id (in that order), and their
 * probabilities renormalised over the chosen experts.
 * logits f32[M][E] (device, finite values); topk_ids i32[M][k] and
 * topk_weights f32[M][k] (device, written). The choice is taken on the fp32
 * logits (softmax is increasing), so the ids are those of an exact softmax;
 * the weights are computed in fp32 (relative error below 1e-6). One launch,
 * no workspace, deterministic. The router takes num_experts = 512 and
 * top_k <= 32 (else AWQ_ERR_UNSUPPORTED_SHAPE). Errors: host-side only, as
 * the other calls (shape, M in [0, AWQ_MAX_TOKENS], null or misaligned
 * pointers).
 */
AWQ_API awq_status awq_moe_router_topk(const float *logits, int32_t M, const awq_moe_shape *shape,
                                       int32_t *topk_ids, float *topk_weights, void *stream);

/*
 * awq_moe_layer_logits -- awq_moe_layer_ex starting from router logits: the
 * router of awq_moe_router_topk, then the expert stage on its choice.
 * logits f32[M][E] (device); topk_ids i32[M][k] and topk_weights f32[M][k]
 * (device, written with the choice the stage used). For M <= 16 on the fused
 * path the router runs in the persistent kernel's prologue (still one
 * launch); otherwise it is one more launch before the three. Shape limits of
 * the router as awq_moe_router_topk. Other arguments, workspace rules,
 * results and errors as awq_moe_layer_ex (opts may be NULL).
 */
AWQ_API awq_status awq_moe_layer_logits(const uint16_t *x, const float *logits, int32_t M,
                                        const awq_moe_shape *shape, const awq_moe_weights *weights,
                                        uint16_t *out, int32_t *topk_ids, float *topk_weights,
                                        void *workspace, size_t ws_bytes, int32_t *dev_status,
                                        const awq_moe_options *opts, void *stream);

/*
 * awq_moe_layer_static -- awq_moe_layer without a workspace argument, for
 * callers that have no device allocator to provide one (a plain C host, a
 * plugin whose process plans all device memory up front). The pages have no
 * counterpart: it exists only for such callers.
 * Scratch is a fixed array of AWQ_STATIC_SCRATCH_BYTES in the library's own
 * device memory (one per device, created with the module; nothing is
 * allocated or freed by this call). The stage runs as the three launches
 * (route, W13 + SwiGLU, W2 + reduction), whose kernels rewrite every scratch
 * byte they read: nothing has to start at zero. Results are within the same
 * tolerance as awq_moe_layer.
 * Limit: a call needs 256-byte-rounded room for its routing arrays and its
 * fp16 activations (about 2 * M * top_k * inter bytes); a call that does not
 * fit is rejected with AWQ_ERR_WORKSPACE_TOO_SMALL before anything is
 * launched (every M * top_k <= 1024 fits at inter 640). M is limited to
 * AWQ_W2_STAGE_MAX_TOKENS (else AWQ_ERR_UNSUPPORTED_SHAPE).
 * Every call looks up the array's device address in the current device's
 * context (cudaGetSymbolAddress, no allocation); the first call on a device
 * also loads the library's module there (set-up): make it before any stream
 * capture begins. All calls on a device share the
 * array: calls that can run at the same time (other streams, unordered host
 * threads) race on it and give undefined results.
 * Arguments and errors otherwise as awq_moe_layer.
 */
#define AWQ_STATIC_SCRATCH_BYTES (2u << 20)
AWQ_API awq_status awq_moe_layer_static(const uint16_t *x, const int32_t *topk_ids,
                                        const float *topk_weights, int32_t M,
                                        const awq_moe_shape *shape, const awq_moe_weights *weights,
                                        uint16_t *out, int32_t *dev_status, void *stream);

/*
 * awq_moe_latency_floor -- measurement helper, not part of the stage. The
 * dependency chain of the persistent layer call with none of its arithmetic,
 * so that a layer call's time can be read against what that chain costs:
 * wait for the previous launch in the stream; load topk_ids (i32[M][k]) and
 * find the distinct active experts; read every byte of their prepared banks
 * once (bulk copies into discarded shared memory, spread over one CTA per
 * multiprocessor); one grid barrier; write out fp16[M][H] as zeros. Same
 * launch form as the persistent layer kernels (cooperative, programmatic
 * dependent launch) and the same workspace rules (it advances the grid
 * barrier counter of the workspace's counter region). M 0..16; banks
 * prepared; ids outside [0, E) set AWQ_ERR_BAD_EXPERT_ID and are skipped.
 */
AWQ_API awq_status awq_moe_latency_floor(const int32_t *topk_ids, int32_t M, const awq_moe_shape *shape,
                                         const awq_moe_weights *weights, uint16_t *out, void *workspace,
                                         size_t ws_bytes, int32_t *dev_status, void *stream);

/* Workspace bytes awq_moe_layer needs for up to M_max tokens, valid for every
 * M <= M_max and both paths (0 for an invalid shape or M_max). Host-only, no
 * CUDA call. */
AWQ_API size_t awq_moe_workspace_bytes(const awq_moe_shape *shape, int32_t M_max);

/* Static, NUL-terminated description of a status code. Host-only. */
AWQ_API const char *awq_status_string(awq_status status);

#ifdef __cplusplus
}
#endif
#endif /* AWQ_MOE_H */
