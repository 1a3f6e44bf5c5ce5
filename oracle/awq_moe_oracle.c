/*
 * CPU oracle of the AWQ int4 MoE expert stage -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg may load this file's library. It shares no code, header, table or
 * helper with the CUDA library; neither includes or links the other.
 *
 * It is the plain definition of what the stage computes, in FP64, with no
 * blocking, fusion or reordering beyond what the definition states:
 *
 *   decode   w[k][n] = (q[k][n] - zero[k/G][n]) * scale[k/G][n]
 *            (1Cat-vLLM #520 "Narrow Qwen3.8 AWQ active grouped decode",
 *             Purpose: group 32, W13 K2560/N320, W2 K160/N2560;
 *             1Cat-vLLM #522 "Coalesce AWQ QPN W13 compact metadata loads and
 *             enable compact metadata by default", Purpose: a record is
 *             {FP16 scale, u8 zero}; Default switch: the 3-byte and 4-byte
 *             layouts decode to identical weights)
 *   route    the (token, top-k slot) pairs grouped by expert: distinct active
 *            expert ids ascending and CSR offsets of their row segments
 *            (#520, Purpose and Implementation: active_expert_ids /
 *             active_expert_offsets, offsets-based scheduling)
 *   W13      g = x W13[:, 0:I], u = x W13[:, I:2I], h = silu(g) * u
 *            (#520 Purpose: W13 K2560/N320; #522 Operator results:
 *             "W13 + SwiGLU")
 *   W2       out[t] = sum_j w[t][j] * (h[t,j] W2_{e(t,j)}), j in order
 *            (#520 Implementation: grouped-active exact W2 reduction)
 *   router   the stage's inputs from router logits: softmax over the E
 *            experts, the top_k most probable (ties to the lower id), their
 *            probabilities renormalised to sum 1 (1Cat-vLLM #12 "Add opt-in
 *            native-g32 AWQ QPN M1 dispatch", Purpose and stack: int32 top-10
 *            ids and fp32 router weights feed the stage; its quality section:
 *            expert membership follows the router scores)
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes): nibble j of packed word (i, n) is row 8i+j of column n, LSB first;
 * q is stored [K/8][N] and metadata [K/G][N][record], column fastest; record
 * bytes 0-1 are the fp16 scale (little-endian), byte 2 the zero, byte 3 (4-byte
 * layout) padding; silu(g) = g / (1 + exp(-g)); the router weight multiplies
 * each slot's W2 output once; the router's softmax is max-subtracted and its
 * top-k order is (probability descending, expert id ascending).
 *
 * NVFP4 weights (the second weight format; the pages name a native NVFP4
 * kernel only as a comparison column -- #520 Results, #522 Operator results --
 * and do not define the format, so the published NVFP4 definition is taken):
 * each 4-bit code is an FP4 E2M1 value (sign, 2 exponent bits with bias 1, 1
 * mantissa bit: +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}); every block of 16
 * consecutive K elements of a column shares one FP8 E4M3 scale (sign, 4
 * exponent bits with bias 7, 3 mantissa bits; subnormals m * 2^-9; maximum
 * 448; S.1111.111 is NaN); each expert's matrix has one fp32 global scale:
 *   w[k][n] = e2m1(q[k][n]) * e4m3(scale[k/16][n]) * global.
 * Codes are packed like the int4 banks (nibble j of word (i, n) is row 8i+j)
 * and scales are stored [K/16][N], column fastest.
 *
 * Pins: every function here is checked by the "not gpu" tests against facts
 * that do not come from this file (hand-built cases, library routines,
 * invariants, brute force and the sizes the pages print).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "awq_moe_oracle.h"

/* IEEE 754 binary16 -> double, from the format's definition. */
double awqo_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1F;
    int frac = h & 0x3FF;
    double v;
    if (ex == 0)
        v = ldexp((double)frac, -24);                 /* subnormal / zero */
    else if (ex == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), ex - 25);    /* (1 + f/1024) 2^(e-15) */
    return sign ? -v : v;
}

/* One metadata record -> (scale, zero). Both layouts keep the scale in bytes
 * 0-1 and the zero in byte 2; they are decoded by separate functions so that
 * the 3-byte / 4-byte equivalence test compares two independent readers. */
static void record4(const uint8_t *meta, int64_t rec, double *scale, int *zero)
{
    const uint8_t *r = meta + 4 * rec;
    *scale = awqo_half_to_double((uint16_t)(r[0] | (r[1] << 8)));
    *zero = r[2];
}

static void record3(const uint8_t *meta, int64_t rec, double *scale, int *zero)
{
    const uint8_t *r = meta + 3 * rec;
    *scale = awqo_half_to_double((uint16_t)(r[0] | (r[1] << 8)));
    *zero = r[2];
}

int awqo_decode_matrix(const uint32_t *q, const uint8_t *meta, int meta_bytes,
                       int K, int N, int group, double *W)
{
    if (!q || !meta || !W || K <= 0 || N <= 0 || group <= 0 || K % 8 || K % group)
        return 1;
    if (meta_bytes != 3 && meta_bytes != 4)
        return 1;
    for (int k = 0; k < K; ++k) {
        for (int n = 0; n < N; ++n) {
            uint32_t word = q[(int64_t)(k / 8) * N + n];
            int nib = (int)((word >> (4 * (k % 8))) & 0xFu);
            int64_t rec = (int64_t)(k / group) * N + n;
            double scale;
            int zero;
            if (meta_bytes == 4)
                record4(meta, rec, &scale, &zero);
            else
                record3(meta, rec, &scale, &zero);
            W[(int64_t)k * N + n] = (double)(nib - zero) * scale;
        }
    }
    return 0;
}

/* FP4 E2M1 code (low 4 bits) -> double, from the format's definition. */
double awqo_e2m1_to_double(uint8_t code)
{
    const int sign = (code >> 3) & 1, ex = (code >> 1) & 3, man = code & 1;
    const double v = ex == 0 ? 0.5 * man : ldexp(1.0 + 0.5 * man, ex - 1);
    return sign ? -v : v;
}

/* FP8 E4M3 code -> double, from the format's definition (no infinities;
 * S.1111.111 is NaN). */
double awqo_e4m3_to_double(uint8_t code)
{
    const int sign = (code >> 7) & 1, ex = (code >> 3) & 0xF, man = code & 7;
    double v;
    if (ex == 15 && man == 7)
        v = NAN;
    else if (ex == 0)
        v = ldexp((double)man, -9);                   /* (m / 8) * 2^(1 - 7) */
    else
        v = ldexp(1.0 + man / 8.0, ex - 7);
    return sign ? -v : v;
}

int awqo_decode_nvfp4(const uint32_t *q, const uint8_t *scales, float global, int K, int N, double *W)
{
    if (!q || !scales || !W || K <= 0 || N <= 0 || K % 16) return 1;
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n) {
            const uint32_t word = q[(int64_t)(k / 8) * N + n];
            const uint8_t code = (uint8_t)((word >> (4 * (k % 8))) & 0xFu);
            const double s = awqo_e4m3_to_double(scales[(int64_t)(k / 16) * N + n]);
            W[(int64_t)k * N + n] = awqo_e2m1_to_double(code) * s * (double)global;
        }
    return 0;
}

void awqo_prepare_compact(const uint8_t *meta4, uint8_t *meta3, int64_t n_records)
{
    for (int64_t r = 0; r < n_records; ++r) {
        meta3[3 * r + 0] = meta4[4 * r + 0];
        meta3[3 * r + 1] = meta4[4 * r + 1];
        meta3[3 * r + 2] = meta4[4 * r + 2];
    }
}

/* ------------------------------------------------------------------ route */

typedef struct { int32_t expert, slot; } pair_t;

static int pair_cmp(const void *a, const void *b)
{
    const pair_t *x = (const pair_t *)a, *y = (const pair_t *)b;
    if (x->expert != y->expert) return x->expert < y->expert ? -1 : 1;
    return (x->slot > y->slot) - (x->slot < y->slot);
}

int awqo_route(const int32_t *topk_ids, int M, int top_k, int num_experts,
               int32_t *active_ids, int32_t *offsets, int32_t *sorted_slots,
               int32_t *num_active)
{
    int S = M * top_k;
    for (int s = 0; s < S; ++s)
        if (topk_ids[s] < 0 || topk_ids[s] >= num_experts)
            return AWQO_BAD_EXPERT_ID;
    pair_t *p = (pair_t *)malloc(sizeof(pair_t) * (size_t)(S > 0 ? S : 1));
    if (!p) return AWQO_NO_MEMORY;
    for (int s = 0; s < S; ++s) {
        p[s].expert = topk_ids[s];
        p[s].slot = s;                       /* slot s = t * top_k + j */
    }
    qsort(p, (size_t)S, sizeof(pair_t), pair_cmp);
    int A = 0;
    for (int i = 0; i < S; ++i) {
        sorted_slots[i] = p[i].slot;
        if (i == 0 || p[i].expert != p[i - 1].expert) {
            active_ids[A] = p[i].expert;
            offsets[A] = i;
            ++A;
        }
    }
    for (int i = A; i < S; ++i) active_ids[i] = -1;
    for (int i = A; i <= S; ++i) offsets[i] = S;
    *num_active = A;
    free(p);
    return AWQO_OK;
}

/* ----------------------------------------------------------- expert stage */

static double silu(double g) { return g / (1.0 + exp(-g)); }

static int check_layer_args(int M, int top_k, int num_experts, int hidden, int inter,
                            int group, int meta_bytes)
{
    if (M < 0 || top_k <= 0 || num_experts <= 0 || hidden <= 0 || inter <= 0 || group <= 0)
        return AWQO_BAD_ARG;
    if (hidden % 8 || inter % 8 || hidden % group || inter % group)
        return AWQO_BAD_ARG;
    if (meta_bytes != 3 && meta_bytes != 4)
        return AWQO_BAD_ARG;
    return AWQO_OK;
}

/* Decoding of one expert's matrix (K x N) for the stage: the int4 banks with
 * their records, or the NVFP4 banks with their block scales and global. */
typedef struct {
    const uint32_t *const *q;
    const uint8_t *const *meta;
    int meta_bytes, group;       /* int4 banks */
    const float *global;         /* NVFP4 banks: [E][2]; NULL for int4 */
    int which;                   /* 0 W13, 1 W2 (index into global) */
} Bank;

static int decode_bank(const Bank *b, int e, int K, int N, double *W)
{
    if (!b->q[e] || !b->meta[e]) return AWQO_BAD_ARG;
    if (b->global) return awqo_decode_nvfp4(b->q[e], b->meta[e], b->global[2 * e + b->which], K, N, W);
    return awqo_decode_matrix(b->q[e], b->meta[e], b->meta_bytes, K, N, b->group, W) ? AWQO_BAD_ARG : AWQO_OK;
}

static int w13_stage(const uint16_t *x, const int32_t *topk_ids, int M, int top_k, int num_experts, int hidden,
                     int inter, const Bank *bank, double *h_slot)
{
    int rc = AWQO_OK;
    const int S = M * top_k, H = hidden, N = 2 * inter;
    for (int s = 0; s < S; ++s)
        if (topk_ids[s] < 0 || topk_ids[s] >= num_experts) return AWQO_BAD_EXPERT_ID;
    double *W = (double *)malloc(sizeof(double) * (size_t)H * N);
    double *xd = (double *)malloc(sizeof(double) * (size_t)H);
    double *gu = (double *)malloc(sizeof(double) * (size_t)N);
    if (!W || !xd || !gu) { free(W); free(xd); free(gu); return AWQO_NO_MEMORY; }
    for (int e = 0; e < num_experts; ++e) {
        int used = 0;
        for (int s = 0; s < S && !used; ++s) used = topk_ids[s] == e;
        if (!used) continue;
        if ((rc = decode_bank(bank, e, H, N, W))) break;
        for (int s = 0; s < S; ++s) {
            if (topk_ids[s] != e) continue;
            const int t = s / top_k;
            for (int k = 0; k < H; ++k) xd[k] = awqo_half_to_double(x[(int64_t)t * H + k]);
            /* gu[n] = sum_k x[k] * W13[k][n], accumulated in k order */
            for (int n = 0; n < N; ++n) gu[n] = 0.0;
            for (int k = 0; k < H; ++k)
                for (int n = 0; n < N; ++n)
                    gu[n] += xd[k] * W[(int64_t)k * N + n];
            for (int i = 0; i < inter; ++i)
                h_slot[(int64_t)s * inter + i] = silu(gu[i]) * gu[inter + i];
        }
    }
    free(W);
    free(xd);
    free(gu);
    return rc;
}

int awqo_w13_swiglu(const uint16_t *x, const int32_t *topk_ids, int M, int top_k,
                    int num_experts, int hidden, int inter, int group, int meta_bytes,
                    const uint32_t *const *w13_q, const uint8_t *const *w13_meta,
                    double *h_slot)
{
    int rc = check_layer_args(M, top_k, num_experts, hidden, inter, group, meta_bytes);
    if (rc) return rc;
    const Bank b = {w13_q, w13_meta, meta_bytes, group, NULL, 0};
    return w13_stage(x, topk_ids, M, top_k, num_experts, hidden, inter, &b, h_slot);
}

static int w2_stage(const double *h_slot, const int32_t *topk_ids, const float *topk_weights, int M, int top_k,
                    int num_experts, int hidden, int inter, const Bank *bank, double *out)
{
    int rc = AWQO_OK;
    const int S = M * top_k, H = hidden, I = inter;
    for (int s = 0; s < S; ++s)
        if (topk_ids[s] < 0 || topk_ids[s] >= num_experts) return AWQO_BAD_EXPERT_ID;
    double *W = (double *)malloc(sizeof(double) * (size_t)I * H);
    double *y = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1) * H);
    if (!W || !y) { free(W); free(y); return AWQO_NO_MEMORY; }
    /* y[s][c] = sum_i h[s][i] * W2_{e(s)}[i][c] */
    for (int e = 0; e < num_experts; ++e) {
        int used = 0;
        for (int s = 0; s < S && !used; ++s) used = topk_ids[s] == e;
        if (!used) continue;
        if ((rc = decode_bank(bank, e, I, H, W))) break;
        for (int s = 0; s < S; ++s) {
            if (topk_ids[s] != e) continue;
            double *ys = y + (int64_t)s * H;
            for (int c = 0; c < H; ++c) ys[c] = 0.0;
            for (int i = 0; i < I; ++i)          /* accumulated in i order */
                for (int c = 0; c < H; ++c)
                    ys[c] += h_slot[(int64_t)s * I + i] * W[(int64_t)i * H + c];
        }
    }
    /* out[t][c] = sum_j w[t][j] * y[t*k+j][c], summed in j order */
    if (rc == AWQO_OK) {
        for (int t = 0; t < M; ++t)
            for (int c = 0; c < H; ++c) {
                double acc = 0.0;
                for (int j = 0; j < top_k; ++j)
                    acc += (double)topk_weights[t * top_k + j] * y[(int64_t)(t * top_k + j) * H + c];
                out[(int64_t)t * H + c] = acc;
            }
    }
    free(W);
    free(y);
    return rc;
}

int awqo_w2_reduce(const double *h_slot, const int32_t *topk_ids, const float *topk_weights,
                   int M, int top_k, int num_experts, int hidden, int inter, int group,
                   int meta_bytes, const uint32_t *const *w2_q, const uint8_t *const *w2_meta,
                   double *out)
{
    int rc = check_layer_args(M, top_k, num_experts, hidden, inter, group, meta_bytes);
    if (rc) return rc;
    const Bank b = {w2_q, w2_meta, meta_bytes, group, NULL, 1};
    return w2_stage(h_slot, topk_ids, topk_weights, M, top_k, num_experts, hidden, inter, &b, out);
}

int awqo_moe_layer_nvfp4(const uint16_t *x, const int32_t *topk_ids, const float *topk_weights, int M,
                         int top_k, int num_experts, int hidden, int inter,
                         const uint32_t *const *w13_q, const uint8_t *const *w13_scales,
                         const uint32_t *const *w2_q, const uint8_t *const *w2_scales, const float *global,
                         double *h_slot, double *out)
{
    if (M < 0 || top_k <= 0 || num_experts <= 0 || hidden <= 0 || inter <= 0 || hidden % 16 || inter % 16 ||
        !global)
        return AWQO_BAD_ARG;
    const Bank b13 = {w13_q, w13_scales, 0, 16, global, 0};
    const Bank b2 = {w2_q, w2_scales, 0, 16, global, 1};
    int rc = w13_stage(x, topk_ids, M, top_k, num_experts, hidden, inter, &b13, h_slot);
    if (rc) return rc;
    return w2_stage(h_slot, topk_ids, topk_weights, M, top_k, num_experts, hidden, inter, &b2, out);
}

int awqo_moe_layer(const uint16_t *x, const int32_t *topk_ids, const float *topk_weights,
                   int M, int top_k, int num_experts, int hidden, int inter, int group,
                   int meta_bytes, const uint32_t *const *w13_q, const uint8_t *const *w13_meta,
                   const uint32_t *const *w2_q, const uint8_t *const *w2_meta,
                   double *h_slot, double *out)
{
    int rc = awqo_w13_swiglu(x, topk_ids, M, top_k, num_experts, hidden, inter, group,
                             meta_bytes, w13_q, w13_meta, h_slot);
    if (rc) return rc;
    return awqo_w2_reduce(h_slot, topk_ids, topk_weights, M, top_k, num_experts, hidden,
                          inter, group, meta_bytes, w2_q, w2_meta, out);
}

/* ----------------------------------------------------------------- router */

int awqo_router_topk(const float *logits, int M, int num_experts, int top_k,
                     int32_t *topk_ids, double *topk_weights)
{
    if (M < 0 || num_experts < 1 || top_k < 1 || top_k > num_experts) return AWQO_BAD_ARG;
    double *p = (double *)malloc(sizeof(double) * (size_t)num_experts);
    char *taken = (char *)malloc((size_t)num_experts);
    if (!p || !taken) {
        free(p);
        free(taken);
        return AWQO_NO_MEMORY;
    }
    for (int t = 0; t < M; ++t) {
        const float *l = logits + (int64_t)t * num_experts;
        /* softmax over all experts, max-subtracted */
        double mx = (double)l[0];
        for (int e = 1; e < num_experts; ++e)
            if ((double)l[e] > mx) mx = (double)l[e];
        double z = 0.0;
        for (int e = 0; e < num_experts; ++e) {
            p[e] = exp((double)l[e] - mx);
            z += p[e];
        }
        for (int e = 0; e < num_experts; ++e) p[e] /= z;
        /* top_k by probability, ties to the lower id: k selection passes */
        memset(taken, 0, (size_t)num_experts);
        double sel = 0.0;
        for (int j = 0; j < top_k; ++j) {
            int best = -1;
            for (int e = 0; e < num_experts; ++e)
                if (!taken[e] && (best < 0 || p[e] > p[best])) best = e;
            taken[best] = 1;
            topk_ids[(int64_t)t * top_k + j] = best;
            topk_weights[(int64_t)t * top_k + j] = p[best];
            sel += p[best];
        }
        /* renormalise over the chosen experts */
        for (int j = 0; j < top_k; ++j) topk_weights[(int64_t)t * top_k + j] /= sel;
    }
    free(p);
    free(taken);
    return AWQO_OK;
}
