/*
 * CPU oracle of the AWQ int4 MoE expert stage -- TEST INFRASTRUCTURE ONLY.
 * Declarations of oracle/awq_moe_oracle.c; no other part of the repository
 * includes this header. All floating-point results are FP64.
 */
#ifndef AWQ_MOE_ORACLE_H
#define AWQ_MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { AWQO_OK = 0, AWQO_BAD_ARG = 1, AWQO_BAD_EXPERT_ID = 6, AWQO_NO_MEMORY = 7 };

/* fp16 bit pattern -> double (exact). */
double awqo_half_to_double(uint16_t h);

/* Decode one packed matrix to W[K][N] (row k = input index, column n = output):
 * q u32[K/8][N] with row k in nibble k%8 of word (k/8, n); meta u8[K/group][N][meta_bytes]. */
int awqo_decode_matrix(const uint32_t *q, const uint8_t *meta, int meta_bytes,
                       int K, int N, int group, double *W);

/* FP4 E2M1 code (low 4 bits) and FP8 E4M3 code -> double (exact). */
double awqo_e2m1_to_double(uint8_t code);
double awqo_e4m3_to_double(uint8_t code);

/* Decode one NVFP4 matrix to W[K][N]: q u32[K/8][N] of E2M1 codes (nibble k%8
 * of word (k/8, n)), scales u8[K/16][N] of E4M3 codes, one fp32 global:
 * w = e2m1 * e4m3 * global. */
int awqo_decode_nvfp4(const uint32_t *q, const uint8_t *scales, float global, int K, int N, double *W);

/* 4-byte records -> 3-byte records (byte 3 dropped). */
void awqo_prepare_compact(const uint8_t *meta4, uint8_t *meta3, int64_t n_records);

/* Group slots s = t*top_k + j by expert: active ids ascending (rest -1),
 * CSR offsets (entries past the last active expert = S), slots sorted by
 * (expert, slot). Arrays have S = M*top_k entries (offsets S+1). */
int awqo_route(const int32_t *topk_ids, int M, int top_k, int num_experts,
               int32_t *active_ids, int32_t *offsets, int32_t *sorted_slots,
               int32_t *num_active);

/* h_slot[S][I] (slot order) = silu(x W13[:, :I]) * (x W13[:, I:]). Per-expert
 * pointer arrays of length num_experts; unused experts may be NULL. */
int awqo_w13_swiglu(const uint16_t *x, const int32_t *topk_ids, int M, int top_k,
                    int num_experts, int hidden, int inter, int group, int meta_bytes,
                    const uint32_t *const *w13_q, const uint8_t *const *w13_meta,
                    double *h_slot);

/* out[M][H] = sum_j w[t][j] * (h_slot[t*k+j] W2_{e}), from a given h (slot order). */
int awqo_w2_reduce(const double *h_slot, const int32_t *topk_ids, const float *topk_weights,
                   int M, int top_k, int num_experts, int hidden, int inter, int group,
                   int meta_bytes, const uint32_t *const *w2_q, const uint8_t *const *w2_meta,
                   double *out);

/* The whole layer: W13 + SwiGLU then W2 + weighted reduction, h kept in FP64. */
int awqo_moe_layer(const uint16_t *x, const int32_t *topk_ids, const float *topk_weights,
                   int M, int top_k, int num_experts, int hidden, int inter, int group,
                   int meta_bytes, const uint32_t *const *w13_q, const uint8_t *const *w13_meta,
                   const uint32_t *const *w2_q, const uint8_t *const *w2_meta,
                   double *h_slot, double *out);

/* The whole layer with NVFP4 weights: as awqo_moe_layer, each expert's W13
 * and W2 decoded by awqo_decode_nvfp4 with global[2e] (W13) and global[2e+1]
 * (W2). Scales u8[K/16][N] per expert. */
int awqo_moe_layer_nvfp4(const uint16_t *x, const int32_t *topk_ids, const float *topk_weights, int M,
                         int top_k, int num_experts, int hidden, int inter,
                         const uint32_t *const *w13_q, const uint8_t *const *w13_scales,
                         const uint32_t *const *w2_q, const uint8_t *const *w2_scales, const float *global,
                         double *h_slot, double *out);

/* Router: per token, softmax of logits[t][0..E) (max-subtracted), the top_k
 * experts by probability with ties to the lower id, in that order, and their
 * probabilities renormalised over the chosen experts. */
int awqo_router_topk(const float *logits, int M, int num_experts, int top_k,
                     int32_t *topk_ids, double *topk_weights);

#ifdef __cplusplus
}
#endif
#endif
