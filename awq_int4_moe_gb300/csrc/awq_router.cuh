// Router from logits: per token the top_k experts by softmax probability,
// ties to the lower id, and their probabilities renormalised over the chosen
// experts -- the stage's int32 top-10 ids and fp32 router weights (1Cat-vLLM
// #12 "Add opt-in native-g32 AWQ QPN M1 dispatch", Purpose and stack; its
// quality section: expert membership follows the router scores).
//
// Softmax is increasing in the logit, so the choice is made on the fp32
// logits themselves (no exponential, no rounding); the renormalised weights
// are the softmax restricted to the chosen logits:
//   w_j = exp(l_j - l_max) / sum_i exp(l_i - l_max),  i, j over the chosen.
#pragma once

#include <cstdint>

namespace awq {

// Order-preserving integer key of a float (larger float -> larger key; -0
// is taken as +0 so that equal values tie).
__device__ __forceinline__ uint32_t order_key(float f)
{
    uint32_t b = __float_as_uint(f);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One warp routes one token of E = 32 * PER_LANE experts; lane l holds
// experts i * 32 + l. Lanes j < top_k write ids[j] and w[j]. Logits must be
// finite. top_k <= 32. Each choice is two warp reductions: the largest key,
// then the lowest id holding it.
template <int PER_LANE>   // a power of two
__device__ __forceinline__ void warp_router_topk(const float *lg, int top_k, int lane, int32_t *ids,
                                                 float *w)
{
    uint32_t key[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) key[i] = order_key(lg[i * 32 + lane]);
    uint32_t taken = 0;                    // bit i: expert i * 32 + lane chosen
    uint32_t my_key = 0;                   // lane j: key of the j-th choice
    int my_id = 0;
    for (int j = 0; j < top_k; ++j) {
        // the lane's best remaining expert (larger key, then lower id): a
        // pairwise tree over the keys, chosen ones masked to 0 (below the key
        // of every finite float), the lower index kept on ties
        uint32_t tk[PER_LANE];
        int ti[PER_LANE];
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            tk[i] = (taken >> i & 1u) ? 0u : key[i];
            ti[i] = i;
        }
#pragma unroll
        for (int width = PER_LANE / 2; width >= 1; width /= 2)
#pragma unroll
            for (int i = 0; i < width; ++i) {
                const bool hi = tk[2 * i + 1] > tk[2 * i];
                tk[i] = hi ? tk[2 * i + 1] : tk[2 * i];
                ti[i] = hi ? ti[2 * i + 1] : ti[2 * i];
            }
        const uint32_t bk = tk[0];
        const int bi = ti[0];
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t cand = bk == kmax ? static_cast<uint32_t>(bi * 32 + lane) : 0xFFFFFFFFu;
        const uint32_t id = __reduce_min_sync(0xffffffffu, cand);
        if ((id & 31u) == static_cast<uint32_t>(lane)) taken |= 1u << (id >> 5);
        if (lane == j) {
            my_key = kmax;
            my_id = static_cast<int>(id);
        }
    }
    // the first choice holds the largest logit
    const float my_v = key_value(my_key);
    const float lmax = __shfl_sync(0xffffffffu, my_v, 0);
    const float e = lane < top_k ? expf(my_v - lmax) : 0.f;
    float sum = e;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane < top_k) {
        ids[lane] = my_id;
        w[lane] = e / sum;
    }
}

}  // namespace awq
