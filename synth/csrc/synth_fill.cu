// Device-side fill of synthetic expert banks with the same counter-based
// generator as synth/__init__.py (SplitMix64 output function over a
// counter stream per (seed, layer, tensor, expert)), so multi-GB banks never
// cross PCIe. Holds no arithmetic of the expert stage itself.
#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kScaleBase = 2199023256ull;   // round(0.002 * 2^40)
constexpr uint64_t kScaleStep = 18874ull;        // round(0.018 * 2^20)

__device__ __forceinline__ uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t stream_key(uint64_t seed, uint64_t layer, uint64_t tensor,
                                               uint64_t expert)
{
    uint64_t k = mix64(seed + kGamma);
    k = mix64(k ^ ((layer + 1) * kGamma));
    k = mix64(k ^ ((tensor + 1) * kGamma));
    k = mix64(k ^ ((expert + 1) * kGamma));
    return k;
}

// fp16 bits of n * 2^-40 for n in [2^31, 2^35), round to nearest even, with
// integer operations only (the host generator does the same steps).
__device__ __forceinline__ uint16_t scale_bits(uint64_t n)
{
    const int e = 63 - __clzll(static_cast<long long>(n));   // n in [2^e, 2^(e+1))
    const int sh = e - 10;
    uint64_t m = n >> sh;
    const uint64_t rem = n & ((1ull << sh) - 1);
    const uint64_t half = 1ull << (sh - 1);
    if (rem > half || (rem == half && (m & 1))) ++m;
    int ee = e;
    if (m == 2048) {
        m = 1024;
        ++ee;
    }
    return static_cast<uint16_t>(((ee - 40 + 15) << 10) | static_cast<int>(m - 1024));
}

// grid (x: chunks of 2 words per thread, y: expert)
__global__ void fill_q_kernel(uint32_t *dst, int64_t words, int32_t expert0, uint64_t seed,
                              int32_t layer, int32_t tensor)
{
    const int e = blockIdx.y;
    const uint64_t key = stream_key(seed, layer, tensor, expert0 + e);
    uint32_t *base = dst + static_cast<int64_t>(e) * words;
    const int64_t pairs = (words + 1) / 2;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < pairs;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint64_t d = mix64(key + static_cast<uint64_t>(i + 1) * kGamma);
        const int64_t w = 2 * i;
        if (w + 1 < words) {
            reinterpret_cast<uint2 *>(base)[i] = make_uint2(static_cast<uint32_t>(d),
                                                            static_cast<uint32_t>(d >> 32));
        } else {
            base[w] = static_cast<uint32_t>(d);
        }
    }
}

__global__ void fill_meta_kernel(uint8_t *dst, int64_t records, int32_t meta_bytes,
                                 int32_t expert0, uint64_t seed, int32_t layer, int32_t tensor)
{
    const int e = blockIdx.y;
    const uint64_t key = stream_key(seed, layer, tensor, expert0 + e);
    uint8_t *base = dst + static_cast<int64_t>(e) * records * meta_bytes;
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; r < records;
         r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint64_t d = mix64(key + static_cast<uint64_t>(r + 1) * kGamma);
        if (meta_bytes == 1) {   // NVFP4 E4M3 block-scale code: exponent U{0..3}, mantissa U{0..7}
            base[r] = static_cast<uint8_t>((((d >> 32) & 3) << 3) | ((d >> 40) & 7));
            continue;
        }
        const uint32_t zero = static_cast<uint32_t>(d & 0xF);
        const uint64_t r20 = (d >> 32) & 0xFFFFF;
        const uint16_t bits = scale_bits(kScaleBase + r20 * kScaleStep);
        uint8_t *rec = base + r * meta_bytes;
        rec[0] = static_cast<uint8_t>(bits & 0xFF);
        rec[1] = static_cast<uint8_t>(bits >> 8);
        rec[2] = static_cast<uint8_t>(zero);
        if (meta_bytes == 4) rec[3] = 0;
    }
}

}  // namespace

extern "C" {

__attribute__((visibility("default"))) int awq_synth_fill_q(uint32_t *dst, int64_t words_per_expert,
                                                            int32_t expert0, int32_t n_experts,
                                                            uint64_t seed, int32_t layer,
                                                            int32_t tensor, void *stream)
{
    if (!dst || words_per_expert <= 0 || n_experts <= 0 || n_experts > 65535) return 1;
    const int64_t pairs = (words_per_expert + 1) / 2;
    const int blocks = static_cast<int>((pairs + 255) / 256 < 1024 ? (pairs + 255) / 256 : 1024);
    fill_q_kernel<<<dim3(blocks, n_experts), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        dst, words_per_expert, expert0, seed, layer, tensor);
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

__attribute__((visibility("default"))) int awq_synth_fill_meta(uint8_t *dst,
                                                               int64_t records_per_expert,
                                                               int32_t meta_bytes, int32_t expert0,
                                                               int32_t n_experts, uint64_t seed,
                                                               int32_t layer, int32_t tensor,
                                                               void *stream)
{
    if (!dst || records_per_expert <= 0 || n_experts <= 0 || n_experts > 65535 ||
        (meta_bytes != 1 && meta_bytes != 3 && meta_bytes != 4))
        return 1;
    const int blocks = static_cast<int>(
        (records_per_expert + 255) / 256 < 1024 ? (records_per_expert + 255) / 256 : 1024);
    fill_meta_kernel<<<dim3(blocks, n_experts), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        dst, records_per_expert, meta_bytes, expert0, seed, layer, tensor);
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

}  // extern "C"
