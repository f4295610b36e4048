// Synthetic device data for the offline search (lora_tune): bf16 values spread
// uniformly over [-scale, scale), from a counter-based integer hash of (seed, index),
// so that a shape's buffers are filled on the device with no host copy.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace lora {

namespace {

__device__ __forceinline__ uint32_t mix32(uint64_t v)
{
    // 64-bit finaliser (xor-shift / multiply rounds), folded to 32 bits
    v ^= v >> 33;
    v *= 0xff51afd7ed558ccdull;
    v ^= v >> 33;
    v *= 0xc4ceb9fe1a85ec53ull;
    v ^= v >> 33;
    return uint32_t(v);
}

__global__ void k_fill_bf16(uint16_t *dst, uint64_t n, uint64_t seed, float scale)
{
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float u = float(mix32(seed * 0x9e3779b97f4a7c15ull + i) >> 8) * (1.0f / 16777216.0f);
        const __nv_bfloat16 h = __float2bfloat16_rn((2.0f * u - 1.0f) * scale);
        dst[i] = *reinterpret_cast<const uint16_t *>(&h);
    }
}

}  // namespace

cudaError_t launch_fill_bf16(uint16_t *dst, uint64_t n, uint64_t seed, float scale,
                             cudaStream_t stream)
{
    if (n == 0)
        return cudaSuccess;
    const uint64_t blocks = (n + 255) / 256;
    k_fill_bf16<<<unsigned(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(dst, n, seed, scale);
    return cudaGetLastError();
}

}  // namespace lora
