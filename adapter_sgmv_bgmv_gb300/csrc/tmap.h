// TMA tensor-map encoding (host).
#pragma once
#include <cstdint>
#include <cuda.h>

namespace lora {

// 2-D bf16 tensor [outer][inner] with a row stride in bytes (multiple of 16) and
// a box of box_outer rows x box_inner elements; 128-byte swizzle when asked (then
// box_inner * 2 must be 128).  Out-of-range elements load as zero and are not
// stored.  Returns false when the driver refuses the description.
bool encode_bf16_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                    bool swizzle128);

}  // namespace lora
