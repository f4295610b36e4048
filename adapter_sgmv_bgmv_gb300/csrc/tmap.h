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

// The 64 x 16, 64 x 32 and 64 x 64 (columns x rows, 128-byte swizzle) box maps of
// a row matrix; a map whose box is taller than the matrix is left zeroed (no
// block of a matrix that short needs it).
bool encode_row_maps(CUtensorMap maps[3], const void *base, uint64_t width, int64_t nrows,
                     int64_t ld_elems);

}  // namespace lora
