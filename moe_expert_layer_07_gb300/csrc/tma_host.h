// Host-side TMA descriptor encoding shared by the tensor-core kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace moe {

// Tensor map of a row-major [outer, inner] matrix (e4m3 bytes or bf16) with
// a box of 128 bytes x box_rows and 128-byte swizzle; false when the CUDA driver's
// encoder is unavailable or rejects the layout (base not 16-byte aligned,
// row pitch not a multiple of 16 bytes).
bool encode_2d(CUtensorMap *m, const void *base, bool fp8, uint64_t inner, uint64_t outer,
               uint32_t box_rows);

// Tensor map of a row-major fp32 [outer, inner] matrix with a box of 32
// columns (128 bytes) x box_rows and 128-byte swizzle, for TMA stores.
bool encode_2d_f32(CUtensorMap *m, void *base, uint64_t inner, uint64_t outer, uint32_t box_rows);

}  // namespace moe
