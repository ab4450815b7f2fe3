// Tensor-map (TMA descriptor) encoding for the kernels' 2D tiled copies.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace cdb {

// bf16 tensor [outer][inner] with a row stride of `stride` bytes, box
// box_inner x box_outer elements, swizzle of `swizzle` bytes (0, 32, 64 or
// 128).  Descriptors are encoded once per distinct argument set and cached for
// the process; nullptr when the driver entry point is missing or the encoder
// rejects the arguments.
const CUtensorMap* tmap_bf16_2d(const void* p, uint64_t inner, uint64_t outer, uint64_t stride, uint32_t box_inner,
                                uint32_t box_outer, int swizzle);

}  // namespace cdb
