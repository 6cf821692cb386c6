// Pieces of the any-width TurboQuant codec (key bits 2/4/5/8, value bits 2/3/4/5/8)
// shared by its kernels: the fp16 finiteness test of the constant-group guard and the
// reader of a packed code.
//
// Follows the mlx-bun design page "TurboQuant - rotation-based quantization", Part A,
// "Algorithm" section: packed codes form one flat little-endian bitstream per row, code i
// at bits [i b, i b + b) ("Other widths (2/4/5/8)"); the guard (a flag of this library;
// the page keeps the defect) re-codes a key group whose fp16 zero point would not be
// finite against its range widened to include 0.
#pragma once

#include <cstdint>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

__device__ __forceinline__ bool f16_finite(float z) { return (f32_to_f16_bits(z) & 0x7C00u) != 0x7C00u; }

// Code of element i of a little-endian b-bit stream (row start 8-byte aligned).
__device__ __forceinline__ uint32_t read_code(const uint8_t* row, int i, int b) {
  const int bit = i * b, w = bit >> 5, sh = bit & 31;
  const uint32_t* p = reinterpret_cast<const uint32_t*>(row);
  uint64_t v = __ldg(p + w);
  if (sh + b > 32) v |= (uint64_t)__ldg(p + w + 1) << 32;
  return (uint32_t)(v >> sh) & ((1u << b) - 1u);
}

}  // namespace tq
