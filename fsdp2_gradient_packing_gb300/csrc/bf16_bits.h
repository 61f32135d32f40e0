// Conversions between binary32 and bfloat16 on raw bits, shared by the table
// walker (kernels.cu) and the emulated reduce-scatter (reduce.cu).  Device
// code only; included by the .cu files.
#pragma once

#include <cstdint>

namespace fsdp {

__device__ __forceinline__ uint32_t bf16_to_f32_bits(uint32_t h) { return h << 16; }

// IEEE-754 round to nearest, ties to even, from binary32 to bfloat16 (the
// upper 16 bits).  Adding 0x7FFF plus the lowest kept bit carries into the
// kept half exactly when the dropped half is above one half ulp, or equal to
// it with an odd kept half; a carry out of the largest finite value gives
// infinity, as IEEE-754 requires.  NaN keeps its sign and upper payload and
// gets the quiet bit.
__device__ __forceinline__ uint32_t f32_to_bf16_bits(uint32_t u) {
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (u >> 16) | 0x0040u;
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

}  // namespace fsdp
