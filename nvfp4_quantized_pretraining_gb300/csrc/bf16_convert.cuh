// BF16 rounding shared by the elementwise and optimizer-side kernels.
#pragma once

#include <stdint.h>

namespace nvfp4 {

// binary32 -> BF16 bit pattern, round to nearest, ties to even (the PTX conversion).
__device__ __forceinline__ uint32_t bf16_rn_bits(float v) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
  return r;
}

}  // namespace nvfp4
