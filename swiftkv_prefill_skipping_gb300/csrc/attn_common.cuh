// Small helpers shared by the tcgen05 prompt-attention kernels.
#pragma once

#include <stdint.h>

namespace skv {

// max of three floats in one instruction
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two floats to f16x2 (lo in the low half), round to nearest even, saturating at +-65504.
__device__ __forceinline__ uint32_t pack_f16_sat(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

}  // namespace skv
