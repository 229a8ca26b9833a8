// Small helpers shared by the tcgen05 prompt-attention kernels.
#pragma once

#include <stdint.h>

#include "common.cuh"

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

// Softmax weights of one 64-key block as bfloat16 high and low parts (split_pair_bf16), for a
// P V product on bf16 tensor cores that keeps P to about 17 significant bits: w[c] packs the
// high parts of p[2c] (low half) and p[2c + 1], w[32 + c] their low parts.
__device__ __forceinline__ void split_p_bf16(const float* p, uint32_t* w) {
#pragma unroll
  for (int c = 0; c < 32; ++c) split_pair_bf16(p[2 * c], p[2 * c + 1], w[c], w[32 + c]);
}

}  // namespace skv
