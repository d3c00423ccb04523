// f32x2.cuh -- paired fp32 arithmetic of the sm_100 family: one instruction
// works on two fp32 values held in a 64-bit register pair, which halves the
// instruction count of the scale-and-shift before each exponential of the
// softmax; and the three-input maximum, which halves that of the row maxima.
// Plain IEEE round-to-nearest operations, no approximation.
#pragma once

#include <stdint.h>

namespace attn {

__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void f32x2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// a * b + c per lane, rounded once
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

}  // namespace attn
