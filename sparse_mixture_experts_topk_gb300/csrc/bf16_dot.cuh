// Dot-product steps on bf16 operands with fp32 sums, shared by the decode
// router and the weight-streaming expert kernel.
#pragma once

#include <cstdint>

namespace moe {

// acc + x.lo w.lo + x.hi w.hi for bf16 pairs packed in 32-bit words: two
// fused multiply-adds with bf16 operands and an fp32 addend and result.  A
// product of two bf16 values is exact in fp32, so each step rounds once,
// exactly like fmaf on the widened values, without widening them first.
__device__ __forceinline__ float fma2_bf16(uint32_t x, uint32_t w, float acc) {
  asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
      "mov.b32 {xl, xh}, %1;\n\t"
      "mov.b32 {wl, wh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, xl, wl, %0;\n\t"
      "fma.rn.f32.bf16 %0, xh, wh, %0;\n\t}"
      : "+f"(acc)
      : "r"(x), "r"(w));
  return acc;
}
__device__ __forceinline__ float fma8_bf16(const uint4& x, const uint4& w, float acc) {
  acc = fma2_bf16(x.x, w.x, acc);
  acc = fma2_bf16(x.y, w.y, acc);
  acc = fma2_bf16(x.z, w.z, acc);
  return fma2_bf16(x.w, w.w, acc);
}

}  // namespace moe
