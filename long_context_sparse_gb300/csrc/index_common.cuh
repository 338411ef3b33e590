// index_common.cuh -- helpers shared by the indexer and the top-k kernels.
#pragma once

#include "dsa_common.cuh"

namespace dsa {

// Order-preserving image of an fp32 score: larger float -> larger key.
// -0.0 is first made +0.0 so the two compare equal (lower index wins).
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// (a0, a1) += (w0, w1) * (x0, x1) with one packed fp32 FMA (each lane of
// the pair rounds exactly like fmaf).
__device__ __forceinline__ void fma2(float& a0, float& a1, float w0, float w1,
                                     float x0, float x1) {
  asm("{\n\t.reg .b64 ww, xx, aa;\n\t"
      "mov.b64 ww, {%2, %3};\n\tmov.b64 xx, {%4, %5};\n\t"
      "mov.b64 aa, {%0, %1};\n\t"
      "fma.rn.f32x2 aa, ww, xx, aa;\n\t"
      "mov.b64 {%0, %1}, aa;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(w0), "f"(w1), "f"(x0), "f"(x1));
}

}  // namespace dsa
