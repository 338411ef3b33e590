// index_common.cuh -- helpers shared by the indexer and the top-k kernels.
#pragma once

#include <atomic>

#include "dsa_common.cuh"

namespace dsa {

// Raise a kernel's dynamic shared-memory limit on the current device once:
// `done` holds one bit per device, set after the call succeeded, so threads
// and devices may interleave freely (a repeated call is harmless).
template <class Kernel>
inline cudaError_t set_smem_once(Kernel kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

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
