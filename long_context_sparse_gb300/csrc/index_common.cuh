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

// The indexer's epilogue for one pool (this thread's TMEM lane) over one
// half of an N tile: 128 fp32 accumulator columns = 128 / HI queries x HI
// heads, starting at TMEM address `taddr`.  For each query it forms
//   I = sum_h w_h * max(0, x_h)
// in fp32: head pair j of a query (columns 2j, 2j+1) is added with one
// packed FMA into accumulator pair j % NA (NA = min(4, HI / 2) independent
// chains), and the 2 NA partial sums are combined as a balanced tree;
// emit(qi, I) receives query qi of the half (a compile-time constant after
// unrolling).  wr holds the half's 128 weights.  The TMEM load of the next
// 16 columns is issued before the current 16 are used.  Every kernel that
// scores pools calls this, so their scores agree bit for bit.
template <int HI, class Emit>
__device__ __forceinline__ void relu_weighted_sums(uint32_t taddr, const float (&wr)[128],
                                                   Emit emit) {
  static_assert(HI >= 2 && HI <= 128 && (HI & (HI - 1)) == 0, "heads per query");
  constexpr int NPQ = HI / 2;              // head pairs per query
  constexpr int NA = NPQ < 4 ? NPQ : 4;    // accumulator pairs
  float acc[2 * NA];
  uint32_t buf[2][16];
  tmem_ld16(taddr, buf[0]);
  tmem_wait_ld_dep(buf[0]);
#pragma unroll
  for (int g = 0; g < 8; ++g) {            // 16-column groups
    if (g + 1 < 8) tmem_ld16(taddr + (uint32_t)((g + 1) * 16), buf[(g + 1) & 1]);
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      const int col = g * 16 + j;          // column within the half
      const int pq = (col % HI) / 2;       // head pair within the query
      const int ai = pq % NA;
      const float x0 = fmaxf(__uint_as_float(buf[g & 1][j]), 0.f);
      const float x1 = fmaxf(__uint_as_float(buf[g & 1][j + 1]), 0.f);
      if (pq < NA) {                       // first pair of this chain
        acc[2 * ai] = 0.f;
        acc[2 * ai + 1] = 0.f;
      }
      fma2(acc[2 * ai], acc[2 * ai + 1], wr[col], wr[col + 1], x0, x1);
      if (pq == NPQ - 1) {                 // last pair of the query
        float s[2 * NA];
#pragma unroll
        for (int e = 0; e < 2 * NA; ++e) s[e] = acc[e];
#pragma unroll
        for (int w = 1; w < 2 * NA; w *= 2)
#pragma unroll
          for (int e = 0; e < 2 * NA; e += 2 * w) s[e] = s[e] + s[e + w];
        emit(col / HI, s[0]);
      }
    }
    if (g + 1 < 8) tmem_wait_ld_dep(buf[(g + 1) & 1]);
  }
}

}  // namespace dsa
