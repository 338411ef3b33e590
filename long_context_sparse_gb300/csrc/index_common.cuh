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

// Barrier `id` over `n` threads (a multiple of 32).  Unbounded: every
// participating warp must reach it the same number of times.
__device__ __forceinline__ void named_bar(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
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

// The indexer's epilogue for one pool (this thread's TMEM lane) over NC
// consecutive fp32 accumulator columns = NC / HI queries x HI heads,
// starting at TMEM address `taddr`.  For each query it forms
//   I = sum_h w_h * max(0, x_h)
// in fp32: head pair j of a query (columns 2j, 2j+1) is added with one
// packed FMA into accumulator pair j % NA (NA = min(4, HI / 2) independent
// chains, each started by a packed multiply), and the NA pairs are combined
// with packed adds as a balanced tree, then the pair's two halves;
// emit(qi, I) receives query qi of the range (a compile-time constant after
// unrolling).  w4(i) returns the weights of columns 4i .. 4i+3.
//
// kLoadAll = false: the TMEM load of the next 16 columns is issued before
// the current 16 are used.  kLoadAll = true: all NC columns are loaded into
// registers first and released() is called (the accumulator may then be
// overwritten) before any arithmetic.  The arithmetic, and so the result of
// a query, is the same either way and depends only on the query's own HI
// columns, so kernels that split the columns differently among their
// threads agree bit for bit; every kernel that scores pools calls this.
template <int HI, int NC, bool kLoadAll, class W4, class Emit, class Released>
__device__ __forceinline__ void relu_weighted_sums(uint32_t taddr, W4 w4, Emit emit,
                                                   Released released) {
  static_assert(HI >= 2 && HI <= NC && (HI & (HI - 1)) == 0, "heads per query");
  static_assert(NC % 16 == 0, "16-column groups");
  constexpr int NPQ = HI / 2;              // head pairs per query
  constexpr int NA = NPQ < 4 ? NPQ : 4;    // accumulator pairs
  constexpr int NG = NC / 16;
  float2 acc[NA];
  // columns col, col+1 with accumulator bits v0, v1; weights wv
  auto step = [&](int col, uint32_t v0, uint32_t v1, float2 wv) {
    const int pq = (col % HI) / 2;         // head pair within the query
    const int ai = pq % NA;
    const float2 x = make_float2(fmaxf(__uint_as_float(v0), 0.f), fmaxf(__uint_as_float(v1), 0.f));
    acc[ai] = pq < NA ? __fmul2_rn(wv, x)  // first pair of this chain
                      : __ffma2_rn(wv, x, acc[ai]);
    if (pq == NPQ - 1) {                   // last pair of the query
#pragma unroll
      for (int w = 1; w < NA; w *= 2)
#pragma unroll
        for (int e = 0; e < NA; e += 2 * w) acc[e] = __fadd2_rn(acc[e], acc[e + w]);
      emit(col / HI, acc[0].x + acc[0].y);
    }
  };
  if constexpr (kLoadAll) {
    uint32_t vals[NG][16];
#pragma unroll
    for (int g = 0; g < NG; ++g) tmem_ld16(taddr + (uint32_t)(g * 16), vals[g]);
#pragma unroll
    for (int g = 0; g < NG; ++g) tmem_wait_ld_dep(vals[g]);
    released();
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int j4 = 0; j4 < 16; j4 += 4) {
        const float4 wq = w4((g * 16 + j4) / 4);
        step(g * 16 + j4, vals[g][j4], vals[g][j4 + 1], make_float2(wq.x, wq.y));
        step(g * 16 + j4 + 2, vals[g][j4 + 2], vals[g][j4 + 3], make_float2(wq.z, wq.w));
      }
  } else {
    uint32_t buf[2][16];
    tmem_ld16(taddr, buf[0]);
    tmem_wait_ld_dep(buf[0]);
#pragma unroll
    for (int g = 0; g < NG; ++g) {         // 16-column groups
      if (g + 1 < NG) tmem_ld16(taddr + (uint32_t)((g + 1) * 16), buf[(g + 1) & 1]);
#pragma unroll
      for (int j4 = 0; j4 < 16; j4 += 4) {
        const float4 wq = w4((g * 16 + j4) / 4);
        step(g * 16 + j4, buf[g & 1][j4], buf[g & 1][j4 + 1], make_float2(wq.x, wq.y));
        step(g * 16 + j4 + 2, buf[g & 1][j4 + 2], buf[g & 1][j4 + 3], make_float2(wq.z, wq.w));
      }
      if (g + 1 < NG) tmem_wait_ld_dep(buf[(g + 1) & 1]);
    }
    released();
  }
}

}  // namespace dsa
