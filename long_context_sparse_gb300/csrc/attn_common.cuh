// attn_common.cuh -- helpers shared by the tcgen05 sparse attention
// kernels: shared-memory carving, cp.async gathers, group barriers.
#pragma once

#include "dsa_common.cuh"

namespace dsa {

// Shared-memory carving: `n` elements of T at the next 128-byte boundary,
// advancing `p`; carved(b) is the bytes one such region takes at most.
template <typename T>
__device__ __forceinline__ T* carve(uint8_t*& p, int n) {
  uint8_t* a = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 127) &
                                          ~uintptr_t(127));
  p = a + (size_t)n * sizeof(T);
  return reinterpret_cast<T*>(a);
}
__host__ __device__ constexpr uint32_t carved(uint32_t bytes) { return bytes + 128; }

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------- cp.async
// 16-byte global -> shared copy; src_bytes = 0 zero-fills (masked rows).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src,
                                           uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  // arrive on `bar` once every cp.async this thread issued so far has landed
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  // order this thread's shared-memory writes before the tensor core's reads
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// A barrier among the threads of one warp-specialised role, built on an
// mbarrier so that every wait is bounded like the others: a thread whose
// wait gave up cannot leave its peers blocked.
struct GroupBar {
  uint32_t bar;
  uint32_t phase;
  __device__ __forceinline__ bool sync(const Waiter& W) {
    mbar_arrive(bar);
    const bool ok = W.wait(bar, phase & 1u);
    ++phase;
    return ok;
  }
};

__device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity, uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > ns) return false;
  return true;
}

}  // namespace dsa
