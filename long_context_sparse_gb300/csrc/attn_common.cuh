// attn_common.cuh -- warp-level tensor-core fragments, cp.async gathers and
// the per-query key-set builder shared by the sparse attention kernels.
#pragma once

#include "dsa_common.cuh"

namespace dsa {

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
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Rows of D bf16 (D*2 bytes) in shared memory, 16-byte chunks XOR-swizzled
// by (row & 7) so that 8 consecutive rows at one logical chunk hit 8
// different bank groups (conflict-free ldmatrix).
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * (D * 2) + ((chunk ^ (row & 7)) << 4));
}

// ---------------------------------------------------------- ldmatrix/mma
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                        uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr));
}
// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                         uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
      "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void red_add_v2(float* addr, float a, float b) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(addr), "f"(a), "f"(b)
               : "memory");
}

__device__ __forceinline__ void named_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// ------------------------------------------------------------ key set
// Token list of query t into toks[]: the 4 tokens of every selected pool
// (slot 4i+j <-> pool idx[i], token 4p+j), then, for n_loc = 3, those of
// {t-2, t-1, t} (>= 0) that no selected pool already covers.  Slots of
// empty (-1) or out-of-range pools hold -1 (masked); an out-of-range pool
// also latches DSA_ERR_DEVICE_BAD_INDEX.  Valid pools are a prefix of the
// row (ascending, then -1), so the list length is 4*(last valid slot+1)
// plus the locals.  Tail up to a multiple of `pad` is filled with -1.
// Returns the number of slots; every thread of the block must call it.
__device__ __forceinline__ int build_key_list(const int32_t* __restrict__ idx_row,
                                              int64_t t, int K_p, int n_loc,
                                              int pad, int32_t* toks,
                                              int* scratch2, uint32_t* status) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int64_t nf = n_full(t);
  if (tid == 0) {
    scratch2[0] = -1;
    scratch2[1] = 0;
  }
  __syncthreads();
  for (int i = tid; i < K_p; i += nthr) {
    const int32_t p = __ldg(idx_row + i);
    const bool ok = p >= 0 && (int64_t)p < nf;
    if (p >= 0) {
      atomicMax(&scratch2[0], i);
      if (!ok) latch_error(status, DSA_ERR_DEVICE_BAD_INDEX);
    }
    const int32_t base = ok ? 4 * p : -1;
#pragma unroll
    for (int j = 0; j < 4; ++j) toks[4 * i + j] = ok ? base + j : -1;
  }
  __syncthreads();
  const int n_pool_slots = 4 * (scratch2[0] + 1);
  if (n_loc > 0 && tid < 32) {
    int nadd = 0;
    for (int j = n_loc - 1; j >= 0; --j) {
      const int64_t s = t - j;
      if (s < 0) continue;
      const int32_t ps = (int32_t)(s >> 2);
      bool mine = false;
      // covered iff its (complete, earlier) pool is among the selected
      if ((int64_t)ps < nf)
        for (int i = tid; i < K_p; i += 32) mine |= __ldg(idx_row + i) == ps;
      const bool covered = __any_sync(0xffffffffu, mine);
      if (!covered) {
        if (tid == 0) toks[n_pool_slots + nadd] = (int32_t)s;
        ++nadd;
      }
    }
    if (tid == 0) scratch2[1] = nadd;
  }
  __syncthreads();
  const int n = n_pool_slots + scratch2[1];
  const int n_pad = (n + pad - 1) / pad * pad;
  for (int i = n + tid; i < n_pad; i += nthr) toks[i] = -1;
  __syncthreads();
  return n;
}

}  // namespace dsa
