// select.cu -- key pooling (a1) and per-query top-k selection (a4).
//
// Pooling: "the indexer scores every query against every earlier pool of 4
// tokens" ("Scaling Training to 1M Token Context on GLM-5.3-Flash", section
// "DeepSeek Sparse Attention (DSA) Optimizations"); a pool key is the mean of
// its 4 indexer keys, rounded as fp32 ((k0+k1)+(k2+k3))*0.25 -> bf16 RNE.
//
// Selection: the K_p highest-scoring complete earlier pools of each query,
// ties toward the lower pool index, written as int32 in ascending pool order
// (same page, sections "DeepSeek Sparse Attention (DSA) Optimizations" and
// "Across GPUs: Sharding").  Exact radix select on an order-preserving u32
// image of the fp32 score, then one index-ordered compaction pass: the
// result is bit-identical to a stable sort on (score desc, index asc).
#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {

// --------------------------------------------------------------- pooling
// One thread per (pool, pair of dims): 4 x 32-bit loads, fp32 adds in the
// fixed order, one packed bf16x2 store.  HBM-bound, fully coalesced.
__global__ void __launch_bounds__(256) pool4_kernel(const uint32_t* __restrict__ k,
                                                    uint32_t* __restrict__ kp,
                                                    int64_t P, int half_d) {
  const int64_t n = P * half_d;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t p = i / half_d;
    const int64_t c = i - p * half_d;
    const uint32_t* base = k + (4 * p) * half_d + c;
    const uint32_t x0 = __ldg(base), x1 = __ldg(base + half_d),
                   x2 = __ldg(base + 2 * half_d), x3 = __ldg(base + 3 * half_d);
    const float lo = __fmul_rn(__fadd_rn(__fadd_rn(bf16_lo(x0), bf16_lo(x1)),
                                         __fadd_rn(bf16_lo(x2), bf16_lo(x3))),
                               0.25f);
    const float hi = __fmul_rn(__fadd_rn(__fadd_rn(bf16_hi(x0), bf16_hi(x1)),
                                         __fadd_rn(bf16_hi(x2), bf16_hi(x3))),
                               0.25f);
    kp[i] = pack_bf16(lo, hi);
  }
}

cudaError_t launch_pool(const LaunchCtx& c, const __nv_bfloat16* k_idx,
                        __nv_bfloat16* k_pool, int64_t S, int D_I) {
  const int64_t P = S / 4;
  if (P == 0) return cudaSuccess;
  const int64_t n = P * (D_I / 2);
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = (int64_t)c.num_sms * 16;
  if (blocks > cap) blocks = cap;
  pool4_kernel<<<(unsigned)blocks, 256, 0, c.stream>>>(
      reinterpret_cast<const uint32_t*>(k_idx), reinterpret_cast<uint32_t*>(k_pool),
      P, D_I / 2);
  return cudaGetLastError();
}

// ----------------------------------------------------------------- top-k
constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
// Rows of up to this many candidates are staged in shared memory once.
constexpr int kTopkCacheMax = 48 * 1024;

// Order-preserving image of an fp32 score: larger float -> larger key.
// -0.0 is first made +0.0 so the two compare equal (lower index wins).
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void __launch_bounds__(kTopkThreads, 1)
    topk_rows_kernel(const float* __restrict__ scores, int64_t ld, int64_t row0,
                     int64_t rows, int K_p, int32_t* __restrict__ out,
                     int cache_cap) {
  extern __shared__ uint32_t cache[];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t wcnt[2][kTopkWarps];
  __shared__ uint32_t sel_digit, sel_above;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lane_lt = (1u << lane) - 1u;

  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const int64_t t = row0 + r;
    int64_t n = n_full(t);
    if (n > ld) n = ld;
    int32_t* o = out + r * (int64_t)K_p;
    const float* row = scores + r * ld;

    if (n <= K_p) {  // every earlier pool is selected
      for (int i = tid; i < K_p; i += kTopkThreads) o[i] = i < n ? i : -1;
      continue;
    }
    const bool cached = n <= cache_cap;

    // ---- radix select of the K_p-th largest key, 8 bits per pass
    uint32_t prefix = 0u, pmask = 0u, kk = (uint32_t)K_p;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0u;
      __syncthreads();
      for (int64_t b = 0; b < n; b += kTopkThreads) {
        const int64_t i = b + tid;
        uint32_t key = 0u;
        bool live = i < n;
        if (live) {
          if (pass == 0) {
            key = order_key(__ldg(row + i));
            if (cached) cache[i] = key;
          } else {
            key = cached ? cache[i] : order_key(__ldg(row + i));
          }
          live = (key & pmask) == prefix;
        }
        // warp-aggregated histogram update (scores share few exponents)
        const uint32_t digit = live ? (key >> shift) & 255u : 256u;
        const uint32_t peers = __match_any_sync(0xffffffffu, digit);
        if (live && (peers & lane_lt) == 0u) atomicAdd(&hist[digit], __popc(peers));
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns bins 8*(31-l) .. 8*(31-l)+7 (lane 0 = highest bins)
        const int base = 8 * (31 - lane);
        uint32_t c[8], s = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = hist[base + j];
          s += c[j];
        }
        uint32_t incl = s;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const uint32_t x = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += x;
        }
        const uint32_t excl = incl - s;
        if (excl < kk && kk <= incl) {
          uint32_t acc = excl;
          for (int j = 7; j >= 0; --j) {
            if (acc + c[j] >= kk) {
              sel_digit = (uint32_t)(base + j);
              sel_above = acc;
              break;
            }
            acc += c[j];
          }
        }
      }
      __syncthreads();
      prefix |= sel_digit << shift;
      pmask |= 255u << shift;
      kk -= sel_above;
      __syncthreads();
    }
    // prefix = key of the K_p-th best; take every key above it and the kk
    // lowest-index keys equal to it.
    const uint32_t T = prefix;
    const uint32_t want_gt = (uint32_t)K_p - kk;
    uint32_t base_gt = 0u, base_tie = 0u;
    for (int64_t b = 0; b < n; b += kTopkThreads) {
      if (base_gt == want_gt && base_tie >= kk) break;  // uniform
      const int64_t i = b + tid;
      uint32_t key = 0u;
      if (i < n) key = cached ? cache[i] : order_key(__ldg(row + i));
      const bool gt = i < n && key > T;
      const bool tie = i < n && key == T;
      const uint32_t bg = __ballot_sync(0xffffffffu, gt);
      const uint32_t bt = __ballot_sync(0xffffffffu, tie);
      if (lane == 0) {
        wcnt[0][warp] = __popc(bg);
        wcnt[1][warp] = __popc(bt);
      }
      __syncthreads();
      uint32_t wg = 0u, wt = 0u, tg = 0u, tt = 0u;
#pragma unroll
      for (int w = 0; w < kTopkWarps; ++w) {
        const uint32_t a = wcnt[0][w], e = wcnt[1][w];
        if (w < warp) {
          wg += a;
          wt += e;
        }
        tg += a;
        tt += e;
      }
      const uint32_t g_before = base_gt + wg + __popc(bg & lane_lt);
      const uint32_t t_before = base_tie + wt + __popc(bt & lane_lt);
      // (positions are < K_p by construction; the guard keeps a corrupted
      // row from writing into its neighbour)
      const uint32_t pos = gt ? g_before + min(t_before, kk) : g_before + t_before;
      if ((gt || (tie && t_before < kk)) && pos < (uint32_t)K_p) o[pos] = (int32_t)i;
      base_gt += tg;
      base_tie += tt;
      __syncthreads();
    }
    __syncthreads();
  }
}

cudaError_t launch_topk(const LaunchCtx& c, const float* scores, int64_t ld,
                        int64_t row0, int64_t rows, int K_p, int32_t* out) {
  if (rows <= 0) return cudaSuccess;
  int64_t nmax = n_full(row0 + rows - 1);
  if (nmax > ld) nmax = ld;
  int cache_cap = nmax <= kTopkCacheMax ? (int)nmax : 0;
  const size_t smem = (size_t)cache_cap * sizeof(uint32_t);
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(kTopkCacheMax * sizeof(uint32_t)));
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  int64_t grid = rows;
  const int64_t cap = (int64_t)c.num_sms * 8;
  if (grid > cap) grid = cap;
  topk_rows_kernel<<<(unsigned)grid, kTopkThreads, smem, c.stream>>>(
      scores, ld, row0, rows, K_p, out, cache_cap);
  return cudaGetLastError();
}

}  // namespace dsa
