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
constexpr int kBins = 2048;  // 11-bit digits: bits 31-21, 20-10, 9-0

// Order-preserving image of an fp32 score: larger float -> larger key.
// -0.0 is first made +0.0 so the two compare equal (lower index wins).
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Digit d of the highest bins that holds the kk-th largest key; *above =
// number of keys in higher bins.  Warp 0 only; lane l owns 64 bins.
__device__ __forceinline__ void find_digit(const uint32_t* hist, uint32_t kk,
                                           uint32_t* sel_digit, uint32_t* sel_above) {
  const int lane = threadIdx.x & 31;
  const int base = kBins - 64 * (lane + 1);  // lane 0: the top 64 bins
  uint32_t s = 0u;
#pragma unroll
  for (int j = 0; j < 64; j += 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(hist + base + j);
    s += v.x + v.y + v.z + v.w;
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
    for (int j = 63; j >= 0; --j) {
      const uint32_t c = hist[base + j];
      if (acc + c >= kk) {
        *sel_digit = (uint32_t)(base + j);
        *sel_above = acc;
        break;
      }
      acc += c;
    }
  }
}

__global__ void __launch_bounds__(kTopkThreads, 1)
    topk_rows_kernel(const float* __restrict__ scores, int64_t ld, int64_t row0,
                     int64_t rows, int K_p, int32_t* __restrict__ out,
                     int cache_cap) {
  extern __shared__ __align__(16) uint32_t cache[];
  __shared__ __align__(16) uint32_t hist[kBins];
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
    // 16-byte rows (the library's own score chunks always are) are read as
    // float4, four loads in flight per thread, so the first pass does not
    // wait on one L2 round trip per element
    const bool vec = ((reinterpret_cast<uintptr_t>(row) & 15u) == 0);
    const int64_t n4 = vec ? n / 4 : 0;

    // ---- radix select of the K_p-th largest key: digits of 11, 11, 10 bits
    uint32_t prefix = 0u, pmask = 0u, kk = (uint32_t)K_p;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const uint32_t dmask = pass == 2 ? 1023u : 2047u;
      for (int i = tid; i < kBins; i += kTopkThreads) hist[i] = 0u;
      __syncthreads();
      if (pass == 0) {
        // first touch of the row: load, map, cache, count
        const float4* row4 = reinterpret_cast<const float4*>(row);
        for (int64_t b = tid; b < n4; b += 4 * kTopkThreads) {
          float4 x[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int64_t j = b + u * kTopkThreads;
            x[u] = j < n4 ? __ldg(row4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int64_t j = b + u * kTopkThreads;
            if (j < n4) {
              const uint32_t k4[4] = {order_key(x[u].x), order_key(x[u].y),
                                      order_key(x[u].z), order_key(x[u].w)};
              if (cached)
                *reinterpret_cast<uint4*>(cache + 4 * j) = make_uint4(k4[0], k4[1], k4[2], k4[3]);
#pragma unroll
              for (int e = 0; e < 4; ++e) atomicAdd(&hist[k4[e] >> 21], 1u);
            }
          }
        }
        for (int64_t i = 4 * n4 + tid; i < n; i += kTopkThreads) {
          const uint32_t key = order_key(__ldg(row + i));
          if (cached) cache[i] = key;
          atomicAdd(&hist[key >> 21], 1u);
        }
      } else if (cached) {
        for (int64_t i = tid; i < n; i += kTopkThreads) {
          const uint32_t key = cache[i];
          if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & dmask], 1u);
        }
      } else {
        const float4* row4 = reinterpret_cast<const float4*>(row);
        for (int64_t b = tid; b < n4; b += 4 * kTopkThreads) {
          float4 x[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int64_t j = b + u * kTopkThreads;
            x[u] = j < n4 ? __ldg(row4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (b + u * kTopkThreads >= n4) continue;
            const uint32_t k4[4] = {order_key(x[u].x), order_key(x[u].y),
                                    order_key(x[u].z), order_key(x[u].w)};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if ((k4[e] & pmask) == prefix) atomicAdd(&hist[(k4[e] >> shift) & dmask], 1u);
          }
        }
        for (int64_t i = 4 * n4 + tid; i < n; i += kTopkThreads) {
          const uint32_t key = order_key(__ldg(row + i));
          if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & dmask], 1u);
        }
      }
      __syncthreads();
      if (warp == 0) find_digit(hist, kk, &sel_digit, &sel_above);
      __syncthreads();
      prefix |= sel_digit << shift;
      pmask |= dmask << shift;
      kk -= sel_above;
    }
    // prefix = key of the K_p-th best; take every key above it and the kk
    // lowest-index keys equal to it, in index order.  Each warp owns one
    // contiguous segment: count, one block-wide exclusive scan, write.
    const uint32_t T = prefix;
    const int64_t seg = ((n + kTopkWarps - 1) / kTopkWarps + 31) & ~int64_t(31);
    const int64_t b0 = warp * seg;
    const int64_t b1 = b0 + seg < n ? b0 + seg : n;
    uint32_t cg = 0u, ct = 0u;
    for (int64_t i0 = b0; i0 < b1; i0 += 32) {
      const int64_t i = i0 + lane;
      uint32_t key = 0u;
      if (i < b1) key = cached ? cache[i] : order_key(__ldg(row + i));
      cg += __popc(__ballot_sync(0xffffffffu, i < b1 && key > T));
      ct += __popc(__ballot_sync(0xffffffffu, i < b1 && key == T));
    }
    if (lane == 0) {
      wcnt[0][warp] = cg;
      wcnt[1][warp] = ct;
    }
    __syncthreads();
    uint32_t g_base = 0u, t_base = 0u;
#pragma unroll
    for (int w = 0; w < kTopkWarps; ++w) {
      if (w < warp) {
        g_base += wcnt[0][w];
        t_base += wcnt[1][w];
      }
    }
    for (int64_t i0 = b0; i0 < b1; i0 += 32) {
      if (t_base >= kk && g_base + kk >= (uint32_t)K_p) break;  // warp-uniform
      const int64_t i = i0 + lane;
      uint32_t key = 0u;
      if (i < b1) key = cached ? cache[i] : order_key(__ldg(row + i));
      const bool gt = i < b1 && key > T;
      const bool tie = i < b1 && key == T;
      const uint32_t bg = __ballot_sync(0xffffffffu, gt);
      const uint32_t bt = __ballot_sync(0xffffffffu, tie);
      const uint32_t g_before = g_base + __popc(bg & lane_lt);
      const uint32_t t_before = t_base + __popc(bt & lane_lt);
      // (positions are < K_p by construction; the guard keeps a corrupted
      // row from writing into its neighbour)
      const uint32_t pos = gt ? g_before + min(t_before, kk) : g_before + t_before;
      if ((gt || (tie && t_before < kk)) && pos < (uint32_t)K_p) o[pos] = (int32_t)i;
      g_base += __popc(bg);
      t_base += __popc(bt);
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
  static int attr_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(kTopkCacheMax * sizeof(uint32_t)));
    if (e != cudaSuccess) return e;
    attr_dev = dev;
  }
  int64_t grid = rows;
  const int64_t cap = (int64_t)c.num_sms * 8;
  if (grid > cap) grid = cap;
  topk_rows_kernel<<<(unsigned)grid, kTopkThreads, smem, c.stream>>>(
      scores, ld, row0, rows, K_p, out, cache_cap);
  return cudaGetLastError();
}

}  // namespace dsa
