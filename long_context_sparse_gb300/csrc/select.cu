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
#include "index_common.cuh"
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

// --------------------------------------------------------- gated pooling
// "k-pool gate scores that weight each key within a pool" ("Scaling
// Training to 1M Token Context on GLM-5.3-Flash", section "DSA: Gather by
// Token Position"), read as a softmax over the pool's 4 gate scores:
//   w_j = exp(g_j - m) / ((e0 + e1) + (e2 + e3)),  m = max_j g_j
//   k_pool = bf16_rne(((w0 k0 + w1 k1) + (w2 k2 + w3 k3)))      (fp32)
// Equal gates give weights of exactly 1/4, i.e. the mean pooling above.
__global__ void __launch_bounds__(256) pool4_gated_kernel(
    const uint32_t* __restrict__ k, const float* __restrict__ gate,
    uint32_t* __restrict__ kp, int64_t P, int half_d) {
  const int64_t n = P * half_d;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t p = i / half_d;
    const int64_t c = i - p * half_d;
    const float4 g = __ldg(reinterpret_cast<const float4*>(gate) + p);
    const float m = fmaxf(fmaxf(g.x, g.y), fmaxf(g.z, g.w));
    const float e0 = expf(g.x - m), e1 = expf(g.y - m), e2 = expf(g.z - m),
                e3 = expf(g.w - m);
    const float den = __fadd_rn(__fadd_rn(e0, e1), __fadd_rn(e2, e3));
    const float w0 = __fdiv_rn(e0, den), w1 = __fdiv_rn(e1, den),
                w2 = __fdiv_rn(e2, den), w3 = __fdiv_rn(e3, den);
    const uint32_t* base = k + (4 * p) * half_d + c;
    const uint32_t x0 = __ldg(base), x1 = __ldg(base + half_d),
                   x2 = __ldg(base + 2 * half_d), x3 = __ldg(base + 3 * half_d);
    const float lo = __fadd_rn(__fadd_rn(__fmul_rn(w0, bf16_lo(x0)), __fmul_rn(w1, bf16_lo(x1))),
                               __fadd_rn(__fmul_rn(w2, bf16_lo(x2)), __fmul_rn(w3, bf16_lo(x3))));
    const float hi = __fadd_rn(__fadd_rn(__fmul_rn(w0, bf16_hi(x0)), __fmul_rn(w1, bf16_hi(x1))),
                               __fadd_rn(__fmul_rn(w2, bf16_hi(x2)), __fmul_rn(w3, bf16_hi(x3))));
    kp[i] = pack_bf16(lo, hi);
  }
}

cudaError_t launch_pool_gated(const LaunchCtx& c, const __nv_bfloat16* k_idx,
                              const float* gate, __nv_bfloat16* k_pool, int64_t S,
                              int D_I) {
  const int64_t P = S / 4;
  if (P == 0) return cudaSuccess;
  const int64_t n = P * (D_I / 2);
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = (int64_t)c.num_sms * 16;
  if (blocks > cap) blocks = cap;
  pool4_gated_kernel<<<(unsigned)blocks, 256, 0, c.stream>>>(
      reinterpret_cast<const uint32_t*>(k_idx), gate, reinterpret_cast<uint32_t*>(k_pool),
      P, D_I / 2);
  return cudaGetLastError();
}

// ----------------------------------------------------------------- top-k
constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
// Rows of up to this many candidates are staged in shared memory once.
constexpr int kTopkCacheMax = 48 * 1024;
constexpr int kBins = 2048;  // 11-bit digits: bits 31-21, 20-10, 9-0

// Digit d of the highest bins that holds the kk-th largest key; *above =
// number of keys in higher bins.  Warp 0 only: lane l first sums the 64
// bins kBins-64(l+1) .. kBins-64l-1 (lane 0: the top 64), a warp scan finds
// the lane whose range holds the kk-th key, then the whole warp scans that
// range two bins per lane, highest first.
__device__ __forceinline__ void find_digit(const uint32_t* hist, uint32_t kk,
                                           uint32_t* sel_digit, uint32_t* sel_above) {
  const int lane = threadIdx.x & 31;
  const int base = kBins - 64 * (lane + 1);
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
  const uint32_t hit = __ballot_sync(0xffffffffu, incl - s < kk && kk <= incl);
  const int tl = __ffs(hit) - 1;  // exactly one lane (kk <= total count)
  const uint32_t excl_tl = __shfl_sync(0xffffffffu, incl - s, tl);
  // lane l takes bins top - 2l and top - 2l - 1 of lane tl's range
  const int top = kBins - 64 * tl - 1;
  const uint32_t c0 = hist[top - 2 * lane], c1 = hist[top - 2 * lane - 1];
  const uint32_t pair = c0 + c1;
  uint32_t pin = pair;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, pin, d);
    if (lane >= d) pin += x;
  }
  const uint32_t before = excl_tl + pin - pair;  // keys in bins above this pair
  const uint32_t hit2 = __ballot_sync(0xffffffffu, before < kk && kk <= before + pair);
  if (lane == __ffs(hit2) - 1) {
    if (before + c0 >= kk) {
      *sel_digit = (uint32_t)(top - 2 * lane);
      *sel_above = before;
    } else {
      *sel_digit = (uint32_t)(top - 2 * lane - 1);
      *sel_above = before + c0;
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
        const int64_t nb = (n4 + 4 * kTopkThreads - 1) / (4 * kTopkThreads);
        for (int64_t bi = 0; bi < nb; ++bi) {
          const int64_t b = bi * 4 * kTopkThreads + tid;
          float4 x[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int64_t j = b + u * kTopkThreads;
            x[u] = j < n4 ? __ldg(row4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int64_t j = b + u * kTopkThreads;
            const bool in = j < n4;
            const uint32_t k4[4] = {order_key(x[u].x), order_key(x[u].y),
                                    order_key(x[u].z), order_key(x[u].w)};
            if (cached && in)
              *reinterpret_cast<uint4*>(cache + 4 * j) = make_uint4(k4[0], k4[1], k4[2], k4[3]);
            if (in) {
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
    // contiguous segment of whole 128-key blocks (lane l: keys 4l .. 4l+3
    // of a block): count, one block-wide exclusive scan, then write with a
    // warp scan per block.
    const uint32_t T = prefix;
    const float4* row4 = reinterpret_cast<const float4*>(row);
    auto keys4 = [&](int64_t i, int64_t lim, uint32_t (&kq)[4]) {
      if (i + 3 < lim && (cached || vec)) {
        if (cached) {
          const uint4 c4 = *reinterpret_cast<const uint4*>(cache + i);
          kq[0] = c4.x; kq[1] = c4.y; kq[2] = c4.z; kq[3] = c4.w;
        } else {
          const float4 f4 = __ldg(row4 + (i >> 2));
          kq[0] = order_key(f4.x); kq[1] = order_key(f4.y);
          kq[2] = order_key(f4.z); kq[3] = order_key(f4.w);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          kq[e] = i + e < lim ? (cached ? cache[i + e] : order_key(__ldg(row + i + e))) : 0u;
      }
    };
    const int64_t nblk = (n + 127) / 128;
    const int64_t bpw = (nblk + kTopkWarps - 1) / kTopkWarps;
    const int64_t b0 = warp * bpw * 128;
    const int64_t b1 = b0 + bpw * 128 < n ? b0 + bpw * 128 : n;
    uint32_t cg = 0u, ct = 0u;
    for (int64_t i0 = b0; i0 < b1; i0 += 128) {
      const int64_t i = i0 + 4 * lane;
      uint32_t kq[4];
      keys4(i, b1, kq);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool in = i + e < b1;
        cg += in && kq[e] > T;
        ct += in && kq[e] == T;
      }
    }
    cg = __reduce_add_sync(0xffffffffu, cg);
    ct = __reduce_add_sync(0xffffffffu, ct);
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
    for (int64_t i0 = b0; i0 < b1; i0 += 128) {
      if (t_base >= kk && g_base + kk >= (uint32_t)K_p) break;  // warp-uniform
      const int64_t i = i0 + 4 * lane;
      uint32_t kq[4];
      keys4(i, b1, kq);
      uint32_t gl = 0u, tl = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool in = i + e < b1;
        gl += in && kq[e] > T;
        tl += in && kq[e] == T;
      }
      // (above, ties) counts packed as hi/lo 16 bits: at most 128 each
      const uint32_t v = (gl << 16) | tl;
      uint32_t incl = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint32_t x = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += x;
      }
      const uint32_t excl = incl - v;
      uint32_t g_before = g_base + (excl >> 16), t_before = t_base + (excl & 0xFFFFu);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (i + e >= b1) break;
        // (positions are < K_p by construction; the guard keeps a corrupted
        // row from writing into its neighbour)
        if (kq[e] > T) {
          const uint32_t pos = g_before + min(t_before, kk);
          if (pos < (uint32_t)K_p) o[pos] = (int32_t)(i + e);
          ++g_before;
        } else if (kq[e] == T) {
          if (t_before < kk && g_before + t_before < (uint32_t)K_p)
            o[g_before + t_before] = (int32_t)(i + e);
          ++t_before;
        }
      }
      const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
      g_base += tot >> 16;
      t_base += tot & 0xFFFFu;
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
