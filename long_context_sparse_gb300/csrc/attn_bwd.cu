// attn_bwd.cu -- backward of the sparse attention (delta, dQ/dK/dV).
//
// Every backward GEMM depends on the attention weights A ("MTraining:
// Efficient Distributed Training for Ultra-Long Contexts via Dynamic Sparse
// Attention", section 3.2, Eq. 1), so the backward walks exactly the keys the
// forward selected ("Scaling Training to 1M Token Context on GLM-5.3-Flash",
// section "DeepSeek Sparse Attention (DSA) Optimizations") and recomputes
// P = exp(scale q.k - LSE) from the stored LSE:
//   dP = dO V^T, dS = P (dP - delta), dQ = scale dS K   (query-local)
//   dK += scale dS^T Q, dV += P^T dO                     (scattered)
// K and V are shared by all heads, so one gathered key tile serves every
// head of the query (heads = the M dimension of the dQ tile and the K
// dimension of the dK/dV tiles).  dK/dV rows are accumulated in fp32 with
// vector reductions into a workspace and rounded to bf16 once at the end.
#include "attn_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kNK = 16;       // keys per tile
constexpr int kPStride = 48;  // bytes per P / dS row (32 + 16 pad)

template <int D, int HG>
struct BwdCfg {
  static constexpr int kThreads = 64 * HG;
  static constexpr int kRows = 16 * HG;
  static constexpr uint32_t kQBytes = kRows * D * 2;
  static constexpr uint32_t kKVBytes = kNK * D * 2;
  static constexpr uint32_t kPBytes = kRows * kPStride;
  static uint32_t smem(int K_p, int n_loc) {
    const int slots = ((4 * K_p + n_loc) + kNK - 1) / kNK * kNK;
    return 2 * kQBytes + 4 * kKVBytes + 2 * kPBytes + 2 * kRows * 4 + 16 +
           slots * 4;
  }
};

// ------------------------------------------------------- a7 preprocess
// delta[t,h] = sum_d dO[t,h,d] O[t,h,d] (fp32), one warp per (t,h) row.
__global__ void __launch_bounds__(256) bwd_delta_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dO,
    float* __restrict__ delta, int64_t n_rows, int D) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t r = w0; r < n_rows; r += nw) {
    const uint4* a = reinterpret_cast<const uint4*>(o + r * D);
    const uint4* b = reinterpret_cast<const uint4*>(dO + r * D);
    float acc = 0.f;
    for (int i = lane; i < D / 8; i += 32) {
      const uint4 x = __ldg(a + i), y = __ldg(b + i);
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc = fmaf(bf16_lo(xs[j]), bf16_lo(ys[j]), acc);
        acc = fmaf(bf16_hi(xs[j]), bf16_hi(ys[j]), acc);
      }
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) delta[r] = acc;
  }
}

__global__ void __launch_bounds__(256) zero_kernel(float4* __restrict__ a, int64_t n4) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x)
    a[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void __launch_bounds__(256) finalize_kernel(const float4* __restrict__ a,
                                                       uint2* __restrict__ out,
                                                       int64_t n4) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 x = __ldg(a + i);
    out[i] = make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
  }
}

// ------------------------------------------------------------ a8 main
template <int D, int HG>
__global__ void __launch_bounds__(64 * HG, 1)
    attn_bwd_kernel(const __nv_bfloat16* __restrict__ q,
                    const __nv_bfloat16* __restrict__ k,
                    const __nv_bfloat16* __restrict__ v,
                    const __nv_bfloat16* __restrict__ dO,
                    const float* __restrict__ lse, const float* __restrict__ delta,
                    const int32_t* __restrict__ idx, __nv_bfloat16* __restrict__ dq,
                    float* __restrict__ dk_acc, float* __restrict__ dv_acc,
                    int64_t S, int H, int K_p, int n_loc, float scale,
                    int n_hblk, uint32_t* status) {
  using C = BwdCfg<D, HG>;
  constexpr int kChunks = D / 8;
  constexpr int kNW = 2 * HG;           // warps
  constexpr int kDW = D / kNW;          // dK/dV columns per warp
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* pQ = smem;
  uint8_t* pG = pQ + C::kQBytes;        // dO
  uint8_t* pK = pG + C::kQBytes;        // 2 buffers
  uint8_t* pV = pK + 2 * C::kKVBytes;   // 2 buffers
  uint8_t* pP = pV + 2 * C::kKVBytes;
  uint8_t* pS = pP + C::kPBytes;        // dS
  float* lse2_s = reinterpret_cast<float*>(pS + C::kPBytes);
  float* delta_s = lse2_s + C::kRows;
  int* scratch2 = reinterpret_cast<int*>(delta_s + C::kRows);
  int32_t* toks = scratch2 + 4;
  const uint32_t sQ = smem_u32(pQ), sG = smem_u32(pG), sK = smem_u32(pK),
                 sV = smem_u32(pV), sP = smem_u32(pP), sS = smem_u32(pS);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hg = warp % HG, half = warp / HG;
  const int g = lane >> 2, cq = lane & 3;
  const float c2 = scale * kLog2e;
  const int64_t n_items = S * n_hblk;

  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int64_t t = S - 1 - item / n_hblk;
    const int hb = (int)(item % n_hblk);
    const int n = build_key_list(idx + t * K_p, t, K_p, n_loc, kNK, toks,
                                 scratch2, status);
    const int ntiles = (n + kNK - 1) / kNK;

    for (int r = tid; r < C::kRows; r += C::kThreads) {
      const int h = hb * 64 + r;
      lse2_s[r] = h < H ? __ldg(lse + t * H + h) * kLog2e : INFINITY;
      delta_s[r] = h < H ? __ldg(delta + t * H + h) : 0.f;
    }
    auto issue_rows = [&]() {
      for (int e = tid; e < C::kRows * kChunks; e += C::kThreads) {
        const int r = e / kChunks, ch = e % kChunks;
        const int h = hb * 64 + r;
        const bool ok = h < H;
        const int64_t off = (t * H + (ok ? h : 0)) * (int64_t)D + ch * 8;
        cp_async16(sQ + swz<D>(r, ch), q + off, ok ? 16u : 0u);
        cp_async16(sG + swz<D>(r, ch), dO + off, ok ? 16u : 0u);
      }
    };
    auto issue_kv = [&](int tile, int buf) {
      for (int e = tid; e < kNK * kChunks; e += C::kThreads) {
        const int r = e / kChunks, ch = e % kChunks;
        const int32_t tok = toks[tile * kNK + r];
        const int64_t row = tok >= 0 ? tok : 0;
        const uint32_t nb = tok >= 0 ? 16u : 0u;
        const uint32_t off = buf * C::kKVBytes + swz<D>(r, ch);
        cp_async16(sK + off, k + row * D + ch * 8, nb);
        cp_async16(sV + off, v + row * D + ch * 8, nb);
      }
    };

    float dqacc[D / 16][4];
#pragma unroll
    for (int i = 0; i < D / 16; ++i) dqacc[i][0] = dqacc[i][1] = dqacc[i][2] = dqacc[i][3] = 0.f;

    if (ntiles > 0) {
      issue_rows();
      issue_kv(0, 0);
      cp_async_commit();
    }
    for (int j = 0; j < ntiles; ++j) {
      cp_async_wait<0>();
      __syncthreads();
      if (j + 1 < ntiles) {
        issue_kv(j + 1, (j + 1) & 1);
        cp_async_commit();
      }
      const uint32_t kb = sK + (j & 1) * C::kKVBytes;
      const uint32_t vb = sV + (j & 1) * C::kKVBytes;

      // ---- S = Q K^T, dP = dO V^T: heads hg*16.., keys half*8..half*8+7
      float sacc[4] = {0.f, 0.f, 0.f, 0.f}, pacc[4] = {0.f, 0.f, 0.f, 0.f};
      const int arow = hg * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
      const int krow = half * 8 + (lane & 7);
#pragma unroll 4
      for (int k2 = 0; k2 < D / 32; ++k2) {
        uint32_t b0, b1, b2, b3, e0, e1, e2, e3;
        ldsm_x4(kb + swz<D>(krow, k2 * 4 + (lane >> 3)), b0, b1, b2, b3);
        ldsm_x4(vb + swz<D>(krow, k2 * 4 + (lane >> 3)), e0, e1, e2, e3);
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int ch = (k2 * 2 + h2) * 2 + (lane >> 4);
          uint32_t a0, a1, a2, a3, g0, g1, g2, g3;
          ldsm_x4(sQ + swz<D>(arow, ch), a0, a1, a2, a3);
          ldsm_x4(sG + swz<D>(arow, ch), g0, g1, g2, g3);
          if (h2 == 0) {
            mma16816(sacc, a0, a1, a2, a3, b0, b1);
            mma16816(pacc, g0, g1, g2, g3, e0, e1);
          } else {
            mma16816(sacc, a0, a1, a2, a3, b2, b3);
            mma16816(pacc, g0, g1, g2, g3, e2, e3);
          }
        }
      }
      // ---- P, dS -> shared (bf16)
      {
        const int r0 = hg * 16 + g, r1 = r0 + 8;
        const int col = half * 8 + 2 * cq;
        const bool m0 = toks[j * kNK + col] < 0, m1 = toks[j * kNK + col + 1] < 0;
        const float l0 = lse2_s[r0], l1 = lse2_s[r1];
        const float d0 = delta_s[r0], d1 = delta_s[r1];
        const float p00 = m0 ? 0.f : exp2f(sacc[0] * c2 - l0);
        const float p01 = m1 ? 0.f : exp2f(sacc[1] * c2 - l0);
        const float p10 = m0 ? 0.f : exp2f(sacc[2] * c2 - l1);
        const float p11 = m1 ? 0.f : exp2f(sacc[3] * c2 - l1);
        *reinterpret_cast<uint32_t*>(pP + r0 * kPStride + col * 2) = pack_bf16(p00, p01);
        *reinterpret_cast<uint32_t*>(pP + r1 * kPStride + col * 2) = pack_bf16(p10, p11);
        *reinterpret_cast<uint32_t*>(pS + r0 * kPStride + col * 2) =
            pack_bf16(p00 * (pacc[0] - d0), p01 * (pacc[1] - d0));
        *reinterpret_cast<uint32_t*>(pS + r1 * kPStride + col * 2) =
            pack_bf16(p10 * (pacc[2] - d1), p11 * (pacc[3] - d1));
      }
      __syncthreads();
      // ---- dQ[hg rows, half*D/2 ..] += dS K
      {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(sS + arow * kPStride + (lane >> 4) * 16, a0, a1, a2, a3);
        const int vrow = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
        for (int np = 0; np < D / 32; ++np) {
          uint32_t b0, b1, b2, b3;
          const int ch = (half * (D / 2) + np * 16) / 8 + (lane >> 4);
          ldsm_x4_t(kb + swz<D>(vrow, ch), b0, b1, b2, b3);
          mma16816(dqacc[2 * np], a0, a1, a2, a3, b0, b1);
          mma16816(dqacc[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      // ---- dK (dS^T Q) and dV (P^T dO) for this warp's kDW columns
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t sA = which == 0 ? sS : sP;
        const uint32_t sB = which == 0 ? sQ : sG;
        float acc[kDW / 8][4];
#pragma unroll
        for (int i = 0; i < kDW / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
        for (int kh = 0; kh < HG; ++kh) {
          uint32_t a0, a1, a2, a3;
          const int hrow = kh * 16 + (lane & 7) + 8 * (lane >> 4);
          ldsm_x4_t(sA + hrow * kPStride + ((lane >> 3) & 1) * 16, a0, a1, a2, a3);
          const int brow = kh * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
          for (int np = 0; np < kDW / 16; ++np) {
            uint32_t b0, b1, b2, b3;
            const int ch = (warp * kDW + np * 16) / 8 + (lane >> 4);
            ldsm_x4_t(sB + swz<D>(brow, ch), b0, b1, b2, b3);
            mma16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
            mma16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
          }
        }
        float* dst = which == 0 ? dk_acc : dv_acc;
        const float f = which == 0 ? scale : 1.f;
        const int32_t tok0 = toks[j * kNK + g], tok1 = toks[j * kNK + g + 8];
#pragma unroll
        for (int i = 0; i < kDW / 8; ++i) {
          const int col = warp * kDW + i * 8 + 2 * cq;
          if (tok0 >= 0) red_add_v2(dst + (int64_t)tok0 * D + col, f * acc[i][0], f * acc[i][1]);
          if (tok1 >= 0) red_add_v2(dst + (int64_t)tok1 * D + col, f * acc[i][2], f * acc[i][3]);
        }
      }
    }

    // ---- dQ = scale * acc -> bf16 (zero for empty key sets)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int h = hb * 64 + hg * 16 + g + 8 * r;
      if (h >= H) continue;
      __nv_bfloat16* row = dq + (t * H + h) * (int64_t)D + half * (D / 2);
#pragma unroll
      for (int i = 0; i < D / 16; ++i)
        *reinterpret_cast<uint32_t*>(row + i * 8 + 2 * cq) =
            pack_bf16(dqacc[i][2 * r] * scale, dqacc[i][2 * r + 1] * scale);
    }
    __syncthreads();
  }
}

template <int D, int HG>
cudaError_t launch_bwd_t(const LaunchCtx& c, const AttnShape& s,
                         const __nv_bfloat16* q, const __nv_bfloat16* k,
                         const __nv_bfloat16* v, const __nv_bfloat16* dO,
                         const float* lse, const float* delta, const int32_t* idx,
                         __nv_bfloat16* dq, float* dk_acc, float* dv_acc) {
  using C = BwdCfg<D, HG>;
  const uint32_t smem = C::smem(s.K_p, s.n_loc);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D, HG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_bwd_kernel<D, HG>,
                                                    C::kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int n_hblk = (s.H + 63) / 64;
  const int64_t items = s.S * n_hblk;
  int64_t grid = (int64_t)c.num_sms * per_sm;
  if (grid > items) grid = items;
  attn_bwd_kernel<D, HG><<<(unsigned)grid, C::kThreads, smem, c.stream>>>(
      q, k, v, dO, lse, delta, idx, dq, dk_acc, dv_acc, s.S, s.H, s.K_p, s.n_loc,
      s.scale, n_hblk, c.status);
  return cudaGetLastError();
}

int64_t grid_for(const LaunchCtx& c, int64_t n) {
  int64_t g = (n + 255) / 256;
  const int64_t cap = (int64_t)c.num_sms * 8;
  return g < 1 ? 1 : (g > cap ? cap : g);
}

}  // namespace

cudaError_t launch_attn_bwd_pre(const LaunchCtx& c, const AttnShape& s,
                                const __nv_bfloat16* o, const __nv_bfloat16* dO,
                                float* delta, float* dk_acc, float* dv_acc) {
  const int64_t rows = s.S * s.H;
  bwd_delta_kernel<<<(unsigned)grid_for(c, rows * 32), 256, 0, c.stream>>>(
      o, dO, delta, rows, s.D);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t n4 = s.S * s.D / 4;
  zero_kernel<<<(unsigned)grid_for(c, n4), 256, 0, c.stream>>>(
      reinterpret_cast<float4*>(dk_acc), n4);
  zero_kernel<<<(unsigned)grid_for(c, n4), 256, 0, c.stream>>>(
      reinterpret_cast<float4*>(dv_acc), n4);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const LaunchCtx& c, const AttnShape& s,
                            const __nv_bfloat16* q, const __nv_bfloat16* k,
                            const __nv_bfloat16* v, const __nv_bfloat16* dO,
                            const float* lse, const float* delta,
                            const int32_t* idx, __nv_bfloat16* dq, float* dk_acc,
                            float* dv_acc) {
  const int hg = s.H >= 64 ? 4 : (s.H + 15) / 16;
#define DSA_BWD_CASE(DD, HH)                                                     \
  if (s.D == DD && hg == HH)                                                     \
    return launch_bwd_t<DD, HH>(c, s, q, k, v, dO, lse, delta, idx, dq, dk_acc, \
                                dv_acc);
  DSA_BWD_CASE(64, 1) DSA_BWD_CASE(64, 2) DSA_BWD_CASE(64, 3) DSA_BWD_CASE(64, 4)
  DSA_BWD_CASE(128, 1) DSA_BWD_CASE(128, 2) DSA_BWD_CASE(128, 3) DSA_BWD_CASE(128, 4)
  DSA_BWD_CASE(256, 1) DSA_BWD_CASE(256, 2) DSA_BWD_CASE(256, 3) DSA_BWD_CASE(256, 4)
  DSA_BWD_CASE(512, 1) DSA_BWD_CASE(512, 2) DSA_BWD_CASE(512, 3) DSA_BWD_CASE(512, 4)
#undef DSA_BWD_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_bwd_finalize(const LaunchCtx& c, const AttnShape& s,
                                     const float* dk_acc, const float* dv_acc,
                                     __nv_bfloat16* dk, __nv_bfloat16* dv) {
  const int64_t n4 = s.S * s.D / 4;
  finalize_kernel<<<(unsigned)grid_for(c, n4), 256, 0, c.stream>>>(
      reinterpret_cast<const float4*>(dk_acc), reinterpret_cast<uint2*>(dk), n4);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  finalize_kernel<<<(unsigned)grid_for(c, n4), 256, 0, c.stream>>>(
      reinterpret_cast<const float4*>(dv_acc), reinterpret_cast<uint2*>(dv), n4);
  return cudaGetLastError();
}

}  // namespace dsa
