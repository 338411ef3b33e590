// attn_fwd.cu -- causal sparse attention forward over the selected keys.
//
// "the attention reads only those 2048 tokens, so attention cost grows
// linearly" ("Scaling Training to 1M Token Context on GLM-5.3-Flash",
// section "DeepSeek Sparse Attention (DSA) Optimizations"); NoPE q/k and the
// 2,051-key variant (section "Making Sparse Attention Actually Sparse").
// One K row and one V row per token are shared by every query head, so the
// keys of query t are gathered ONCE and reused by all of its heads: the
// heads form the M dimension of each tensor-core tile.
//
// Per CTA: one query (x one block of <= 64 heads) at a time, persistent.
//   Q[t] (16*HG heads x D) resident in shared memory;
//   key tiles of 32 gathered K and V rows, double-buffered with cp.async;
//   S = Q K^T and O += P V on warp tensor cores (bf16 in, fp32 accumulate);
//   online softmax in base 2; LSE stored in natural log.
// Warp (hg, half): heads 16*hg..16*hg+15; keys 16*half.. of each tile for S,
// value columns half*D/2.. for O.  The two warps of a head group exchange
// row maxima and P through shared memory.
#include "attn_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kNK = 32;          // keys per tile
constexpr int kPStride = 80;     // bytes per P row (64 + 16 pad: no conflicts)

template <int D, int HG>
struct FwdCfg {
  static constexpr int kThreads = 64 * HG;
  static constexpr int kRows = 16 * HG;
  static constexpr uint32_t kQBytes = kRows * D * 2;
  static constexpr uint32_t kKVBytes = kNK * D * 2;
  static constexpr uint32_t kPBytes = kRows * kPStride;
  static uint32_t smem(int K_p, int n_loc) {
    const int slots = ((4 * K_p + n_loc) + kNK - 1) / kNK * kNK;
    return kQBytes + 4 * kKVBytes + kPBytes + 2 * kRows * 4 + 16 + slots * 4;
  }
};

template <int D, int HG>
__global__ void __launch_bounds__(64 * HG, 1)
    attn_fwd_kernel(const __nv_bfloat16* __restrict__ q,
                    const __nv_bfloat16* __restrict__ k,
                    const __nv_bfloat16* __restrict__ v,
                    const int32_t* __restrict__ idx, __nv_bfloat16* __restrict__ o,
                    float* __restrict__ lse, int64_t S, int H, int K_p, int n_loc,
                    float scale_log2, int n_hblk, uint32_t* status) {
  using C = FwdCfg<D, HG>;
  constexpr int kChunks = D / 8;  // 16-byte chunks per row
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* pQ = smem;
  uint8_t* pK = pQ + C::kQBytes;               // 2 buffers
  uint8_t* pV = pK + 2 * C::kKVBytes;          // 2 buffers
  uint8_t* pP = pV + 2 * C::kKVBytes;
  float* mx = reinterpret_cast<float*>(pP + C::kPBytes);  // [2][kRows]
  int* scratch2 = reinterpret_cast<int*>(mx + 2 * C::kRows);
  int32_t* toks = scratch2 + 4;
  const uint32_t sQ = smem_u32(pQ), sK = smem_u32(pK), sV = smem_u32(pV),
                 sP = smem_u32(pP);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hg = warp % HG, half = warp / HG;
  const int g = lane >> 2, cq = lane & 3;
  const int64_t n_items = S * n_hblk;

  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int64_t t = S - 1 - item / n_hblk;
    const int hb = (int)(item % n_hblk);
    const int n = build_key_list(idx + t * K_p, t, K_p, n_loc, kNK, toks,
                                 scratch2, status);
    const int ntiles = (n + kNK - 1) / kNK;

    // rows of this CTA: heads hb*64 + 0 .. kRows-1 (beyond H: zero, unused)
    auto issue_q = [&]() {
      for (int e = tid; e < C::kRows * kChunks; e += C::kThreads) {
        const int r = e / kChunks, ch = e % kChunks;
        const int h = hb * 64 + r;
        const bool ok = h < H;
        const __nv_bfloat16* src = q + ((t * H + (ok ? h : 0)) * (int64_t)D + ch * 8);
        cp_async16(sQ + swz<D>(r, ch), src, ok ? 16u : 0u);
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

    float oacc[D / 16][4];
#pragma unroll
    for (int i = 0; i < D / 16; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    if (ntiles > 0) {
      issue_q();
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

      // ---- S = Q K^T for heads hg*16.., keys half*16..half*16+15
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int arow = hg * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
      const int krow = half * 16 + (lane & 7) + 8 * (lane >> 4);
#pragma unroll 8
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(sQ + swz<D>(arow, ks * 2 + (lane >> 4)), a0, a1, a2, a3);
        ldsm_x4(kb + swz<D>(krow, ks * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
        mma16816(sacc[0], a0, a1, a2, a3, b0, b1);
        mma16816(sacc[1], a0, a1, a2, a3, b2, b3);
      }
      // ---- mask, scale, row max over this warp's 16 keys
      float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int slot = j * kNK + half * 16 + nt * 8 + 2 * cq + (e & 1);
          float s = sacc[nt][e] * scale_log2;
          if (toks[slot] < 0) s = -INFINITY;
          sacc[nt][e] = s;
          tmax[e >> 1] = fmaxf(tmax[e >> 1], s);
        }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 1));
        tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 2));
      }
      if (cq == 0) {
        mx[half * C::kRows + hg * 16 + g] = tmax[0];
        mx[half * C::kRows + hg * 16 + g + 8] = tmax[1];
      }
      named_sync(1 + hg, 64);
      float alpha[2], muse[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float other = mx[(1 - half) * C::kRows + hg * 16 + g + 8 * r];
        const float mnew = fmaxf(m_run[r], fmaxf(tmax[r], other));
        muse[r] = mnew == -INFINITY ? 0.f : mnew;
        alpha[r] = exp2f(m_run[r] - muse[r]);
        m_run[r] = mnew;
      }
      // ---- P = exp2(s - m), row sums, P -> shared (bf16)
      float psum[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const float p0 = exp2f(sacc[nt][0] - muse[0]);
        const float p1 = exp2f(sacc[nt][1] - muse[0]);
        const float p2 = exp2f(sacc[nt][2] - muse[1]);
        const float p3 = exp2f(sacc[nt][3] - muse[1]);
        psum[0] += p0 + p1;
        psum[1] += p2 + p3;
        const int col = half * 16 + nt * 8 + 2 * cq;
        *reinterpret_cast<uint32_t*>(pP + (hg * 16 + g) * kPStride + col * 2) =
            pack_bf16(p0, p1);
        *reinterpret_cast<uint32_t*>(pP + (hg * 16 + g + 8) * kPStride + col * 2) =
            pack_bf16(p2, p3);
      }
      l_run[0] = l_run[0] * alpha[0] + psum[0];
      l_run[1] = l_run[1] * alpha[1] + psum[1];
#pragma unroll
      for (int i = 0; i < D / 16; ++i) {
        oacc[i][0] *= alpha[0];
        oacc[i][1] *= alpha[0];
        oacc[i][2] *= alpha[1];
        oacc[i][3] *= alpha[1];
      }
      named_sync(1 + hg, 64);
      // ---- O[:, half*D/2 ..] += P V
      const int prow = hg * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
      for (int kk = 0; kk < kNK / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(sP + prow * kPStride + (kk * 2 + (lane >> 4)) * 16, a0, a1, a2, a3);
        const int vrow = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
        for (int np = 0; np < D / 32; ++np) {
          uint32_t b0, b1, b2, b3;
          const int ch = (half * (D / 2) + np * 16) / 8 + (lane >> 4);
          ldsm_x4_t(vb + swz<D>(vrow, ch), b0, b1, b2, b3);
          mma16816(oacc[2 * np], a0, a1, a2, a3, b0, b1);
          mma16816(oacc[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }

    // ---- normalise, store O (bf16) and LSE
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
    }
    __syncthreads();
    if (cq == 0) {
      mx[half * C::kRows + hg * 16 + g] = l_run[0];
      mx[half * C::kRows + hg * 16 + g + 8] = l_run[1];
    }
    __syncthreads();
    float inv[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float l = l_run[r] + mx[(1 - half) * C::kRows + hg * 16 + g + 8 * r];
      inv[r] = l > 0.f ? 1.f / l : 0.f;
      const int h = hb * 64 + hg * 16 + g + 8 * r;
      if (half == 0 && cq == 0 && h < H)
        lse[t * H + h] = l > 0.f ? (m_run[r] + log2f(l)) * kLn2 : -INFINITY;
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int h = hb * 64 + hg * 16 + g + 8 * r;
      if (h >= H) continue;
      __nv_bfloat16* orow = o + (t * H + h) * (int64_t)D + half * (D / 2);
#pragma unroll
      for (int i = 0; i < D / 16; ++i) {
        *reinterpret_cast<uint32_t*>(orow + i * 8 + 2 * cq) =
            pack_bf16(oacc[i][2 * r] * inv[r], oacc[i][2 * r + 1] * inv[r]);
      }
    }
    __syncthreads();
  }
}

template <int D, int HG>
cudaError_t launch_fwd_t(const LaunchCtx& c, const AttnShape& s,
                         const __nv_bfloat16* q, const __nv_bfloat16* k,
                         const __nv_bfloat16* v, const int32_t* idx,
                         __nv_bfloat16* o, float* lse) {
  using C = FwdCfg<D, HG>;
  const uint32_t smem = C::smem(s.K_p, s.n_loc);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, HG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_fwd_kernel<D, HG>,
                                                    C::kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int n_hblk = (s.H + 63) / 64;
  const int64_t items = s.S * n_hblk;
  int64_t grid = (int64_t)c.num_sms * per_sm;
  if (grid > items) grid = items;
  attn_fwd_kernel<D, HG><<<(unsigned)grid, C::kThreads, smem, c.stream>>>(
      q, k, v, idx, o, lse, s.S, s.H, s.K_p, s.n_loc, s.scale * kLog2e, n_hblk,
      c.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const LaunchCtx& c, const AttnShape& s,
                            const __nv_bfloat16* q, const __nv_bfloat16* k,
                            const __nv_bfloat16* v, const int32_t* idx,
                            __nv_bfloat16* o, float* lse) {
  const int hg = s.H >= 64 ? 4 : (s.H + 15) / 16;
#define DSA_FWD_CASE(DD, HH) \
  if (s.D == DD && hg == HH) return launch_fwd_t<DD, HH>(c, s, q, k, v, idx, o, lse);
  DSA_FWD_CASE(64, 1) DSA_FWD_CASE(64, 2) DSA_FWD_CASE(64, 3) DSA_FWD_CASE(64, 4)
  DSA_FWD_CASE(128, 1) DSA_FWD_CASE(128, 2) DSA_FWD_CASE(128, 3) DSA_FWD_CASE(128, 4)
  DSA_FWD_CASE(256, 1) DSA_FWD_CASE(256, 2) DSA_FWD_CASE(256, 3) DSA_FWD_CASE(256, 4)
  DSA_FWD_CASE(512, 1) DSA_FWD_CASE(512, 2) DSA_FWD_CASE(512, 3) DSA_FWD_CASE(512, 4)
#undef DSA_FWD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace dsa
