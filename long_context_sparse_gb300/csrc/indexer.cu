// indexer.cu -- the DSA lightning indexer on 5th-generation tensor cores.
//
//   I[t,p] = sum_h w[t,h] * max(0, q_idx[t,h,:] . k_pool[p,:])
//
// "A lightweight indexer ... scores every query against every earlier pool
// of 4 tokens" -- the dense, quadratic part of DSA ("Scaling Training to 1M
// Token Context on GLM-5.3-Flash", section "DeepSeek Sparse Attention (DSA)
// Optimizations"), run one chunk of queries at a time (section "Splitting
// the DSA Indexer / Over Time: Chunking").
//
// GEMM mapping (one CTA per SM, persistent over tiles):
//   M = 128 pools      -> TMEM lanes; A = k_pool tile [128 x D_I], K-major
//   N = 256 columns    -> (query, head) pairs, 256/H_I queries x H_I heads;
//                         B = q_idx rows [256 x D_I], K-major
//   K = D_I            -> D_I/16 tcgen05.mma (kind::f16, bf16 -> fp32)
// Each epilogue thread owns one pool (one TMEM lane) and a quarter of the
// tile's columns: ReLU, times w[t,h], summed over heads in fp32 (up to four
// independent chains of packed fp32x2 FMAs, the TMEM load of the next 16
// columns in flight), then one coalesced store per query.
// No cross-lane traffic.
//
// Warp roles (608 threads): warp 0 TMA producer, warps 1-2 MMA issuers
// (alternate tiles; warp 1 also allocates TMEM), warps 3-18 epilogue (four
// per TMEM lane quadrant, one per quarter of the columns).  The epilogue's ALU work per tile fits under the
// MMA time only when four warps per SM sub-partition hide each other's
// latencies (with two, the tile took 1.8x its MMA time); the head weights
// of the N tile sit in shared memory and are read as broadcast 16-byte
// loads, which leaves the warps' registers for the accumulator values.  A
// tiles stream through a 4-stage TMA ring;
// the B tile stays resident while consecutive tiles share it; accumulators
// are double-buffered in TMEM (2 x 256 columns) so the epilogue of one tile
// overlaps the MMAs of the next.
#include "index_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kBM = 128;  // pools per tile
constexpr int kBN = 256;  // (query, head) columns per tile
constexpr int kEpiWarps = 16;            // four per SM sub-partition
constexpr int kEpiWarp0 = 3;             // warps 0 TMA, 1-2 MMA issuers
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
constexpr int kEpiCols = kBN / (kEpiWarps / 4);  // columns per epilogue warp
// registers: the fullest SM sub-partition holds ceil(19 / 4) = 5 warps
constexpr int kMaxReg = (16384 / (((kThreads / 32) + 3) / 4 * 32)) & ~7;
static_assert(kMaxReg == 96, "register budget");

template <int DI>
struct IdxCfg {
  static constexpr int KB = DI / 64;                 // 128-byte k-boxes
  static constexpr int kStages = DI == 64 ? 8 : 4;
  static constexpr uint32_t kABytes = kBM * DI * 2;  // one pool tile
  static constexpr uint32_t kBBytes = kBN * DI * 2;  // one query tile
  // + barriers (256) + weights of two N tiles (2 x kBN floats) + alignment
  static constexpr uint32_t kSmem = kBBytes + kStages * kABytes + 256 + 8 * kBN + 1024;
};

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity,
                                           uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
  return true;
}

template <int HI, int DI>
__global__ void __maxnreg__(kMaxReg)
    indexer_kernel(const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap k_map,
                   const float* __restrict__ w, int64_t t0, int64_t q0,
                   int64_t rows, int64_t p_lim, float* __restrict__ scores, int64_t ld,
                   int n_ptiles, int64_t n_items, uint32_t* status,
                   uint64_t timeout_ns) {
  using C = IdxCfg<DI>;
  constexpr int QT = kBN / HI;  // queries per N tile
  constexpr uint32_t IDESC = idesc_bf16(kBM, kBN, 0, 0);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sB = base;
  const uint32_t sA = base + C::kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + C::kBBytes + C::kStages * C::kABytes);
  // head weights of the current and the previous N tile: [2][kBN]
  float* wsm = reinterpret_cast<float*>(gbase + C::kBBytes + C::kStages * C::kABytes + 256);
  // barrier slots
  const uint32_t bar0 = smem_u32(bars);
  auto a_full = [&](int s) { return bar0 + 8u * s; };
  auto a_empty = [&](int s) { return bar0 + 8u * (C::kStages + s); };
  const uint32_t b_full = bar0 + 8u * (2 * C::kStages);
  const uint32_t b_empty = b_full + 8u;
  auto acc_full = [&](int a) { return b_full + 16u + 8u * a; };
  auto acc_empty = [&](int a) { return b_full + 32u + 8u * a; };
  const uint32_t done_bar = b_full + 48u;      // [2], one per MMA issuer: slots +48, +72
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(bars + 2 * C::kStages + 7);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::kStages + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Waiter W{abort_flag, status, timeout_ns};

  const int64_t beg = (int64_t)blockIdx.x * n_items / gridDim.x;
  const int64_t end = (int64_t)(blockIdx.x + 1) * n_items / gridDim.x;
  // item = nt * n_ptiles + pt (N tile, pool tile); every role steps the
  // pair instead of dividing a 64-bit item number per tile (an emulated
  // division costs several hundred cycles on the epilogue's critical path)
  const int64_t nt_beg = beg / n_ptiles;
  const int pt_beg = (int)(beg - nt_beg * n_ptiles);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(a_full(s), 1);
      mbar_init(a_empty(s), 1);
    }
    mbar_init(b_full, 1);
    mbar_init(b_empty, 2);  // both MMA issuers release each B tile
    for (int a = 0; a < 2; ++a) {
      mbar_init(acc_full(a), 1);
      mbar_init(acc_empty(a), kEpiWarps);
    }
    mbar_init(done_bar, 1);
    mbar_init(done_bar + 24u, 1);
    *abort_flag = 0u;
    fence_mbar_init();
    prefetch_tensormap(&q_map);
    prefetch_tensormap(&k_map);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int64_t it = 0;
      int bcount = 0;
      int64_t cur_nt = -1;
      int64_t nt = nt_beg;
      int pt = pt_beg;
      for (int64_t item = beg; item < end; ++item, pt = pt + 1 == n_ptiles ? 0 : pt + 1,
                   nt += pt == 0 ? 1 : 0) {
        if (nt != cur_nt) {
          if (!W.wait(b_empty, (bcount & 1) ^ 1)) break;
          mbar_expect_tx(b_full, C::kBBytes);
          const int32_t row = (int32_t)((t0 - q0) * HI + nt * kBN);
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_2d(sB + kb * (kBN * 128), &q_map, kb * 64, row, b_full);
          cur_nt = nt;
          ++bcount;
        }
        const int s = (int)(it % C::kStages);
        const uint32_t u = (uint32_t)(it / C::kStages);
        if (!W.wait(a_empty(s), (u & 1u) ^ 1u)) break;
        mbar_expect_tx(a_full(s), C::kABytes);
        const uint32_t dst = sA + s * C::kABytes;
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_2d(dst + kb * (kBM * 128), &k_map, kb * 64, (int32_t)(pt * kBM),
                      a_full(s));
        ++it;
      }
      // Let every copy this thread issued land before the CTA can exit.
      for (int64_t j = it > C::kStages ? it - C::kStages : 0; j < it; ++j)
        drain_wait(a_full((int)(j % C::kStages)), (uint32_t)(j / C::kStages) & 1u,
                   timeout_ns);
      if (bcount > 0) drain_wait(b_full, (uint32_t)(bcount - 1) & 1u, timeout_ns);
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------ MMA issuers
    // Issuer me takes the CTA's tiles k with k % 2 == me into accumulator
    // me: while one waits on its barriers and commits, the other's MMAs
    // keep the tensor core busy (one issuer left it idle half the time,
    // since an MMA issue blocks until the tensor core's short queue takes
    // it).  Stages and tiles keep their order; only the issuing thread
    // alternates.
    const int me = warp - 1;
    if (lane == 0) {
      int64_t it = 0, local = 0;
      int bcount = 0;
      int64_t cur_nt = -1;
      bool issued = false, issued_nt = false;
      int64_t nt = nt_beg;
      int pt = pt_beg;
      bool ok = true;
      for (int64_t item = beg; item < end; ++item, ++it, pt = pt + 1 == n_ptiles ? 0 : pt + 1,
                   nt += pt == 0 ? 1 : 0) {
        if (nt != cur_nt) {
          if (!(ok = W.wait(b_full, bcount & 1))) break;
          ++bcount;
          cur_nt = nt;
          issued_nt = false;
        }
        if (((item - beg) & 1) == me) {
          const uint32_t v = (uint32_t)local;
          if (!(ok = W.wait(acc_empty(me), (v & 1u) ^ 1u))) break;
          const int s = (int)(it % C::kStages);
          const uint32_t u = (uint32_t)(it / C::kStages);
          if (!(ok = W.wait(a_full(s), u & 1u))) break;
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(me * kBN);
          const uint32_t a_tile = sA + s * C::kABytes;
#pragma unroll
          for (int ks = 0; ks < DI / 16; ++ks) {
            const int kb = ks >> 2, kin = ks & 3;
            const uint64_t ad = sdesc_sw128(a_tile + kb * (kBM * 128) + kin * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(sB + kb * (kBN * 128) + kin * 32, 16, 1024);
            tc_mma(d, ad, bd, IDESC, ks > 0 ? 1u : 0u);
          }
          issued = issued_nt = true;
          tc_commit(a_empty(s));
          tc_commit(acc_full(me));
          ++local;
        }
        // last pool tile of this N tile in the CTA's range: this issuer is
        // done with the B tile (after its MMAs complete, if it issued any)
        if (pt + 1 == n_ptiles || item + 1 == end) {
          if (issued_nt) tc_commit(b_empty);
          else mbar_arrive(b_empty);
        }
      }
      (void)ok;
      if (issued) {
        tc_commit(done_bar + 24u * me);
        drain_wait(done_bar + 24u * me, 0, timeout_ns);
      }
    }
  } else {
    // --------------------------------------------------------- epilogue
    const int ew = warp - kEpiWarp0;          // epilogue warp 0..15
    const int quad = warp & 3;                // TMEM lane quadrant
    const int part = ew >> 2;                 // columns part*kEpiCols .. +kEpiCols-1
    int64_t cur_nt = -1, local = 0;
    int wbuf = 1;
    int64_t nt = nt_beg;
    int pt = pt_beg;
    for (int64_t item = beg; item < end; ++item, pt = pt + 1 == n_ptiles ? 0 : pt + 1,
                 nt += pt == 0 ? 1 : 0) {
      if (nt != cur_nt) {
        // the N tile's weights into the other buffer: every epilogue warp
        // has finished the tiles of two N tiles ago (previous barrier), so
        // nobody still reads it
        wbuf ^= 1;
        for (int col = ew * 32 + lane; col < kBN; col += 32 * kEpiWarps) {
          const int64_t qrow = nt * QT + col / HI;
          wsm[wbuf * kBN + col] =
              qrow < rows ? __ldg(w + (t0 - q0 + qrow) * HI + (col % HI)) : 0.f;
        }
        named_bar(1, 32 * kEpiWarps);
        cur_nt = nt;
      }
      const float* wv = wsm + wbuf * kBN + part * kEpiCols;
      const int a = (int)(local & 1);
      const uint32_t v = (uint32_t)(local >> 1);
      ++local;
      // after a failed wait (the CTA is aborting, every later wait returns
      // at once) the warp skips the tile but keeps iterating, so that all
      // epilogue warps reach the same weight barriers
      if (!W.wait(acc_full(a), v & 1u)) continue;
      tc_fence_after();
      const int64_t p = pt * kBM + quad * 32 + lane;
      const bool p_ok = p < p_lim;
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) +
                             (uint32_t)(a * kBN + part * kEpiCols);
      // this part's queries: rows q_part + 0 .. kEpiCols/HI - 1 of the chunk
      const int64_t q_part = nt * QT + (int64_t)part * (kEpiCols / HI);
      float* const sp = scores + q_part * ld + p;
      if constexpr (HI == 1) {  // one column per query
#pragma unroll
        for (int c = 0; c < kEpiCols / 32; ++c) {
          uint32_t r0[16], r1[16];
          tmem_ld16(taddr + c * 32, r0);
          tmem_ld16(taddr + c * 32 + 16, r1);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int qi = c * 32 + j;
            const float x = __uint_as_float(j < 16 ? r0[j] : r1[j - 16]);
            if (p_ok && q_part + qi < rows && DSA_IN_BOUNDS(p < ld, status))
              sp[qi * ld] = wv[qi] * fmaxf(x, 0.f);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty(a));
      } else {
        // the warp's 64 columns come into registers first and the
        // accumulator is released before the arithmetic, so the next
        // tile's MMAs into it need not wait for the epilogue
        relu_weighted_sums<HI, kEpiCols, true>(
            taddr, [&](int i) { return reinterpret_cast<const float4*>(wv)[i]; },
            [&](int qi, float score) {
              if (p_ok && q_part + qi < rows && DSA_IN_BOUNDS(p < ld, status))
                sp[qi * ld] = score;
            },
            [&] {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(acc_empty(a));
            });
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int HI, int DI>
cudaError_t launch_indexer_t(const LaunchCtx& c, const CUtensorMap& q_map,
                             const CUtensorMap& k_map, const float* w,
                             int64_t t0, int64_t q0, int64_t rows, int64_t p_lim,
                             float* scores, int64_t ld) {
  using C = IdxCfg<DI>;
  constexpr int QT = kBN / HI;
  const int64_t n_ntiles = (rows + QT - 1) / QT;
  const int n_ptiles = (int)((p_lim + kBM - 1) / kBM);
  const int64_t n_items = n_ntiles * n_ptiles;
  if (n_items == 0) return cudaSuccess;
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = set_smem_once(indexer_kernel<HI, DI>, (int)C::kSmem, smem_set);
  if (e != cudaSuccess) return e;
  int64_t grid = n_items < c.num_sms ? n_items : c.num_sms;
  indexer_kernel<HI, DI><<<(unsigned)grid, kThreads, C::kSmem, c.stream>>>(
      q_map, k_map, w, t0, q0, rows, p_lim, scores, ld, n_ptiles, n_items, c.status,
      c.timeout_ns);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer(const LaunchCtx& c, const CUtensorMap& q_map,
                           const CUtensorMap& k_map, const float* w, int H_I,
                           int D_I, int64_t t0, int64_t q0, int64_t rows,
                           int64_t p_lim, float* scores, int64_t ld) {
#define DSA_IDX_CASE(HI, DI)                                                   \
  if (H_I == HI && D_I == DI)                                                  \
    return launch_indexer_t<HI, DI>(c, q_map, k_map, w, t0, q0, rows, p_lim,    \
                                    scores, ld);
  DSA_IDX_CASE(1, 64) DSA_IDX_CASE(2, 64) DSA_IDX_CASE(4, 64)
  DSA_IDX_CASE(8, 64) DSA_IDX_CASE(16, 64) DSA_IDX_CASE(32, 64)
  DSA_IDX_CASE(64, 64)
  DSA_IDX_CASE(1, 128) DSA_IDX_CASE(2, 128) DSA_IDX_CASE(4, 128)
  DSA_IDX_CASE(8, 128) DSA_IDX_CASE(16, 128) DSA_IDX_CASE(32, 128)
  DSA_IDX_CASE(64, 128)
#undef DSA_IDX_CASE
  return cudaErrorInvalidValue;
}

}  // namespace dsa
