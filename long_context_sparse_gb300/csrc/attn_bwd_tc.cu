// attn_bwd_tc.cu -- backward of the sparse attention on tcgen05 + TMEM.
//
// Every backward product depends on the attention weights ("MTraining:
// Efficient Distributed Training for Ultra-Long Contexts via Dynamic Sparse
// Attention", section 3.2, Eq. 1), so the backward walks exactly the keys the
// forward selected ("Scaling Training to 1M Token Context on
// GLM-5.3-Flash", section "DeepSeek Sparse Attention (DSA) Optimizations")
// and recomputes P from the stored LSE.  Per query t and 128-key tile:
//
//   S^T  [key, h] = K_tile Q^T          dP^T [key, h] = V_tile dO^T
//   P = exp2(S c2 - LSE2), dS = P (dP - delta)      (thread = key lane)
//   dV^T [d, key] = dO^T P^T            dK^T [d, key] = Q^T dS^T
//   dQ^T [d, h]  += K_tile^T dS          (TMEM-resident over the tiles)
//
// with K/V rows gathered once per tile (K a second time for dQ, from L2).
// Order per tile: S^T, dP^T; dS -> dQ^T, dK^T; P -> dV^T, so the gather
// ring is free for the next tile while the dK/dV chunks are scattered.
// dV^T / dK^T are produced in [128 d x 64 key] chunks with d on the TMEM
// lanes, so each thread holds one d of a key row and a warp's fp32
// reduction covers one contiguous 128-byte segment of that row: the scatter
// into the fp32 dK/dV accumulators is fully coalesced.
//
// Heads are padded to N = 64 (padding heads get P = 0 through LSE = +inf).
// Warps: 0-7 softmax / scatter / dQ epilogue (two warpgroups of 32 heads;
// warp w reads TMEM lane quadrant w % 4), 8-9 gather producers (cp.async
// into 128-byte-swizzled 16 KB stages), 10 MMA issuer and TMEM owner.  Q
// and dO come in by TMA.  Every wait is bounded (DSA_ERR_DEVICE_TIMEOUT).
#include "attn_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int NH = 64;                 // heads per CTA tile (N), padded
constexpr int kTileK = 128;            // keys per tile
constexpr int kStages = 4;             // 16 KB stages: [128 keys x 64 dims]
constexpr uint32_t kStageBytes = 16384;
constexpr int kSmThreads = 256;
constexpr int kProdThreads = 64;
constexpr int kThreads = kSmThreads + kProdThreads + 32;  // 11 warps
constexpr int kMmaWarp = 10;
constexpr int kBarEvery = 2;           // key tiles between grid-wide meetings
constexpr int kMaskWords = (2048 * 4 + 3 + kTileK + 31) / 32;
// the fullest SM sub-partition holds 3 of the 11 warps
constexpr int kMaxReg = (16384 / (((kThreads / 32) + 3) / 4 * 32)) & ~7;

template <int D>
struct BwdTcCfg {
  static constexpr int kAtoms = D / 64;   // 64-dim atoms (stages per pass)
  static constexpr int kDChunks = D / 128;
  static constexpr uint32_t kQBytes = NH * D * 2;
  static constexpr uint32_t kBufBytes = kTileK * NH * 2;  // P / dS [key x 64 h]
  static uint32_t smem(int K_p) {
    return 1024 + 2 * kQBytes + kBufBytes + kStages * kStageBytes +
           carved(2 * (K_p + 8) * 4) + 2 * carved(2 * kTileK * 4) +
           carved(2 * kMaskWords * 4) + 2 * carved(2 * NH * 4) + carved(32) +
           carved(32 * 8);
  }
};

__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
// 32 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t a[16], b[16];
  tmem_ld16(taddr, a);
  tmem_ld16(taddr + 16, b);
  tmem_wait_ld();
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    v[e] = __uint_as_float(a[e]);
    v[16 + e] = __uint_as_float(b[e]);
  }
}

template <int D>
__global__ void __maxnreg__(kMaxReg)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap q_map,
                       const __grid_constant__ CUtensorMap g_map,
                       const __nv_bfloat16* __restrict__ k,
                       const __nv_bfloat16* __restrict__ v,
                       const float* __restrict__ lse,
                       const float* __restrict__ delta,
                       const int32_t* __restrict__ idx,
                       __nv_bfloat16* __restrict__ dq, float* __restrict__ dk_acc,
                       float* __restrict__ dv_acc, int64_t S, int H, int K_p,
                       int n_loc, float scale, int n_hblk, uint32_t* status,
                       uint64_t timeout_ns, uint32_t* grid_ctr, int bar_every,
                       int bar_points) {
  using C = BwdTcCfg<D>;
  constexpr uint32_t ID_KK = idesc_bf16(128, NH, 0, 0);  // S^T, dP^T
  constexpr uint32_t ID_MK = idesc_bf16(128, 64, 1, 0);  // dV^T, dK^T
  constexpr uint32_t ID_MM = idesc_bf16(128, NH, 1, 1);  // dQ^T

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  const uint32_t sQ = base;                      // Q   [64 h x D], atoms of 8 KB
  const uint32_t sG = sQ + C::kQBytes;           // dO  [64 h x D]
  const uint32_t sB = sG + C::kQBytes;           // P / dS [128 key x 64 h]
  const uint32_t sStage = sB + C::kBufBytes;     // ring, 1024-aligned
  // tail regions, each starting on a 128-byte boundary (vector accesses)
  uint8_t* tail = gb + 2 * C::kQBytes + C::kBufBytes + kStages * kStageBytes;
  int32_t* pools = carve<int32_t>(tail, 2 * (K_p + 8));      // [2][K_p+8]
  int32_t* tile_tok = carve<int32_t>(tail, 2 * kTileK);      // [2][128]
  uint32_t* vmask = carve<uint32_t>(tail, 2 * kMaskWords);   // [2][words]
  int32_t* sm_tok = carve<int32_t>(tail, 2 * kTileK);        // [2][128]
  float* lse2_s = carve<float>(tail, 2 * NH);                // [2][NH]
  float* delta_s = carve<float>(tail, 2 * NH);               // [2][NH]
  int* misc = carve<int>(tail, 8);                 // ntok[2], npool[2], last, nadd
  uint64_t* bars = carve<uint64_t>(tail, 32);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  const uint32_t b1 = bar0 + 8u * (2 * kStages);
  const uint32_t qd_full = b1, qd_empty = b1 + 8, sdp_full = b1 + 16,
                 pbuf_full = b1 + 24, pbuf_free = b1 + 32, dsbuf_full = b1 + 40,
                 dsbuf_free = b1 + 48, dq_done = b1 + 56, tq_empty = b1 + 64,
                 done_bar = b1 + 72, sm_grp = b1 + 80, prod_grp = b1 + 88;
  auto chunk_full = [&](int b) { return b1 + 96u + 8u * b; };
  auto chunk_empty = [&](int b) { return b1 + 112u + 8u * b; };
  auto toks_full = [&](int b) { return b1 + 128u + 8u * b; };
  auto toks_empty = [&](int b) { return b1 + 144u + 8u * b; };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(bars + 2 * kStages + 20);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 21);
  int* ntok = misc;        // [2]
  int* npool_s = misc + 2; // [2]
  int* s_last = misc + 4;
  int* s_nadd = misc + 5;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Waiter W{abort_flag, status, timeout_ns};
  const int64_t n_items = S * n_hblk;
  const float c2 = scale * kLog2e;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), kProdThreads);
      mbar_init(empty(s), 1);
    }
    mbar_init(qd_full, 1);
    mbar_init(qd_empty, 1);
    mbar_init(sdp_full, 1);
    mbar_init(pbuf_full, kSmThreads);
    mbar_init(pbuf_free, 1);
    mbar_init(dsbuf_full, kSmThreads);
    mbar_init(dsbuf_free, 1);
    mbar_init(dq_done, 1);
    mbar_init(tq_empty, kSmThreads);
    mbar_init(done_bar, 1);
    mbar_init(sm_grp, kSmThreads);
    mbar_init(prod_grp, kProdThreads);
    for (int b = 0; b < 2; ++b) {
      mbar_init(chunk_full(b), 1);
      mbar_init(chunk_empty(b), kSmThreads);
      mbar_init(toks_full(b), kProdThreads);
      mbar_init(toks_empty(b), kSmThreads);
    }
    *abort_flag = 0u;
    fence_mbar_init();
    prefetch_tensormap(&q_map);
    prefetch_tensormap(&g_map);
  }
  if (warp == kMmaWarp) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;            // S^T   [128 key x 64 h]
  const uint32_t tP = tmem + 64;       // dP^T  [128 key x 64 h]
  const uint32_t tQ = tmem + 128;      // dQ^T  [128 d x 64 h] x D/128
  const uint32_t tC = tmem + 384;      // 2 x [128 d x 64 key] chunk accumulators

  if (warp == 8 || warp == 9) {
    // ============================================ gather producers (64)
    const int ptid = tid - kSmThreads;
    GroupBar G{prod_grp, 0u};
    uint32_t u = 0, nq = 0;
    int qi = 0;
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x, ++qi) {
      if (W.aborted()) break;
      const int64_t t = S - 1 - item / n_hblk;
      const int hb = (int)(item % n_hblk);
      const int buf = qi & 1;
      if (!W.wait(toks_empty(buf), ((qi >> 1) & 1) ^ 1)) break;
      // ---- key list of query t as pool ids + local tokens; LSE/delta rows
      const int32_t* row = idx + t * K_p;
      const int64_t nf = n_full(t);
      int32_t* pl = pools + buf * (K_p + 8);
      int32_t* lc = pl + K_p;
      uint32_t* vm = vmask + buf * kMaskWords;
      if (ptid == 0) {
        *s_last = -1;
        *s_nadd = 0;
      }
      for (int w = ptid; w < kMaskWords; w += kProdThreads) vm[w] = 0u;
      for (int h = ptid; h < NH; h += kProdThreads) {
        const int hg = hb * 64 + h;
        lse2_s[buf * NH + h] = hg < H ? __ldg(lse + t * H + hg) * kLog2e : INFINITY;
        delta_s[buf * NH + h] = hg < H ? __ldg(delta + t * H + hg) : 0.f;
      }
      if (!G.sync(W)) break;
      for (int i = ptid; i < K_p; i += kProdThreads) {
        const int32_t p = __ldg(row + i);
        const bool okp = p >= 0 && (int64_t)p < nf;
        if (p >= 0) {
          atomicMax(s_last, i);
          if (!okp) latch_error(status, DSA_ERR_DEVICE_BAD_INDEX);
        }
        pl[i] = okp ? p : -1;
        if (okp) atomicOr(&vm[(4 * i) >> 5], 0xFu << ((4 * i) & 31));
      }
      if (!G.sync(W)) break;
      const int npool = 4 * (*s_last + 1);
      if (n_loc > 0 && ptid < 32) {
        int nadd = 0;
        for (int j = n_loc - 1; j >= 0; --j) {
          const int64_t s = t - j;
          if (s < 0) continue;
          const int32_t ps = (int32_t)(s >> 2);
          bool mine = false;
          if ((int64_t)ps < nf)
            for (int i = ptid; i < K_p; i += 32) mine |= __ldg(row + i) == ps;
          if (!__any_sync(0xffffffffu, mine)) {
            if (ptid == 0) {
              lc[nadd] = (int32_t)s;
              atomicOr(&vm[(npool + nadd) >> 5], 1u << ((npool + nadd) & 31));
            }
            ++nadd;
          }
        }
        if (ptid == 0) *s_nadd = nadd;
      }
      if (!G.sync(W)) break;
      const int n = npool + *s_nadd;
      const int ntiles = (n + kTileK - 1) / kTileK;
      if (ptid == 0) {
        ntok[buf] = n;
        npool_s[buf] = npool;
      }
      if (!G.sync(W)) break;
      mbar_arrive(toks_full(buf));  // releases list, mask, LSE, delta, counts
      if (ntiles == 0) continue;
      // ---- Q and dO rows of this head block by TMA (box {64, 64})
      if (ptid == 0 && W.wait(qd_empty, (nq & 1u) ^ 1u)) {
        mbar_expect_tx(qd_full, 2 * C::kQBytes);
#pragma unroll
        for (int a = 0; a < C::kAtoms; ++a) {
          tma_load_2d(sQ + a * (NH * 128), &q_map, a * 64, (int32_t)(t * H + hb * 64),
                      qd_full);
          tma_load_2d(sG + a * (NH * 128), &g_map, a * 64, (int32_t)(t * H + hb * 64),
                      qd_full);
        }
      }
      ++nq;
      // ---- per tile: K (for S^T), V (for dP^T), K again (for dQ^T), one
      // 64-dim atom per stage.  A warp instruction copies 4 rows x 128 B.
      auto tok_of = [&](int slot) -> int32_t {
        if (slot < npool) {
          const int32_t p = pl[slot >> 2];
          return p >= 0 ? 4 * p + (slot & 3) : -1;
        }
        return slot < n ? lc[slot - npool] : -1;
      };
      const int pw = ptid >> 5, plane = ptid & 31;
      const int rsub = plane >> 3, ch8 = plane & 7;
      bool ok = true;
      for (int j = 0; j < ntiles && ok; ++j) {
        int32_t* tt = tile_tok + (j & 1) * kTileK;
        for (int r = ptid; r < kTileK; r += kProdThreads) tt[r] = tok_of(j * kTileK + r);
        if (!(ok = G.sync(W))) break;
        for (int pass = 0; pass < 3 && ok; ++pass) {
          const __nv_bfloat16* src = pass == 1 ? v : k;
          for (int a = 0; a < C::kAtoms; ++a, ++u) {
            const int s = (int)(u % kStages);
            if (!(ok = W.wait(empty(s), ((u / kStages) & 1u) ^ 1u))) break;
            const uint32_t st = sStage + s * kStageBytes;
#pragma unroll 4
            for (int i = 0; i < 16; ++i) {
              const int r = pw * 64 + 4 * i + rsub;
              const int32_t tok = tt[r];
              const __nv_bfloat16* sp =
                  src + (int64_t)(tok >= 0 ? tok : 0) * D + a * 64 + ch8 * 8;
              cp_async16(st + r * 128 + ((ch8 ^ (r & 7)) << 4), sp, tok >= 0 ? 16u : 0u);
            }
            cp_async_mbar_arrive(full(s));
          }
        }
      }
      if (!ok) break;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kMmaWarp) {
    // ================================================== MMA issuer
    if (lane == 0) {
      uint32_t u = 0, T = 0, nq = 0, chunk = 0;
      int qi = 0;
      bool ok = true, issued = false;
      for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++qi) {
        const int buf = qi & 1;
        if (!(ok = W.wait(toks_full(buf), (qi >> 1) & 1))) break;
        const int ntiles = (ntok[buf] + kTileK - 1) / kTileK;
        if (ntiles == 0) continue;
        if (!(ok = W.wait(qd_full, nq & 1u))) break;
        for (int j = 0; j < ntiles && ok; ++j, ++T) {
          // ---- S^T = K Q^T, then dP^T = V dO^T (one 64-dim atom per stage)
          for (int pass = 0; pass < 2 && ok; ++pass) {
            const uint32_t dst = pass == 0 ? tS : tP;
            const uint32_t bsrc = pass == 0 ? sQ : sG;
            for (int a = 0; a < C::kAtoms; ++a, ++u) {
              const int s = (int)(u % kStages);
              if (!(ok = W.wait(full(s), (u / kStages) & 1u))) break;
              fence_proxy_async();
              tc_fence_after();
              const uint32_t st = sStage + s * kStageBytes;
#pragma unroll
              for (int kin = 0; kin < 4; ++kin)
                tc_mma(dst, sdesc_sw128(st + kin * 32, 16, 1024),
                       sdesc_sw128(bsrc + a * (NH * 128) + kin * 32, 16, 1024), ID_KK,
                       (a | kin) != 0 ? 1u : 0u);
              issued = true;
              tc_commit(empty(s));
            }
          }
          if (!ok) break;
          tc_commit(sdp_full);
          // ---- dS in sB: dQ^T += K^T dS^T first (K re-gathered, two atoms
          // per 128-dim chunk), so the stage ring is free for the next tile's
          // gather while the chunks below are scattered
          if (!(ok = W.wait(dsbuf_full, T & 1u))) break;
          tc_fence_after();
          if (j == 0 && !(ok = W.wait(tq_empty, (nq & 1u) ^ 1u))) break;
          for (int dc = 0; dc < C::kDChunks && ok; ++dc, u += 2) {
            const int s0 = (int)(u % kStages);  // u is even: s0, s0+1 adjacent
            if (!(ok = W.wait(full(s0), (u / kStages) & 1u))) break;
            if (!(ok = W.wait(full(s0 + 1), ((u + 1) / kStages) & 1u))) break;
            fence_proxy_async();
            tc_fence_after();
            const uint32_t st = sStage + s0 * kStageBytes;
#pragma unroll
            for (int ks = 0; ks < kTileK / 16; ++ks)
              tc_mma(tQ + dc * NH,
                     // A = K^T [128 d x 16 key]: MN-major, atoms 16 KB apart
                     sdesc_sw128(st + ks * 2048, kStageBytes, 1024),
                     // B = dS^T [64 h x 16 key]: MN-major rows of 64 heads
                     sdesc_sw128(sB + ks * 2048, 16, 1024), ID_MM,
                     (j | ks) != 0 ? 1u : 0u);
            tc_commit(empty(s0));
            tc_commit(empty(s0 + 1));
          }
          if (!ok) break;
          // ---- dK^T (dS in sB), then dV^T (P in sB): [128 d x 64 key] chunks
          for (int which = 0; which < 2 && ok; ++which) {
            if (which == 1) {
              tc_commit(dsbuf_free);  // dQ^T and dK^T have read dS
              if (!(ok = W.wait(pbuf_full, T & 1u))) break;
              tc_fence_after();
            }
            const uint32_t asrc = which == 0 ? sQ : sG;
            for (int q = 0; q < 2 * C::kDChunks; ++q, ++chunk) {
              const int dc = q >> 1, kh = q & 1;
              const int b = (int)(chunk & 1u);
              if (!(ok = W.wait(chunk_empty(b), ((chunk >> 1) & 1u) ^ 1u))) break;
              tc_fence_after();
#pragma unroll
              for (int ks = 0; ks < NH / 16; ++ks)
                tc_mma(tC + b * 64,
                       // A = X^T [128 d x 16 h]: MN-major, 64-dim atoms 8 KB apart
                       sdesc_sw128(asrc + (2 * dc) * (NH * 128) + ks * 2048, NH * 128, 1024),
                       // B = dS or P [64 key x 16 h]: K-major rows of 64 heads
                       sdesc_sw128(sB + kh * 64 * 128 + ks * 32, 16, 1024), ID_MK,
                       ks > 0 ? 1u : 0u);
              tc_commit(chunk_full(b));
            }
          }
          if (!ok) break;
          tc_commit(pbuf_free);  // dV^T has read P: the next tile's dS may go in
          if (j == ntiles - 1) {
            tc_commit(dq_done);
            tc_commit(qd_empty);
          }
        }
        ++nq;
      }
      if (issued) {
        tc_commit(done_bar);
        drain(done_bar, 0, timeout_ns);
      }
    }
  } else {
    // ============ softmax, dK/dV scatter and dQ epilogue (2 x 128 threads)
    const int i = tid & 127;              // key lane / d lane
    const int grp = tid >> 7;             // heads grp*32 .. +31, keys grp*32 ..
    const int wq = warp & 3;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    GroupBar G{sm_grp, 0u};
    uint32_t T = 0, nq = 0, chunk = 0, passed = 0;
    int qi = 0;
    bool ok = true;
    // Grid-wide lock-step of the scatter (bar_every > 0): CTAs process
    // generation g = their g-th query together (queries t of one generation
    // lie within gridDim.x of each other, so tile j of each covers the same
    // band of keys) and meet every bar_every tiles; the live band of the
    // dK/dV accumulators then stays L2-resident.  bar_points barrier points
    // per generation for every CTA, tiles or not (the grid is co-resident).
    auto grid_sync = [&]() -> bool {
      if (!G.sync(W)) return false;
      bool okg = true;
      if (tid == 0) {
        asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(grid_ctr) : "memory");
        const uint32_t target = (passed + 1u) * gridDim.x;
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
          uint32_t cur;
          asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(cur) : "l"(grid_ctr) : "memory");
          if ((int32_t)(cur - target) >= 0) break;
          if (*abort_flag) { okg = false; break; }
          if (globaltimer_ns() - t0 > timeout_ns) {
            W.fail(DSA_ERR_DEVICE_TIMEOUT);
            okg = false;
            break;
          }
          __nanosleep(256);
        }
      }
      ++passed;
      return G.sync(W) && okg && !W.aborted();
    };
    const int64_t n_gens = (n_items + gridDim.x - 1) / gridDim.x;
    for (int64_t gen = 0; gen < n_gens && ok; ++gen) {
      const int64_t item = blockIdx.x + gen * gridDim.x;
      if (item >= n_items) {  // no query left here: keep the others moving
        for (int k2 = 0; bar_every > 0 && k2 < bar_points && ok; ++k2) ok = grid_sync();
        continue;
      }
      const int64_t t = S - 1 - item / n_hblk;
      const int hb = (int)(item % n_hblk);
      const int buf = qi & 1;
      if (!(ok = W.wait(toks_full(buf), (qi >> 1) & 1))) break;
      const int n = ntok[buf];
      const int npool = npool_s[buf];
      const int32_t* pl = pools + buf * (K_p + 8);
      const int32_t* lc = pl + K_p;
      const uint32_t* vm = vmask + buf * kMaskWords;
      const float* l2 = lse2_s + buf * NH + grp * 32;
      const float* dl = delta_s + buf * NH + grp * 32;
      const int ntiles = (n + kTileK - 1) / kTileK;
      auto tok_of = [&](int slot) -> int32_t {
        if (slot < npool) {
          const int32_t p = pl[slot >> 2];
          return p >= 0 ? 4 * p + (slot & 3) : -1;
        }
        return slot < n ? lc[slot - npool] : -1;
      };
      const int hcount = H - hb * 64 < 64 ? H - hb * 64 : 64;
      if (ntiles == 0) {  // empty key set: dQ = 0, no dK/dV contribution
        for (int e = tid; e < hcount * D; e += kSmThreads)
          dq[(t * H + hb * 64) * (int64_t)D + e] = __float2bfloat16_rn(0.f);
      }
      const int jmax = bar_every > 0 ? bar_points * bar_every : ntiles;
      for (int j = 0; j < jmax && ok; ++j) {
        if (bar_every > 0 && j > 0 && j % bar_every == 0 && !(ok = grid_sync())) break;
        if (j >= ntiles) continue;
        // ---- P and dS for key i, heads grp*32 .. +31
        if (!(ok = W.wait(sdp_full, T & 1u))) break;
        tc_fence_after();
        float sv[32], pv[32];
        tmem_ld32(tS + lane_base + grp * 32, sv);
        tmem_ld32(tP + lane_base + grp * 32, pv);
        const int slot = j * kTileK + i;
        const bool valid = (vm[slot >> 5] >> (slot & 31)) & 1u;
        int32_t* stt = sm_tok + (T & 1u) * kTileK;  // scatter targets of this tile
        if (grp == 0) stt[i] = tok_of(slot);
        uint32_t pb[16], db[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = valid ? exp2f(sv[e] * c2 - l2[e]) : 0.f;
          const float p1 = valid ? exp2f(sv[e + 1] * c2 - l2[e + 1]) : 0.f;
          pb[e >> 1] = pack_bf16(p0, p1);
          db[e >> 1] = pack_bf16(p0 * (pv[e] - dl[e]), p1 * (pv[e + 1] - dl[e + 1]));
        }
        // row i of the [key x 64 h] buffer: this group's 64 bytes = 4 chunks.
        // dS goes in first (dQ^T, dK^T), then P (dV^T).
        const uint32_t rowa = sB + (uint32_t)i * 128u;
        if (!(ok = W.wait(pbuf_free, (T & 1u) ^ 1u))) break;  // previous P read
#pragma unroll
        for (int c = 0; c < 4; ++c)
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(
                           rowa + (((uint32_t)(grp * 4 + c) ^ (uint32_t)(i & 7)) << 4)),
                       "r"(db[4 * c]), "r"(db[4 * c + 1]), "r"(db[4 * c + 2]),
                       "r"(db[4 * c + 3])
                       : "memory");
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(dsbuf_full);
        if (!(ok = G.sync(W))) break;  // stt[] complete
        // ---- scatter the dK^T chunks, then (after P is in place) dV^T
        for (int which = 0; which < 2 && ok; ++which) {
          if (which == 1) {
            // dQ^T and dK^T have read every dS: put P in the buffer for dV^T
            if (!(ok = W.wait(dsbuf_free, T & 1u))) break;
#pragma unroll
            for (int c = 0; c < 4; ++c)
              asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(
                               rowa + (((uint32_t)(grp * 4 + c) ^ (uint32_t)(i & 7)) << 4)),
                           "r"(pb[4 * c]), "r"(pb[4 * c + 1]), "r"(pb[4 * c + 2]),
                           "r"(pb[4 * c + 3])
                           : "memory");
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(pbuf_full);
          }
          float* acc = which == 0 ? dk_acc : dv_acc;
          const float f = which == 0 ? scale : 1.f;
          for (int q = 0; q < 2 * C::kDChunks; ++q, ++chunk) {
            const int dc = q >> 1, kh = q & 1;
            const int b = (int)(chunk & 1u);
            if (!(ok = W.wait(chunk_full(b), (chunk >> 1) & 1u))) break;
            tc_fence_after();
            float cv[32];  // d = dc*128 + i, keys kh*64 + grp*32 + e
            tmem_ld32(tC + b * 64 + lane_base + grp * 32, cv);
            tc_fence_before();
            mbar_arrive(chunk_empty(b));
            float* dst = acc + dc * 128 + i;
            const int4* tk4 = reinterpret_cast<const int4*>(stt + kh * 64 + grp * 32);
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
              const int4 tk = tk4[e4];  // warp-uniform tokens of 4 keys
              const int32_t tks[4] = {tk.x, tk.y, tk.z, tk.w};
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (tks[e] >= 0) red_add_f32(dst + (int64_t)tks[e] * D, f * cv[4 * e4 + e]);
            }
          }
        }
        ++T;
      }
      if (!ok) break;
      if (bar_every > 0 && !(ok = grid_sync())) break;  // last point of the generation
      if (ntiles == 0) {
        mbar_arrive(toks_empty(buf));
        ++qi;
        continue;
      }
      // ---- dQ = scale * dQ^T -> bf16 (thread = d within each 128-d chunk)
      if (!(ok = W.wait(dq_done, nq & 1u))) break;
      tc_fence_after();
#pragma unroll 1
      for (int dc = 0; dc < C::kDChunks; ++dc) {
        float qv[32];
        tmem_ld32(tQ + dc * NH + lane_base + grp * 32, qv);
        const int d = dc * 128 + i;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int h = grp * 32 + e;
          if (h < hcount)
            dq[(t * H + hb * 64 + h) * (int64_t)D + d] = __float2bfloat16_rn(qv[e] * scale);
        }
      }
      tc_fence_before();
      mbar_arrive(tq_empty);
      mbar_arrive(toks_empty(buf));
      ++nq;
      ++qi;
    }
  }

  // ---- teardown: every role has left its loop, no MMA or copy in flight
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

template <int D>
cudaError_t launch_t(const LaunchCtx& c, const AttnShape& s, const CUtensorMap& qm,
                     const CUtensorMap& gm, const __nv_bfloat16* k,
                     const __nv_bfloat16* v, const float* lse, const float* delta,
                     const int32_t* idx, __nv_bfloat16* dq, float* dk_acc,
                     float* dv_acc) {
  using C = BwdTcCfg<D>;
  const uint32_t smem = C::smem(s.K_p);
  if (smem > 232448) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_tc_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_bwd_tc_kernel<D>,
                                                    kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) {
    cudaFuncAttributes fa;
    cudaFuncGetAttributes(&fa, attn_bwd_tc_kernel<D>);
    set_error_detail("attn_bwd_tc occupancy 0: regs=%d threads=%d dyn_smem=%u "
                     "max_threads=%d",
                     fa.numRegs, kThreads, smem, fa.maxThreadsPerBlock);
    return cudaErrorLaunchOutOfResources;
  }
  const int n_hblk = (s.H + 63) / 64;
  const int64_t items = s.S * n_hblk;
  int64_t grid = c.num_sms;
  if (grid > items) grid = items;
  // lock-step scatter only when the fp32 dK/dV accumulators outgrow L2
  const int max_tiles = (4 * s.K_p + s.n_loc + kTileK - 1) / kTileK;
  int bar_every = (double)s.S * s.D * 8.0 > 96.0 * (1 << 20) ? kBarEvery : 0;
  if (grid < 2) bar_every = 0;
  int bar_points = bar_every > 0 ? (max_tiles + bar_every - 1) / bar_every : 0;
  uint32_t* grid_ctr = c.status + 32;  // zeroed by the delta kernel
  if (bar_every == 0) {
    attn_bwd_tc_kernel<D><<<(unsigned)grid, kThreads, smem, c.stream>>>(
        qm, gm, k, v, lse, delta, idx, dq, dk_acc, dv_acc, s.S, s.H, s.K_p, s.n_loc,
        s.scale, n_hblk, c.status, c.timeout_ns, grid_ctr, bar_every, bar_points);
    return cudaGetLastError();
  }
  // the CTAs wait on one another: a cooperative launch guarantees that
  // every CTA of the grid is resident at once (or refuses the launch)
  const CUtensorMap q_arg = qm, g_arg = gm;
  int64_t S_arg = s.S;
  int H_arg = s.H, K_arg = s.K_p, nl_arg = s.n_loc, nh_arg = n_hblk;
  float sc_arg = s.scale;
  uint32_t* st_arg = c.status;
  uint64_t to_arg = c.timeout_ns;
  void* args[] = {(void*)&q_arg, (void*)&g_arg, (void*)&k, (void*)&v, (void*)&lse,
                  (void*)&delta, (void*)&idx, (void*)&dq, (void*)&dk_acc,
                  (void*)&dv_acc, (void*)&S_arg, (void*)&H_arg, (void*)&K_arg,
                  (void*)&nl_arg, (void*)&sc_arg, (void*)&nh_arg, (void*)&st_arg,
                  (void*)&to_arg, (void*)&grid_ctr, (void*)&bar_every,
                  (void*)&bar_points};
  return cudaLaunchCooperativeKernel((const void*)attn_bwd_tc_kernel<D>,
                                     dim3((unsigned)grid), dim3(kThreads), args, smem,
                                     c.stream);
}

}  // namespace

cudaError_t launch_attn_bwd_tc(const LaunchCtx& c, const AttnShape& s,
                               const CUtensorMap& q_map, const CUtensorMap& g_map,
                               const __nv_bfloat16* k, const __nv_bfloat16* v,
                               const float* lse, const float* delta,
                               const int32_t* idx, __nv_bfloat16* dq, float* dk_acc,
                               float* dv_acc) {
  if (s.D == 128)
    return launch_t<128>(c, s, q_map, g_map, k, v, lse, delta, idx, dq, dk_acc, dv_acc);
  if (s.D == 256)
    return launch_t<256>(c, s, q_map, g_map, k, v, lse, delta, idx, dq, dk_acc, dv_acc);
  if (s.D == 512)
    return launch_t<512>(c, s, q_map, g_map, k, v, lse, delta, idx, dq, dk_acc, dv_acc);
  return cudaErrorInvalidValue;
}

}  // namespace dsa
