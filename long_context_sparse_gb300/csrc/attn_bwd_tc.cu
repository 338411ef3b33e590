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
//   dQ^T [d, h]  += K_tile^T dS          (TMEM-resident over the tiles)
//   dK^T [d, key] = Q^T dS^T            dV^T [d, key] = dO^T P^T
//
// dK^T / dV^T are produced in [128 d x 32 key] chunks with d on the TMEM
// lanes, so a warp's fp32 reduction into the dK/dV accumulators covers one
// contiguous 128-byte segment of a key row (fully coalesced).  The softmax
// scale is folded into dS, so dQ and dK need no rescaling.  That scatter
// carries 4 KB per (query, key) pair at d = 512 and is the bound of the
// whole backward, so the kernel is organised to keep it running without a
// break: eight warps do nothing but drain chunks from TMEM into
// red.global.add, while the products of the next chunks and tiles proceed
// behind them.
//
// Roles (20 warps):
//   0-3   softmax: P and dS of a tile (thread = key lane), written to two
//         separate shared buffers; the dQ epilogue of each query.
//   4-11  scatter: TMEM chunk -> fp32 reductions (warp w reads lane quadrant
//         w % 4); warps 4-7 drain the even chunks, 8-11 the odd ones, each
//         half double-buffered in TMEM.
//   12-17 producers: key lists, Q/dO by TMA, K/V rows gathered with cp.async
//         into 128-byte-swizzled 16 KB stages.  The gather rate grows with
//         the number of issuing warps, not with the bytes in flight, hence
//         six (the register budget is the same for 18 and 20 warps).  (TMA
//         tile::gather4 moves the same rows, but at 128 bytes per row
//         segment one issuing thread reaches only a fraction of it.)
//   18    MMA issuer A (TMEM owner): S^T, dP^T and dQ^T, in ring order.
//   19    MMA issuer B: the dK^T and dV^T chunks.
// Two issuers keep the chunk stream independent of the gather ring: A runs
// up to a tile ahead of B.
//
// K = V (one tensor serving as both, as an MLA latent does): S^T and dP^T
// take their A operand from the same gathered K stage (a third less
// gathering), and each chunk accumulates dK^T and dV^T of the same rows in
// TMEM before one scatter into the single dKV accumulator (half the
// reduction bytes).  Heads are padded to N = 64 (padding heads get
// P = 0 through LSE = +inf).  Every wait is bounded (DSA_ERR_DEVICE_TIMEOUT).
//
// Scheduling.  CTAs take queries from a global counter in descending t, so
// SMs that run slower take fewer.  For L2 locality every CTA should touch
// the same band of keys at the same time: a query's key list is sorted, so
// tile j of every recent query covers about the same key range.  Query
// number i starts at tile (i * ntiles / CTAs) mod ntiles, the band the grid
// has reached when it is taken, and wraps around.  The live part of the
// fp32 dK/dV accumulators and of K/V then stays small without any
// grid-wide barrier, and a query's tile order (hence its fp32 sum order)
// does not depend on timing.
#include "attn_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int NH = 64;                 // heads per CTA tile (N), padded
constexpr int kTileK = 128;            // keys per tile
constexpr int kStages = 3;             // 16 KB gather stages
constexpr uint32_t kStageBytes = 16384;
constexpr int kSmThreads = 128;        // softmax warps 0-3
constexpr int kScThreads = 256;        // scatter warps 4-11
constexpr int kProdThreads = 192;      // producer warps 12-17
constexpr int kProdWarps = kProdThreads / 32;
constexpr int kScWarp0 = 4, kProdWarp0 = 12, kMmaA = 18, kMmaB = 19;
constexpr int kThreads = 640;
constexpr int kMaskWords = (2048 * 4 + 3 + kTileK + 31) / 32;
// the fullest SM sub-partition holds five of the 20 warps
constexpr int kMaxReg = (16384 / (((kThreads / 32) + 3) / 4 * 32)) & ~7;
static_assert(kMaxReg == 96, "register budget");

template <int D>
struct BwdTcCfg {
  static constexpr int kAtoms = D / 64;   // 64-dim atoms: S / dP stages per tile
  static constexpr int kDChunks = D / 128;
  static constexpr uint32_t kQBytes = NH * D * 2;
  static constexpr uint32_t kBufBytes = kTileK * NH * 2;  // P or dS [key x 64 h]
  static uint32_t smem(int K_p) {
    return 1024 + 2 * kQBytes + 2 * kBufBytes + kStages * kStageBytes +
           carved(2 * (K_p + 8) * 4) + carved(2 * kTileK * 4) +
           carved(2 * kMaskWords * 4) + 2 * carved(2 * NH * 4) + carved(48) +
           carved(40 * 8);
  }
};

__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
// The four keys of pool p are consecutive rows: one address, the other three
// rows at immediate offsets of D floats.
template <int D>
__device__ __forceinline__ void red_add_pool(float* r, float a, float b, float c,
                                             float d) {
  asm volatile(
      "red.global.add.f32 [%0], %1;\n\t"
      "red.global.add.f32 [%0+%5], %2;\n\t"
      "red.global.add.f32 [%0+%6], %3;\n\t"
      "red.global.add.f32 [%0+%7], %4;" ::"l"(r),
      "f"(a), "f"(b), "f"(c), "f"(d), "n"(D * 4), "n"(D * 8), "n"(D * 12)
      : "memory");
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

template <int D, bool KV>
__global__ void __maxnreg__(kMaxReg)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap q_map,
                       const __grid_constant__ CUtensorMap g_map,
                       const __nv_bfloat16* __restrict__ k,
                       const __nv_bfloat16* __restrict__ v,
                       const float* __restrict__ lse,
                       const float* __restrict__ delta,
                       const int32_t* __restrict__ idx,
                       __nv_bfloat16* __restrict__ dq, float* __restrict__ dk_acc,
                       float* __restrict__ dv_acc, int64_t t_lo, int64_t t_hi,
                       int64_t item0, int rot_div, int H, int K_p,
                       int n_loc, float scale, int n_hblk, uint32_t* status,
                       uint64_t timeout_ns, uint32_t* sched) {
  using C = BwdTcCfg<D>;
  constexpr uint32_t ID_KK = idesc_bf16(128, NH, 0, 0);  // S^T, dP^T
  constexpr uint32_t ID_MK = idesc_bf16(128, 32, 1, 0);  // dV^T, dK^T chunks
  constexpr uint32_t ID_MM = idesc_bf16(128, NH, 1, 1);  // dQ^T

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  const uint32_t sQ = base;                      // Q   [64 h x D], atoms of 8 KB
  const uint32_t sG = sQ + C::kQBytes;           // dO  [64 h x D]
  const uint32_t sDS = sG + C::kQBytes;          // dS  [128 key x 64 h]
  const uint32_t sP = sDS + C::kBufBytes;        // P   [128 key x 64 h]
  const uint32_t sStage = sP + C::kBufBytes;     // ring, 1024-aligned
  // tail regions, each starting on a 128-byte boundary (vector accesses)
  uint8_t* tail = gb + 2 * C::kQBytes + 2 * C::kBufBytes + kStages * kStageBytes;
  int32_t* pools = carve<int32_t>(tail, 2 * (K_p + 8));      // [2][K_p+8]
  int32_t* tile_tok = carve<int32_t>(tail, 2 * kTileK);      // [2][128]
  uint32_t* vmask = carve<uint32_t>(tail, 2 * kMaskWords);   // [2][words]
  float* lse2_s = carve<float>(tail, 2 * NH);                // [2][NH]
  float* delta_s = carve<float>(tail, 2 * NH);               // [2][NH]
  int* misc = carve<int>(tail, 12);  // ntok[2] npool[2] last nadd item[2] rot[2]
  uint64_t* bars = carve<uint64_t>(tail, 40);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  const uint32_t b1 = bar0 + 8u * (2 * kStages);
  const uint32_t qd_full = b1, qd_empty = b1 + 8, sdp_full = b1 + 16,
                 sdp_free = b1 + 24, ds_full = b1 + 32, ds_free = b1 + 40,
                 p_full = b1 + 48, p_free = b1 + 56, dq_done = b1 + 64,
                 tq_empty = b1 + 72, done_a = b1 + 80, done_b = b1 + 88,
                 prod_grp = b1 + 96;
  auto chunk_full = [&](int b) { return b1 + 104u + 8u * b; };   // [4]
  auto chunk_empty = [&](int b) { return b1 + 136u + 8u * b; };  // [4]
  auto toks_full = [&](int b) { return b1 + 168u + 8u * b; };
  auto toks_empty = [&](int b) { return b1 + 184u + 8u * b; };
  // 6 ring barriers + 25 above = 31 of the 40 slots; slot 38 abort, 39 TMEM
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(bars + 38);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 39);
  int* ntok = misc;        // [2]
  int* npool_s = misc + 2; // [2]
  int* s_last = misc + 4;
  int* s_nadd = misc + 5;
  int* item_s = misc + 6;  // [2] query of the buffer (>= n_items: no more)
  int* rot_s = misc + 8;   // [2] first tile of the query (rotation)
  uint32_t* work_ctr = sched;  // next query to take

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Waiter W{abort_flag, status, timeout_ns};
  // queries t_lo .. t_hi-1, latest first; row r = t - t_lo of q, dO, idx,
  // lse, delta and dq; item0 + item numbers the query as a whole-sequence
  // call would
  const int64_t n_items = (t_hi - t_lo) * n_hblk;
  const float c2 = scale * kLog2e;
  // every consumer of a query's key list releases it once
  constexpr uint32_t kToksUsers = kSmThreads + kScThreads + 2;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), kProdThreads);
      mbar_init(empty(s), 1);
    }
    mbar_init(qd_full, 1);
    mbar_init(qd_empty, 1);
    mbar_init(sdp_full, 1);
    mbar_init(sdp_free, kSmThreads);
    mbar_init(ds_full, kSmThreads);
    mbar_init(ds_free, 2);              // issuer A (dQ^T) and issuer B (dK^T)
    mbar_init(p_full, kSmThreads);
    mbar_init(p_free, 1);
    mbar_init(dq_done, 1);
    mbar_init(tq_empty, kSmThreads);
    mbar_init(done_a, 1);
    mbar_init(done_b, 1);
    mbar_init(prod_grp, kProdThreads);
    for (int b = 0; b < 4; ++b) {
      mbar_init(chunk_full(b), 1);
      mbar_init(chunk_empty(b), kScThreads / 2);  // one half of the scatter warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(toks_full(b), kProdThreads);
      mbar_init(toks_empty(b), kToksUsers);
    }
    *abort_flag = 0u;
    fence_mbar_init();
    prefetch_tensormap(&q_map);
    prefetch_tensormap(&g_map);
  }
  if (warp == kMmaA) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;            // S^T   [128 key x 64 h]
  const uint32_t tP = tmem + 64;       // dP^T  [128 key x 64 h]
  const uint32_t tQ = tmem + 128;      // dQ^T  [128 d x 64 h] x D/128
  const uint32_t tC = tmem + 384;      // 4 x [128 d x 32 key] chunk accumulators

  // token of key slot `slot` of a query's list (-1: empty or invalid)
  auto tok_of = [&](const int32_t* pl, const int32_t* lc, int npool, int n,
                    int slot) -> int32_t {
    if (slot < npool) {
      const int32_t p = pl[slot >> 2];
      return p >= 0 ? 4 * p + (slot & 3) : -1;
    }
    return slot < n ? lc[slot - npool] : -1;
  };

  if (warp >= kProdWarp0 && warp < kMmaA) {
    // =========================================== gather producers (192)
    const int ptid = tid - kProdWarp0 * 32;
    GroupBar G{prod_grp, 0u};
    uint32_t u = 0, nq = 0;
    int qi = 0;
    for (;; ++qi) {
      if (W.aborted()) break;
      const int buf = qi & 1;
      if (!W.wait(toks_empty(buf), ((qi >> 1) & 1) ^ 1)) break;
      if (ptid == 0) item_s[buf] = (int)atomicAdd(work_ctr, 1u);
      if (!G.sync(W)) break;
      const int64_t item = item_s[buf];
      if (item >= n_items) {  // no query left: tell the other roles
        mbar_arrive(toks_full(buf));
        break;
      }
      const int64_t t = t_hi - 1 - item / n_hblk, r = t - t_lo;
      const int hb = (int)(item % n_hblk);
      // ---- key list of query t as pool ids + local tokens; LSE/delta rows
      const int32_t* row = idx + r * K_p;
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
        lse2_s[buf * NH + h] = hg < H ? __ldg(lse + r * H + hg) * kLog2e : INFINITY;
        delta_s[buf * NH + h] = hg < H ? __ldg(delta + r * H + hg) : 0.f;
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
        // tile band of this query's generation: queries are taken in order
        // and every CTA works through ntiles tiles per query, so about
        // item * ntiles / gridDim.x tiles per CTA have been gathered when
        // it starts (a pure function of the query: results repeat exactly)
        rot_s[buf] = ntiles > 0
                         ? (int)(((uint64_t)(item0 + item) * (uint64_t)ntiles / (uint64_t)rot_div) %
                                 (uint64_t)ntiles)
                         : 0;
      }
      if (!G.sync(W)) break;
      mbar_arrive(toks_full(buf));  // releases list, mask, LSE, delta, counts
      if (ntiles == 0) continue;
      // ---- Q and dO rows of this head block by TMA (box {64, 64})
      if (ptid == 0 && W.wait(qd_empty, (nq & 1u) ^ 1u)) {
        mbar_expect_tx(qd_full, 2 * C::kQBytes);
#pragma unroll
        for (int a = 0; a < C::kAtoms; ++a) {
          tma_load_2d(sQ + a * (NH * 128), &q_map, a * 64, (int32_t)(r * H + hb * 64),
                      qd_full);
          tma_load_2d(sG + a * (NH * 128), &g_map, a * 64, (int32_t)(r * H + hb * 64),
                      qd_full);
        }
      }
      ++nq;
      // ---- per tile: K atoms [128 key x 64 d] (S^T), V atoms (dP^T), then
      // K again in [2 x (64 key x 64 d)] stages, one per (128-d chunk, key
      // half), for dQ^T.  A warp instruction copies 4 rows x 128 B; empty
      // slots are zero-filled.
      const int pw = ptid >> 5, plane = ptid & 31;
      const int rsub = plane >> 3, ch8 = plane & 7;
      const int rot = rot_s[buf];
      bool ok = true;
      for (int j = 0; j < ntiles && ok; ++j) {
        const int jr = j + rot < ntiles ? j + rot : j + rot - ntiles;
        int32_t* tt = tile_tok + (j & 1) * kTileK;
        for (int r = ptid; r < kTileK; r += kProdThreads)
          tt[r] = tok_of(pl, lc, npool, n, jr * kTileK + r);
        if (!(ok = G.sync(W))) break;
        for (int pass = 0; pass < 3 && ok; ++pass) {
          if (KV && pass == 1) continue;  // the V atoms are the K atoms
          const __nv_bfloat16* src = pass == 1 ? v : k;
          for (int a = 0; a < C::kAtoms; ++a, ++u) {
            const int s = (int)(u % kStages);
            if (!(ok = W.wait(empty(s), ((u / kStages) & 1u) ^ 1u))) break;
            const uint32_t st = sStage + s * kStageBytes;
            if (pass < 2) {
              // 32 four-row groups per stage, dealt round-robin to the warps
              for (int g = pw; g < kTileK / 4; g += kProdWarps) {
                const int r = 4 * g + rsub;
                const int32_t tok = tt[r];
                const __nv_bfloat16* sp =
                    src + (int64_t)(tok >= 0 ? tok : 0) * D + a * 64 + ch8 * 8;
                const uint32_t dst = st + r * 128 + ((ch8 ^ (r & 7)) << 4);
                if (DSA_IN_BOUNDS(dst - sStage < (uint32_t)(kStages * kStageBytes) && tok <= t,
                                  status))
                  cp_async16(dst, sp, tok >= 0 ? 16u : 0u);
              }
            } else {
              // stage a = (dc, kh): keys kh*64 .. +63, dims dc*128 .. +127
              const int dc = a >> 1, kh = a & 1;
              for (int g = pw; g < kTileK / 4; g += kProdWarps) {
                const int rr = 4 * g + rsub;             // 0..127
                const int blk = rr >> 6, r = rr & 63;    // d block, key row
                const int32_t tok = tt[kh * 64 + r];
                const __nv_bfloat16* sp = src + (int64_t)(tok >= 0 ? tok : 0) * D +
                                          dc * 128 + blk * 64 + ch8 * 8;
                const uint32_t dst = st + blk * 8192 + r * 128 + ((ch8 ^ (r & 7)) << 4);
                if (DSA_IN_BOUNDS(dst - sStage < (uint32_t)(kStages * kStageBytes) && tok <= t,
                                  status))
                  cp_async16(dst, sp, tok >= 0 ? 16u : 0u);
              }
            }
            cp_async_mbar_arrive(full(s));
          }
        }
      }
      if (!ok) break;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kMmaA) {
    // ======================== MMA issuer A: S^T, dP^T, dQ^T (ring order)
    if (lane == 0) {
      uint32_t u = 0, T = 0, nq = 0;
      int qi = 0;
      bool ok = true, issued = false;
      for (;; ++qi) {
        const int buf = qi & 1;
        if (!(ok = W.wait(toks_full(buf), (qi >> 1) & 1))) break;
        if (item_s[buf] >= n_items) break;
        const int ntiles = (ntok[buf] + kTileK - 1) / kTileK;
        mbar_arrive(toks_empty(buf));
        if (ntiles == 0) continue;
        if (!(ok = W.wait(qd_full, nq & 1u))) break;
        for (int j = 0; j < ntiles && ok; ++j, ++T) {
          // S^T / dP^T of the previous tile have been read
          if (!(ok = W.wait(sdp_free, (T & 1u) ^ 1u))) break;
          tc_fence_after();
          for (int pass = 0; pass < (KV ? 1 : 2) && ok; ++pass) {
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
              if (KV)  // dP^T = K dO^T from the same stage
#pragma unroll
                for (int kin = 0; kin < 4; ++kin)
                  tc_mma(tP, sdesc_sw128(st + kin * 32, 16, 1024),
                         sdesc_sw128(sG + a * (NH * 128) + kin * 32, 16, 1024), ID_KK,
                         (a | kin) != 0 ? 1u : 0u);
              issued = true;
              tc_commit(empty(s));
            }
          }
          if (!ok) break;
          tc_commit(sdp_full);
          // ---- dQ^T += K^T dS^T, one [128 d x 64 key] stage at a time
          if (!(ok = W.wait(ds_full, T & 1u))) break;
          tc_fence_after();
          if (j == 0 && !(ok = W.wait(tq_empty, (nq & 1u) ^ 1u))) break;
          for (int a = 0; a < C::kAtoms && ok; ++a, ++u) {
            const int dc = a >> 1, kh = a & 1;
            const int s = (int)(u % kStages);
            if (!(ok = W.wait(full(s), (u / kStages) & 1u))) break;
            fence_proxy_async();
            tc_fence_after();
            const uint32_t st = sStage + s * kStageBytes;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc_mma(tQ + dc * NH,
                     // A = K^T [128 d x 16 key]: MN-major, d blocks 8 KB apart
                     sdesc_sw128(st + ks * 2048, 8192, 1024),
                     // B = dS^T [16 key x 64 h]: MN-major rows of 64 heads
                     sdesc_sw128(sDS + (kh * 64 + ks * 16) * 128, 16, 1024), ID_MM,
                     (j | kh | ks) != 0 ? 1u : 0u);
            tc_commit(empty(s));
          }
          if (!ok) break;
          tc_commit(ds_free);
          if (j == ntiles - 1) tc_commit(dq_done);
        }
        ++nq;
      }
      if (issued) {
        tc_commit(done_a);
        drain(done_a, 0, timeout_ns);
      }
    }
  } else if (warp == kMmaB) {
    // ============================ MMA issuer B: dK^T, dV^T chunks
    if (lane == 0) {
      uint32_t T = 0, nq = 0, chunk = 0;
      int qi = 0;
      bool ok = true, issued = false;
      for (;; ++qi) {
        const int buf = qi & 1;
        if (!(ok = W.wait(toks_full(buf), (qi >> 1) & 1))) break;
        if (item_s[buf] >= n_items) break;
        const int ntiles = (ntok[buf] + kTileK - 1) / kTileK;
        mbar_arrive(toks_empty(buf));
        if (ntiles == 0) continue;
        if (!(ok = W.wait(qd_full, nq & 1u))) break;
        for (int j = 0; j < ntiles && ok; ++j, ++T) {
          if (KV) {
            // one chunk per (d chunk, key quarter): dK^T then dV^T into it
            if (!(ok = W.wait(ds_full, T & 1u))) break;
            if (!(ok = W.wait(p_full, T & 1u))) break;
            tc_fence_after();
            for (int q = 0; q < 4 * C::kDChunks; ++q, ++chunk) {
              const int dc = q >> 2, kq = q & 3;
              const int b = (int)(chunk & 3u);
              if (!(ok = W.wait(chunk_empty(b), ((chunk >> 2) & 1u) ^ 1u))) break;
              tc_fence_after();
#pragma unroll
              for (int x = 0; x < 2; ++x)
#pragma unroll
                for (int ks = 0; ks < NH / 16; ++ks)
                  tc_mma(tC + b * 32,
                         sdesc_sw128((x == 0 ? sQ : sG) + (2 * dc) * (NH * 128) + ks * 2048,
                                     NH * 128, 1024),
                         sdesc_sw128((x == 0 ? sDS : sP) + kq * 32 * 128 + ks * 32, 16, 1024),
                         ID_MK, (x | ks) != 0 ? 1u : 0u);
              issued = true;
              tc_commit(chunk_full(b));
            }
            if (!ok) break;
            tc_commit(ds_free);
            tc_commit(p_free);
            if (j == ntiles - 1) tc_commit(qd_empty);
            continue;
          }
          for (int which = 0; which < 2 && ok; ++which) {
            const uint32_t bsrc = which == 0 ? sDS : sP;
            const uint32_t asrc = which == 0 ? sQ : sG;
            if (!(ok = W.wait(which == 0 ? ds_full : p_full, T & 1u))) break;
            tc_fence_after();
            for (int q = 0; q < 4 * C::kDChunks; ++q, ++chunk) {
              const int dc = q >> 2, kq = q & 3;
              const int b = (int)(chunk & 3u);
              if (!(ok = W.wait(chunk_empty(b), ((chunk >> 2) & 1u) ^ 1u))) break;
              tc_fence_after();
#pragma unroll
              for (int ks = 0; ks < NH / 16; ++ks)
                tc_mma(tC + b * 32,
                       // A = X^T [128 d x 16 h]: MN-major, 64-dim atoms 8 KB apart
                       sdesc_sw128(asrc + (2 * dc) * (NH * 128) + ks * 2048, NH * 128, 1024),
                       // B = dS or P [32 key x 16 h]: K-major rows of 64 heads
                       sdesc_sw128(bsrc + kq * 32 * 128 + ks * 32, 16, 1024), ID_MK,
                       ks > 0 ? 1u : 0u);
              issued = true;
              tc_commit(chunk_full(b));
            }
            if (!ok) break;
            tc_commit(which == 0 ? ds_free : p_free);
          }
          if (!ok) break;
          if (j == ntiles - 1) tc_commit(qd_empty);  // last read of Q and dO
        }
        ++nq;
      }
      if (issued) {
        tc_commit(done_b);
        drain(done_b, 0, timeout_ns);
      }
    }
  } else if (warp < kScWarp0) {
    // ==================== softmax (128 threads, thread = key lane) + dQ
    const int i = tid;                     // key lane / d lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    uint32_t T = 0, nq = 0;
    int qi = 0;
    bool ok = true;
    for (;; ++qi) {
      const int buf = qi & 1;
      if (!(ok = W.wait(toks_full(buf), (qi >> 1) & 1))) break;
      const int64_t item = item_s[buf];
      if (item >= n_items) break;
      const int64_t r = t_hi - 1 - item / n_hblk - t_lo;  // row of dq
      const int hb = (int)(item % n_hblk);
      const int n = ntok[buf];
      const int rot = rot_s[buf];
      const uint32_t* vm = vmask + buf * kMaskWords;
      const float* l2 = lse2_s + buf * NH;
      const float* dl = delta_s + buf * NH;
      const int ntiles = (n + kTileK - 1) / kTileK;
      const int hcount = H - hb * 64 < 64 ? H - hb * 64 : 64;
      if (ntiles == 0) {  // empty key set: dQ = 0, no dK/dV contribution
        for (int e = i; e < hcount * D; e += kSmThreads)
          dq[(r * H + hb * 64) * (int64_t)D + e] = __float2bfloat16_rn(0.f);
        mbar_arrive(toks_empty(buf));
        continue;
      }
      const uint32_t rowa = (uint32_t)i * 128u;  // row i of a [key x 64 h] buffer
      for (int j = 0; j < ntiles && ok; ++j, ++T) {
        const int jr = j + rot < ntiles ? j + rot : j + rot - ntiles;
        const int slot = jr * kTileK + i;
        const bool valid = (vm[slot >> 5] >> (slot & 31)) & 1u;
        // dQ^T, dK^T and dV^T of the previous tile have read dS and P (by
        // the time the softmax gets here they almost always have)
        if (!(ok = W.wait(ds_free, (T & 1u) ^ 1u))) break;
        if (!(ok = W.wait(p_free, (T & 1u) ^ 1u))) break;
        if (!(ok = W.wait(sdp_full, T & 1u))) break;
        tc_fence_after();
#pragma unroll
        for (int qh = 0; qh < 4; ++qh) {  // 16 heads at a time
          uint32_t sa[16], pa[16];
          tmem_ld16(tS + lane_base + qh * 16, sa);
          tmem_ld16(tP + lane_base + qh * 16, pa);
          tmem_wait_ld();
          uint32_t pb[8], db[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const int h = qh * 16 + e;
            const float p0 =
                valid ? exp2f(__uint_as_float(sa[e]) * c2 - l2[h]) : 0.f;
            const float p1 =
                valid ? exp2f(__uint_as_float(sa[e + 1]) * c2 - l2[h + 1]) : 0.f;
            pb[e >> 1] = pack_bf16(p0, p1);
            db[e >> 1] = pack_bf16(scale * p0 * (__uint_as_float(pa[e]) - dl[h]),
                                   scale * p1 * (__uint_as_float(pa[e + 1]) - dl[h + 1]));
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint32_t off = rowa + (((uint32_t)(qh * 2 + c) ^ (uint32_t)(i & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(sDS + off),
                         "r"(db[4 * c]), "r"(db[4 * c + 1]), "r"(db[4 * c + 2]),
                         "r"(db[4 * c + 3])
                         : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(sP + off),
                         "r"(pb[4 * c]), "r"(pb[4 * c + 1]), "r"(pb[4 * c + 2]),
                         "r"(pb[4 * c + 3])
                         : "memory");
          }
        }
        tc_fence_before();
        mbar_arrive(sdp_free);
        fence_proxy_async();
        mbar_arrive(ds_full);
        mbar_arrive(p_full);
      }
      if (!ok) break;
      // ---- dQ = dQ^T -> bf16 (thread = d within each 128-d chunk)
      if (!(ok = W.wait(dq_done, nq & 1u))) break;
      tc_fence_after();
#pragma unroll 1
      for (int dc = 0; dc < C::kDChunks; ++dc) {
        const int d = dc * 128 + i;
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          float qv[32];
          tmem_ld32(tQ + dc * NH + lane_base + hh * 32, qv);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int h = hh * 32 + e;
            if (h < hcount)
              dq[(r * H + hb * 64 + h) * (int64_t)D + d] = __float2bfloat16_rn(qv[e]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tq_empty);
      mbar_arrive(toks_empty(buf));
      ++nq;
    }
  } else {
    // ========== scatter (256 threads): TMEM chunk -> fp32 reductions
    const int quad = warp & 3, half = (warp - kScWarp0) >> 2;  // chunk parity
    const int di = quad * 32 + lane;          // d within a 128-d chunk
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    uint32_t chunk = 0;
    int qi = 0;
    bool ok = true;
    for (;; ++qi) {
      const int buf = qi & 1;
      if (!(ok = W.wait(toks_full(buf), (qi >> 1) & 1))) break;
      if (item_s[buf] >= n_items) break;
      const int n = ntok[buf];
      const int npool = npool_s[buf];
      const int rot = rot_s[buf];
      const int32_t* pl = pools + buf * (K_p + 8);
      const int32_t* lc = pl + K_p;
      const int ntiles = (n + kTileK - 1) / kTileK;
#ifdef DSA_CHECKS
      const int64_t tq = t_hi - 1 - (int64_t)item_s[buf] / n_hblk;  // the query
#endif
      for (int j = 0; j < ntiles && ok; ++j) {
        const int jr = j + rot < ntiles ? j + rot : j + rot - ntiles;
        for (int which = 0; which < (KV ? 1 : 2) && ok; ++which) {
          float* acc = (which == 0 ? dk_acc : dv_acc) + di;  // KV: dKV
          // this half's chunks: q = half, half + 2, ... (chunk parity = half)
          for (int q = half; q < 4 * C::kDChunks; q += 2) {
            const uint32_t c = chunk + (uint32_t)q;
            const int dc = q >> 2, kq = q & 3;
            const int b = (int)(c & 3u);
            if (!(ok = W.wait(chunk_full(b), (c >> 2) & 1u))) break;
            tc_fence_after();
            float cv[32];  // d = dc*128 + di, keys kq*32 + e
            tmem_ld32(tC + b * 32 + lane_base, cv);
            tc_fence_before();
            mbar_arrive(chunk_empty(b));
            float* dst = acc + dc * 128;
            const int slot0 = jr * kTileK + kq * 32;
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
              const int s4 = slot0 + 4 * e4;  // 4 keys of one pool (or locals)
              if (s4 < npool) {
                const int32_t p = pl[s4 >> 2];
                // the pool's four keys come at or before the query
                if (p >= 0 && DSA_IN_BOUNDS((int64_t)4 * p + 3 <= tq, status))
                  red_add_pool<D>(dst + (int64_t)(4 * p) * D, cv[4 * e4], cv[4 * e4 + 1],
                                  cv[4 * e4 + 2], cv[4 * e4 + 3]);
              } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  if (s4 + e < n &&
                      DSA_IN_BOUNDS(lc[s4 + e - npool] >= 0 && lc[s4 + e - npool] <= tq, status))
                    red_add_f32(dst + (int64_t)lc[s4 + e - npool] * D, cv[4 * e4 + e]);
              }
            }
          }
          chunk += 4 * C::kDChunks;
        }
      }
      if (!ok) break;
      mbar_arrive(toks_empty(buf));
    }
  }

  // ---- teardown: every role has left its loop, no MMA or copy in flight
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaA) tmem_dealloc(tmem, 512);
}

template <int D, bool KV>
cudaError_t launch_t(const LaunchCtx& c, const AttnShape& s, const CUtensorMap& qm,
                     const CUtensorMap& gm, const __nv_bfloat16* k,
                     const __nv_bfloat16* v, const float* lse, const float* delta,
                     const int32_t* idx, __nv_bfloat16* dq, float* dk_acc,
                     float* dv_acc) {
  using C = BwdTcCfg<D>;
  const uint32_t smem = C::smem(s.K_p);
  if (smem > 232448) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_tc_kernel<D, KV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_bwd_tc_kernel<D, KV>,
                                                    kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) {
    cudaFuncAttributes fa;
    cudaFuncGetAttributes(&fa, attn_bwd_tc_kernel<D, KV>);
    set_error_detail("attn_bwd_tc occupancy 0: regs=%d threads=%d dyn_smem=%u "
                     "max_threads=%d",
                     fa.numRegs, kThreads, smem, fa.maxThreadsPerBlock);
    return cudaErrorLaunchOutOfResources;
  }
  const int n_hblk = (s.H + 63) / 64;
  const int64_t items = (s.t_hi - s.t_lo) * n_hblk;
  // the whole-sequence CTA count sets the tile rotation of every query
  const int64_t rot_div = (int64_t)c.num_sms < s.S * n_hblk ? c.num_sms : s.S * n_hblk;
  int64_t grid = c.num_sms;
  if (grid > items) grid = items;
  if (items <= 0) return cudaSuccess;
  // sched[0]: work counter; zeroed by the delta kernel
  uint32_t* sched = c.status + 32;
  attn_bwd_tc_kernel<D, KV><<<(unsigned)grid, kThreads, smem, c.stream>>>(
      qm, gm, k, v, lse, delta, idx, dq, dk_acc, dv_acc, s.t_lo, s.t_hi,
      (s.S - s.t_hi) * n_hblk, (int)rot_div, s.H, s.K_p, s.n_loc,
      s.scale, n_hblk, c.status, c.timeout_ns, sched);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd_tc(const LaunchCtx& c, const AttnShape& s,
                               const CUtensorMap& q_map, const CUtensorMap& g_map,
                               const __nv_bfloat16* k, const __nv_bfloat16* v,
                               const float* lse, const float* delta,
                               const int32_t* idx, __nv_bfloat16* dq, float* dk_acc,
                               float* dv_acc) {
  // dv_acc == nullptr: K and V are one tensor (k == v), dk_acc receives dKV
  const bool kv = dv_acc == nullptr;
#define DSA_BWD_CASE(DD)                                                          \
  if (s.D == DD)                                                                  \
    return kv ? launch_t<DD, true>(c, s, q_map, g_map, k, k, lse, delta, idx, dq,  \
                                   dk_acc, dk_acc)                                \
              : launch_t<DD, false>(c, s, q_map, g_map, k, v, lse, delta, idx, dq, \
                                    dk_acc, dv_acc);
  DSA_BWD_CASE(128) DSA_BWD_CASE(256) DSA_BWD_CASE(512)
#undef DSA_BWD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace dsa
