// indexer_topk.cu -- the lightning indexer with the top-k selection fused
// into its epilogue: no score is ever written to memory.
//
// The pages chunk the indexer over queries so that the score matrix never
// exists whole ("Scaling Training to 1M Token Context on GLM-5.3-Flash",
// section "Splitting the DSA Indexer / Over Time: Chunking"); this kernel
// goes to the end of that road.  One CTA owns an N tile of queries (256 /
// H_I of them, all their heads) and streams through every earlier pool in
// tiles of 128: the MMA and the score epilogue are those of indexer.cu
// (bit-identical fp32 scores), and each score is then offered to its
// query's running selection in shared memory instead of being stored.
//
// Streaming selection, exact under the lower-index tie rule.  A query keeps
// candidates (order key, pool) in pool order.  Until its first compaction
// every pool is a candidate; when the list passes kCap - kBM entries a warp
// compacts it to exactly K_p with a radix select (keys above the K-th, then
// the lowest-index ties), and from then on only keys strictly above that
// K-th key T are appended.  That is exact: the K_p kept entries all have
// key >= T and a lower pool index than any pool still to come, so a later
// key <= T can never be among the final K_p.  At the end of the tile the
// same select gives the answer, already in ascending pool order.
//
// Appends keep pool order: within a tile of 128 pools the four warps of a
// column half (one per TMEM lane quadrant, 32 pools each) exchange their
// counts and write at quadrant-ordered offsets.
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 TMEM allocator and
// MMA issuer, warps 2-9 epilogue and selection.  N tiles are dealt in
// descending query order (long rows first).
#include "attn_common.cuh"
#include "index_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kBM = 128;          // pools per tile
constexpr int kBN = 256;          // (query, head) columns per tile
constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kStages = 3;
constexpr int kCap = 1024;        // candidate slots per query
constexpr int kMaxK = kCap - 2 * kBM;  // K_p limit: a compaction frees >= kBM

template <int DI>
struct FusedCfg {
  static constexpr int KB = DI / 64;
  static constexpr uint32_t kABytes = kBM * DI * 2;
  static constexpr uint32_t kBBytes = kBN * DI * 2;
};

template <int HI, int DI>
constexpr uint32_t fused_smem() {
  return 1024 + FusedCfg<DI>::kBBytes + kStages * FusedCfg<DI>::kABytes +
         (kBN / HI) * kCap * 8 + 2 * 4 * 8 * 4 + 3 * 8 * 4 + 32 * 8;
}

// Hardware barriers among the epilogue warps (ids 1-3; 0 is __syncthreads).
// They cost a few cycles where an mbarrier round trip costs far more, and
// they are safe here: the only wait before them that can give up is the
// accumulator wait, whose outcome the warps first agree on with bar_and.
// Barrier that also ANDs one flag over all participating threads.
__device__ __forceinline__ bool bar_and(uint32_t id, uint32_t n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0u;
}

// Barrier that ORs one flag over all participating threads.
__device__ __forceinline__ bool bar_or(uint32_t id, uint32_t n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0u;
}

// Warp-wide exact selection over keys[0..n) (n > K, n <= 32 * 63): find
// the K-th largest key T by radix select over eight 4-bit digits, each lane
// counting its keys in a register-packed histogram (six bits per bin: bins
// 0-9 in one 64-bit word, 10-15 in another; no shared-memory atomics, which
// serialise when keys of similar magnitude share their top digits), then
// compact in place, in order, to the K entries that rank first under
// (key desc, position asc).  Returns T.
__device__ uint32_t warp_select(uint32_t* keys, int32_t* pools, int n, int K) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t prefix = 0u, pmask = 0u, kk = (uint32_t)K;
#pragma unroll 1
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 28 - 4 * pass;
    uint64_t lo = 0ull, hi = 0ull;
    for (int i = lane; i < n; i += 32) {
      const uint32_t key = keys[i];
      if ((key & pmask) == prefix) {
        const uint32_t d = (key >> shift) & 15u;
        if (d < 10u) lo += 1ull << (6u * d);
        else hi += 1ull << (6u * (d - 10u));
      }
    }
    uint32_t above = 0u, dsel = 0u;
#pragma unroll 1
    for (int b = 15; b >= 0; --b) {
      const uint32_t mine =
          (uint32_t)((b < 10 ? lo >> (6 * b) : hi >> (6 * (b - 10))) & 63ull);
      const uint32_t c = __reduce_add_sync(0xffffffffu, mine);
      if (above + c >= kk) {
        dsel = (uint32_t)b;
        break;
      }
      above += c;
    }
    prefix |= dsel << shift;
    pmask |= 15u << shift;
    kk -= above;
  }
  const uint32_t T = prefix;
  uint32_t gb = 0u, tb = 0u;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t key = i < n ? keys[i] : 0u;
    const int32_t pool = i < n ? pools[i] : 0;
    const bool gt = i < n && key > T;
    const bool tie = i < n && key == T;
    const uint32_t bg = __ballot_sync(0xffffffffu, gt);
    const uint32_t bt = __ballot_sync(0xffffffffu, tie);
    const uint32_t g_before = gb + __popc(bg & lt), t_before = tb + __popc(bt & lt);
    const bool keep = gt || (tie && t_before < kk);
    const uint32_t pos = gt ? g_before + min(t_before, kk) : g_before + t_before;
    __syncwarp();  // every read of this block precedes the writes (pos <= i)
    if (keep) {
      keys[pos] = key;
      pools[pos] = pool;
    }
    gb += __popc(bg);
    tb += __popc(bt);
    __syncwarp();
  }
  return T;
}

template <int HI, int DI>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_topk_kernel(const __grid_constant__ CUtensorMap q_map,
                        const __grid_constant__ CUtensorMap k_map,
                        const float* __restrict__ w, int64_t t_begin, int64_t t_end,
                        int K_p, int32_t* __restrict__ out, int64_t n_ntiles,
                        uint32_t* status, uint64_t timeout_ns) {
  using C = FusedCfg<DI>;
  constexpr int QT = kBN / HI;  // queries per N tile
  constexpr int QH = QT / 2;    // queries per column half
  constexpr uint32_t IDESC = idesc_bf16(kBM, kBN, 0, 0);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sB = base;
  const uint32_t sA = base + C::kBBytes;
  uint8_t* tail = gbase + C::kBBytes + kStages * C::kABytes;
  uint32_t* cand_key = reinterpret_cast<uint32_t*>(tail);              // [QT][kCap]
  int32_t* cand_pool = reinterpret_cast<int32_t*>(cand_key + QT * kCap);  // [QT][kCap]
  uint32_t* cw = reinterpret_cast<uint32_t*>(cand_pool + QT * kCap);  // [2][4][8]
  uint32_t* cnt = cw + 2 * 4 * 8;          // [8] candidates per query
  uint32_t* thr = cnt + 8;                 // [8] key threshold (after a compaction)
  uint32_t* compf = thr + 8;               // [8] compacted yet?
  uint64_t* bars = reinterpret_cast<uint64_t*>(compf + 8);
  const uint32_t bar0 = smem_u32(bars);
  auto a_full = [&](int s) { return bar0 + 8u * s; };
  auto a_empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  const uint32_t b_full = bar0 + 8u * (2 * kStages);
  const uint32_t b_empty = b_full + 8u;
  auto acc_full = [&](int a) { return b_full + 16u + 8u * a; };
  auto acc_empty = [&](int a) { return b_full + 32u + 8u * a; };
  const uint32_t done_bar = b_full + 48u;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(bars + 2 * kStages + 7);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Waiter W{abort_flag, status, timeout_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(a_full(s), 1);
      mbar_init(a_empty(s), 1);
    }
    mbar_init(b_full, 1);
    mbar_init(b_empty, 1);
    for (int a = 0; a < 2; ++a) {
      mbar_init(acc_full(a), 1);
      mbar_init(acc_empty(a), kEpiWarps);
    }
    mbar_init(done_bar, 1);
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

  // N tile k of this CTA, in descending query order; its pool tiles
  auto tile_of = [&](int64_t k, int64_t& nt, int64_t& tq0, int& n_pt) -> bool {
    const int64_t idx = blockIdx.x + k * gridDim.x;
    if (idx >= n_ntiles) return false;
    nt = n_ntiles - 1 - idx;
    tq0 = t_begin + nt * QT;
    const int64_t tql = tq0 + QT - 1 < t_end - 1 ? tq0 + QT - 1 : t_end - 1;
    n_pt = (int)((n_full(tql) + kBM - 1) / kBM);
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint64_t it = 0;
      int bcount = 0;
      int64_t nt, tq0;
      int n_pt;
      bool ok = true;
      for (int64_t k = 0; ok && tile_of(k, nt, tq0, n_pt); ++k) {
        if (n_pt == 0) continue;
        if (!(ok = W.wait(b_empty, (bcount & 1) ^ 1))) break;
        mbar_expect_tx(b_full, C::kBBytes);
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_2d(sB + kb * (kBN * 128), &q_map, kb * 64, (int32_t)(nt * kBN), b_full);
        ++bcount;
        for (int pt = 0; pt < n_pt && ok; ++pt, ++it) {
          const int s = (int)(it % kStages);
          if (!(ok = W.wait(a_empty(s), (uint32_t)((it / kStages) & 1u) ^ 1u))) break;
          mbar_expect_tx(a_full(s), C::kABytes);
#pragma unroll
          for (int kb = 0; kb < C::KB; ++kb)
            tma_load_2d(sA + s * C::kABytes + kb * (kBM * 128), &k_map, kb * 64,
                        (int32_t)(pt * kBM), a_full(s));
        }
      }
      // let every copy this thread issued land before the CTA can exit
      for (uint64_t j = it > (uint64_t)kStages ? it - kStages : 0; j < it; ++j)
        drain(a_full((int)(j % kStages)), (uint32_t)(j / kStages) & 1u, timeout_ns);
      if (bcount > 0) drain(b_full, (uint32_t)(bcount - 1) & 1u, timeout_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint64_t it = 0, local = 0;
      int bcount = 0;
      bool issued = false, ok = true;
      int64_t nt, tq0;
      int n_pt;
      for (int64_t k = 0; ok && tile_of(k, nt, tq0, n_pt); ++k) {
        if (n_pt == 0) continue;
        if (!(ok = W.wait(b_full, bcount & 1))) break;
        ++bcount;
        for (int pt = 0; pt < n_pt && ok; ++pt, ++it, ++local) {
          const int a = (int)(local & 1);
          const uint32_t v = (uint32_t)(local >> 1);
          if (!(ok = W.wait(acc_empty(a), (v & 1u) ^ 1u))) break;
          const int s = (int)(it % kStages);
          if (!(ok = W.wait(a_full(s), (uint32_t)(it / kStages) & 1u))) break;
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(a * kBN);
          const uint32_t a_tile = sA + s * C::kABytes;
#pragma unroll
          for (int ks = 0; ks < DI / 16; ++ks) {
            const int kb = ks >> 2, kin = ks & 3;
            tc_mma(d, sdesc_sw128(a_tile + kb * (kBM * 128) + kin * 32, 16, 1024),
                   sdesc_sw128(sB + kb * (kBN * 128) + kin * 32, 16, 1024), IDESC,
                   ks > 0 ? 1u : 0u);
          }
          issued = true;
          tc_commit(a_empty(s));
          tc_commit(acc_full(a));
        }
        if (ok) tc_commit(b_empty);
      }
      if (issued) {
        tc_commit(done_bar);
        drain(done_bar, 0, timeout_ns);
      }
    }
  } else {
    // ------------------------------------- epilogue + streaming selection
    const int ew = warp - 2;                // 0..7
    const int quad = warp & 3;              // TMEM lane quadrant
    const int half = ew >> 2;               // columns half*128 .. +127
    const uint32_t lt = (1u << lane) - 1u;
    uint64_t local = 0;
    float2 wr[kBN / 4];  // weights of this half's columns, in pairs (all lanes alike)
    int64_t nt, tq0;
    int n_pt;
    bool ok = true;
    for (int64_t k = 0; ok && tile_of(k, nt, tq0, n_pt); ++k) {
      const int64_t nq = t_end - tq0 < QT ? t_end - tq0 : QT;  // live queries
#pragma unroll
      for (int j = 0; j < kBN / 2; ++j) {
        const int col = half * (kBN / 2) + j;
        const int64_t qr = nt * QT + col / HI;  // row of w
        const float wj = col / HI < nq ? __ldg(w + qr * HI + (col % HI)) : 0.f;
        if (j & 1) wr[j >> 1].y = wj; else wr[j >> 1].x = wj;
      }
      if (ew < QT && lane == 0) {
        cnt[ew] = 0u;
        thr[ew] = 0u;
        compf[ew] = 0u;
      }
      named_bar(1, 32 * kEpiWarps);
      for (int pt = 0; pt < n_pt; ++pt, ++local) {
        const int a = (int)(local & 1);
        const uint32_t v = (uint32_t)(local >> 1);
        const bool got = W.wait(acc_full(a), v & 1u);
        if (!(ok = bar_and(1, 32 * kEpiWarps, got))) break;  // all warps agree
        tc_fence_after();
        const int64_t p = (int64_t)pt * kBM + quad * 32 + lane;
        const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) +
                               (uint32_t)(a * kBN + half * (kBN / 2));
        // scores of this half's queries, computed exactly as indexer.cu does
        float sc[QH];
        relu_weighted_sums<HI, kBN / 2, false>(
            taddr,
            [&](int i) {
              return make_float4(wr[2 * i].x, wr[2 * i].y, wr[2 * i + 1].x, wr[2 * i + 1].y);
            },
            [&](int qi, float score) { sc[qi] = score; }, [] {});
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty(a));
        // offer the scores: ballots per query, quadrant-ordered offsets
        uint32_t bal[QH];
        uint32_t keyv[QH];
        bool any = false;
#pragma unroll
        for (int qi = 0; qi < QH; ++qi) {
          const int q = half * QH + qi;
          const int64_t t = tq0 + q;
          const bool valid = q < nq && p < n_full(t);
          keyv[qi] = order_key(sc[qi]);
          const bool take = valid && (compf[q] == 0u || keyv[qi] > thr[q]);
          bal[qi] = __ballot_sync(0xffffffffu, take);
          any = any || bal[qi] != 0u;
          if (lane == 0) cw[(half * 4 + quad) * 8 + qi] = (uint32_t)__popc(bal[qi]);
        }
        // once the thresholds have risen most pool tiles add nothing: then
        // the append and compaction phases are skipped by every warp alike
        if (!bar_or(1, 32 * kEpiWarps, any)) continue;
#pragma unroll
        for (int qi = 0; qi < QH; ++qi) {
          const int q = half * QH + qi;
          uint32_t off = cnt[q];
          for (int qq = 0; qq < quad; ++qq) off += cw[(half * 4 + qq) * 8 + qi];
          if ((bal[qi] >> lane) & 1u) {
            const uint32_t pos = off + (uint32_t)__popc(bal[qi] & lt);
            cand_key[q * kCap + pos] = keyv[qi];
            cand_pool[q * kCap + pos] = (int32_t)p;
          }
        }
        named_bar(1, 32 * kEpiWarps);
        // warp ew updates query ew's count and compacts it when nearly full
        if (ew < QT) {
          const int h = ew / QH, qi = ew % QH;
          uint32_t add = 0u;
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) add += cw[(h * 4 + qq) * 8 + qi];
          uint32_t n = cnt[ew] + add;
          if (n > (uint32_t)(kCap - kBM)) {
            const uint32_t T = warp_select(cand_key + ew * kCap, cand_pool + ew * kCap,
                                           (int)n, K_p);
            n = (uint32_t)K_p;
            if (lane == 0) {
              thr[ew] = T;
              compf[ew] = 1u;
            }
          }
          __syncwarp();
          if (lane == 0) cnt[ew] = n;
        }
        named_bar(1, 32 * kEpiWarps);
      }
      if (!ok) break;
      // ---- the answer: the K_p best candidates, already in pool order
      if (ew < QT && ew < nq) {
        const int64_t t = tq0 + ew;
        uint32_t n = cnt[ew];
        if (n > (uint32_t)K_p) {
          warp_select(cand_key + ew * kCap, cand_pool + ew * kCap, (int)n, K_p);
          n = (uint32_t)K_p;
        }
        int32_t* o = out + (t - t_begin) * (int64_t)K_p;
        for (int i = lane; i < K_p; i += 32)
          o[i] = i < (int)n ? cand_pool[ew * kCap + i] : -1;
      }
      named_bar(1, 32 * kEpiWarps);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int HI, int DI>
cudaError_t launch_t(const LaunchCtx& c, const CUtensorMap& q_map, const CUtensorMap& k_map,
                     const float* w, int64_t t_begin, int64_t t_end, int K_p,
                     int32_t* out) {
  constexpr uint32_t smem = fused_smem<HI, DI>();
  static_assert(smem <= 232448, "shared memory");
  constexpr int QT = kBN / HI;
  const int64_t n_ntiles = (t_end - t_begin + QT - 1) / QT;
  if (n_ntiles == 0) return cudaSuccess;
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = set_smem_once(indexer_topk_kernel<HI, DI>, (int)smem, smem_set);
  if (e != cudaSuccess) return e;
  const int64_t grid = n_ntiles < c.num_sms ? n_ntiles : c.num_sms;
  indexer_topk_kernel<HI, DI><<<(unsigned)grid, kThreads, smem, c.stream>>>(
      q_map, k_map, w, t_begin, t_end, K_p, out, n_ntiles, c.status, c.timeout_ns);
  return cudaGetLastError();
}

}  // namespace

bool indexer_topk_supported(int H_I, int D_I, int K_p) {
  return (H_I == 32 || H_I == 64) && (D_I == 64 || D_I == 128) && K_p >= 1 &&
         K_p <= kMaxK;
}

cudaError_t launch_indexer_topk(const LaunchCtx& c, const CUtensorMap& q_map,
                                const CUtensorMap& k_map, const float* w, int H_I,
                                int D_I, int64_t t_begin, int64_t t_end, int K_p,
                                int32_t* out) {
  if (!indexer_topk_supported(H_I, D_I, K_p)) return cudaErrorInvalidValue;
  if (H_I == 32 && D_I == 128) return launch_t<32, 128>(c, q_map, k_map, w, t_begin, t_end, K_p, out);
  if (H_I == 32 && D_I == 64) return launch_t<32, 64>(c, q_map, k_map, w, t_begin, t_end, K_p, out);
  if (H_I == 64 && D_I == 128) return launch_t<64, 128>(c, q_map, k_map, w, t_begin, t_end, K_p, out);
  return launch_t<64, 64>(c, q_map, k_map, w, t_begin, t_end, K_p, out);
}

}  // namespace dsa
