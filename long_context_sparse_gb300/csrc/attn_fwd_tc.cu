// attn_fwd_tc.cu -- causal sparse attention forward on 5th-generation tensor
// cores (tcgen05 + TMEM), one query per CTA at a time, persistent.
//
// "the attention reads only those 2048 tokens, so attention cost grows
// linearly" ("Scaling Training to 1M Token Context on GLM-5.3-Flash",
// section "DeepSeek Sparse Attention (DSA) Optimizations"); NoPE q/k and the
// 2,051-key variant (section "Making Sparse Attention Actually Sparse").
//
// One K row and one V row per token serve every head of the query, so a
// gathered tile of 128 keys is the M dimension of both products and the
// query's heads are N:
//   S^T[key, h]   = K_tile[key, :] . Q[h, :]        M=128 keys, N=heads, K=D
//   O^T[dv, h]   += V_tile[:, dv]^T . P^T[key, h]    M=128 dv,   N=heads,
//                                                    K=128 keys (per 128 dv)
// S^T (double-buffered) and O^T live in TMEM (fp32).  The gather runs one
// tile ahead for K: K(j+1) is fetched before V(j), so S^T of the next tile
// is computed while the softmax of this one runs, and the tensor core does
// not wait for it.  Each softmax thread owns one key (one
// TMEM lane): it reads its row of S^T, column maxima are taken across the
// 128 lanes, and it writes P (bf16) into shared memory as the B operand of
// the second product: with 64 heads as a row of 64 heads per key (16-byte
// stores, MN-major operand), with fewer as a row of 128 keys per head.  A running maximum is only
// raised when a tile beats it by more than 2^8, so O^T is rarely rescaled
// (the final normalisation uses the same maximum, so the result is exact).
//
// Warps: 4 or 8 softmax / epilogue warps (one warpgroup per 32 heads; warp
// w reads TMEM lane quadrant w % 4), 7 gather producers (cp.async of the
// selected K/V rows into 128-byte-swizzled stages, completion signalled on
// an mbarrier; the gather rate grows with the number of issuing warps, and
// 16 warps have the same register budget as 13), 1 MMA issuer and TMEM
// owner.  Q comes in by TMA.  Every wait is bounded
// (DSA_ERR_DEVICE_TIMEOUT).
//
// Scheduling: CTAs take queries from a global counter in descending t, and
// query number i starts at tile (i * ntiles / CTAs) mod ntiles, wrapping
// around: the band of tiles the grid has reached when the query is taken.
// A query's key list is sorted, so tile j of every recent query covers
// about the same band of keys: the CTAs then gather from the same
// L2-resident band of K/V at any time.  The order is a function of the
// query alone, so results repeat bit for bit.
#include "attn_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kTileK = 128;            // keys per tile (MMA M)
constexpr int kStages = 4;             // gather ring depth
constexpr uint32_t kStageBytes = 32768;  // 128 keys x 128 dims (2 atoms)
constexpr int kProdThreads = 224;    // 7 gather warps
constexpr int kProdWarps = kProdThreads / 32;
constexpr float kMaxSlack = 8.0f;      // log2 headroom before raising a max
constexpr int kMaskWords = (2048 * 4 + 3 + kTileK + 31) / 32;

template <int D, int NH>
struct TcFwdCfg {
  // softmax warpgroups: each owns HPG heads of all 128 keys
  static constexpr int kGroups = NH > 32 ? 2 : 1;
  static constexpr int HPG = NH / kGroups;
  static constexpr int kSoftmaxThreads = 128 * kGroups;
  static constexpr int kProdWarp0 = 4 * kGroups;       // first producer warp
  static constexpr int kMmaWarp = kProdWarp0 + kProdThreads / 32;
  static constexpr int kThreads = kSoftmaxThreads + kProdThreads + 32;
  // registers per thread: warps are spread over the SM's 4 sub-partitions
  // of 16K registers each, so the fullest one holds ceil(warps/4) warps
  static constexpr int kRegFit = (16384 / (((kThreads / 32) + 3) / 4 * 32)) & ~7;
  static constexpr int kMaxReg = kRegFit > 255 ? 255 : kRegFit;
  static constexpr int kChunks = D / 128;  // 128-wide d slices
  static constexpr uint32_t kQBytes = NH * D * 2;
  static constexpr uint32_t kPBytes = NH * kTileK * 2;
  static constexpr uint32_t kTmemCols = 2 * NH + kChunks * NH <= 256 ? 256 : 512;
  static constexpr bool kPRows = NH == 64;  // P as [key][64 heads] rows
  // dynamic shared memory for a key list of `cap` entries
  // dynamic shared memory: the selected pool ids (K_p) + 4 local tokens
  static uint32_t smem(int K_p) {
    return 1024 + kQBytes + kPBytes + kStages * kStageBytes + carved((K_p + 4) * 4) +
           carved(2 * kMaskWords * 4) + carved(4 * NH * 4) +
           3 * carved(NH * 4) + carved(48) + carved(32 * 8);
  }
};


// NH consecutive fp32 columns of this thread's TMEM lane.
template <int NH>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, float (&v)[NH]) {
  uint32_t r[NH];
#pragma unroll
  for (int c = 0; c < NH; c += 16)
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,"
        "%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[c + 0]), "=r"(r[c + 1]), "=r"(r[c + 2]), "=r"(r[c + 3]),
          "=r"(r[c + 4]), "=r"(r[c + 5]), "=r"(r[c + 6]), "=r"(r[c + 7]),
          "=r"(r[c + 8]), "=r"(r[c + 9]), "=r"(r[c + 10]), "=r"(r[c + 11]),
          "=r"(r[c + 12]), "=r"(r[c + 13]), "=r"(r[c + 14]), "=r"(r[c + 15])
        : "r"(taddr + c));
  tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < NH; ++c) v[c] = __uint_as_float(r[c]);
}


template <int D, int NH>
__global__ void __maxnreg__((TcFwdCfg<D, NH>::kMaxReg))
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap q_map,
                       const __nv_bfloat16* __restrict__ k,
                       const __nv_bfloat16* __restrict__ v,
                       const int32_t* __restrict__ idx,
                       __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                       int64_t t_lo, int64_t t_hi, int64_t item0, int rot_div,
                       int H, int K_p, int n_loc, float scale_log2,
                       int n_hblk, uint32_t* status,
                       uint64_t timeout_ns, uint32_t* sched) {
  using C = TcFwdCfg<D, NH>;
  constexpr int HPG = C::HPG;
  constexpr int kSoftmaxThreads = C::kSoftmaxThreads;
  constexpr uint32_t IDESC_S = idesc_bf16(128, NH, 0, 0);  // K-major A and B
  constexpr uint32_t IDESC_O = idesc_bf16(128, NH, 1, C::kPRows ? 1 : 0);  // MN-major A

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sP = sQ + C::kQBytes;
  const uint32_t sStage = sP + C::kPBytes;  // 1024-aligned (sizes are)
  // key list of the current query as pool ids (slot 4i+j <-> token
  // 4*pools[i]+j, -1 = empty) followed by up to 3 local tokens; each tail
  // region starts on a 128-byte boundary
  uint8_t* tail = gb + C::kQBytes + C::kPBytes + kStages * kStageBytes;
  int32_t* pools = carve<int32_t>(tail, K_p + 4);
  int32_t* locs = pools + K_p;
  uint32_t* vmask = carve<uint32_t>(tail, 2 * kMaskWords);    // [2][words]
  float* red = carve<float>(tail, 4 * NH);                    // [4][NH]
  float* m_s = carve<float>(tail, NH);                        // [NH]
  float* alpha_s = carve<float>(tail, NH);                    // [NH]
  float* inv_s = carve<float>(tail, NH);                      // [NH]
  int* misc = carve<int>(tail, 12);  // ntok[2] last nadd flag[2] item[2] rot[2]
  uint64_t* bars = carve<uint64_t>(tail, 32);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  const uint32_t q_full = bar0 + 8u * (2 * kStages);
  const uint32_t q_empty = q_full + 8u;
  const uint32_t p_full = q_full + 16u;
  const uint32_t pv_done = q_full + 24u;
  const uint32_t o_empty = q_full + 32u;
  const uint32_t done_bar = q_full + 40u;
  auto toks_full = [&](int b) { return q_full + 48u + 8u * b; };
  auto toks_empty = [&](int b) { return q_full + 64u + 8u * b; };
  const uint32_t sm_grp = q_full + 80u;    // softmax group barrier
  const uint32_t prod_grp = q_full + 88u;  // producer group barrier
  auto s_full = [&](int b) { return q_full + 96u + 8u * b; };   // S^T buffer b ready
  auto s_free = [&](int b) { return q_full + 112u + 8u * b; };  // S^T buffer b read
  const uint32_t p_done = q_full + 128u;  // a PV product completed (P, O^T free)
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(bars + 2 * kStages + 17);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 18);
  int* ntok = misc;
  int* s_last = misc + 2;
  int* s_nadd = misc + 3;
  volatile int* flags = misc + 4;
  int* item_s = misc + 6;  // [2] query of the buffer (>= n_items: no more)
  int* rot_s = misc + 8;   // [2] first tile of the query (rotation)
  uint32_t* work_ctr = sched;  // next query to take

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Waiter W{abort_flag, status, timeout_ns};
  // queries t_lo .. t_hi-1, latest first; row r = t - t_lo of q, idx, o
  // and lse; item0 + item numbers the query as a whole-sequence call would
  const int64_t n_items = (t_hi - t_lo) * n_hblk;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), kProdThreads);
      mbar_init(empty(s), 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(s_free(b), kSoftmaxThreads);
    }
    mbar_init(p_done, 1);
    mbar_init(p_full, kSoftmaxThreads);
    mbar_init(pv_done, 1);
    mbar_init(o_empty, kSoftmaxThreads);
    mbar_init(done_bar, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(toks_full(b), kProdThreads);
      mbar_init(toks_empty(b), kSoftmaxThreads);
    }
    mbar_init(sm_grp, kSoftmaxThreads);
    mbar_init(prod_grp, kProdThreads);
    *abort_flag = 0u;
    flags[0] = flags[1] = 0;
    fence_mbar_init();
    prefetch_tensormap(&q_map);
  }
  if (warp == C::kMmaWarp) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;           // S^T: 2 buffers x NH columns
  const uint32_t tO = tmem + 2 * NH;  // O^T: kChunks x NH columns

  if (warp >= C::kProdWarp0 && warp < C::kMmaWarp) {
    // ============================================ gather producers (128)
    const int ptid = tid - kSoftmaxThreads;
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
      // ---- key list of query t: tokens of the selected pools, then the
      // local tokens no selected pool covers; validity bits for softmax
      const int32_t* row = idx + r * K_p;
      const int64_t nf = n_full(t);
      uint32_t* vm = vmask + buf * kMaskWords;
      if (ptid == 0) {
        *s_last = -1;
        *s_nadd = 0;
      }
      for (int w = ptid; w < kMaskWords; w += kProdThreads) vm[w] = 0u;
      if (!G.sync(W)) break;
      for (int i = ptid; i < K_p; i += kProdThreads) {
        const int32_t p = __ldg(row + i);
        const bool okp = p >= 0 && (int64_t)p < nf;
        if (p >= 0) {
          atomicMax(s_last, i);
          if (!okp) latch_error(status, DSA_ERR_DEVICE_BAD_INDEX);
        }
        pools[i] = okp ? p : -1;
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
              locs[nadd] = (int32_t)s;
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
      if (!G.sync(W)) break;
      if (ptid == 0) {
        ntok[buf] = n;
        // tile band of this query's generation: queries are taken in order
        // and every CTA works through ntiles tiles per query, so about
        // item * ntiles / CTAs tiles per CTA have been gathered when it
        // starts; counted in whole-sequence items over the whole-sequence
        // CTA count, a pure function of the query, so that results repeat
        // exactly, whatever range the call covers
        rot_s[buf] = ntiles > 0
                         ? (int)(((uint64_t)(item0 + item) * (uint64_t)ntiles / (uint64_t)rot_div) %
                                 (uint64_t)ntiles)
                         : 0;
      }
      if (!G.sync(W)) break;
      mbar_arrive(toks_full(buf));  // release: list, mask, count, rotation
      if (ntiles == 0) continue;
      // ---- Q rows of this head block by TMA (box {64, NH} per 64-wide d)
      if (ptid == 0 && W.wait(q_empty, (nq & 1u) ^ 1u)) {
        mbar_expect_tx(q_full, C::kQBytes);
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          tma_load_2d(sQ + a * (NH * 128), &q_map, a * 64,
                      (int32_t)(r * H + hb * 64), q_full);
      }
      ++nq;
      // ---- K then V slices of every tile through the stage ring; thread
      // ptid copies key rows ptid and ptid+64 of the tile (256 B per slice)
      auto tok_of = [&](int slot) -> int32_t {
        if (slot < npool) {
          const int32_t p = pools[slot >> 2];
          return p >= 0 ? 4 * p + (slot & 3) : -1;
        }
        return slot < n ? locs[slot - npool] : -1;
      };
      // Coalesced gather: one warp instruction copies 2 key rows x 256
      // contiguous bytes (lanes 0-15 row r, lanes 16-31 row r+1; lane&15 =
      // the 16-byte chunk); the 64 row pairs of a stage are dealt
      // round-robin to the producer warps.
      const int pw = ptid >> 5, pl = ptid & 31;
      const int sub = pl >> 4, c16 = pl & 15;     // row of the pair, chunk
      const int a16 = c16 >> 3, ch8 = c16 & 7;    // 64-dim atom, 16B chunk
      const int rot = rot_s[buf];
      bool ok = true;
      // order: K(0), then K(j), V(j-1) for j = 1 .. ntiles-1, then V(last).
      // Each lane keeps the tokens of its own rows (r = 2g + sub, g = pw +
      // x * kProdWarps) in registers: those of tile j for K, and the
      // previous tile's for V, so the producer warps share no table and
      // need no barrier between tiles (they stay within the ring's reach of
      // each other through the stage barriers)
      constexpr int kRowsPerLane = (kTileK / 2 + kProdWarps - 1) / kProdWarps;
      int32_t tokK[kRowsPerLane], tokV[kRowsPerLane];
#pragma unroll
      for (int x = 0; x < kRowsPerLane; ++x) tokK[x] = -1;
      for (int j = 0; j <= ntiles && ok; ++j) {
#pragma unroll
        for (int x = 0; x < kRowsPerLane; ++x) tokV[x] = tokK[x];
        if (j < ntiles) {
          const int jr = j + rot < ntiles ? j + rot : j + rot - ntiles;
#pragma unroll
          for (int x = 0; x < kRowsPerLane; ++x) {
            const int g = pw + x * kProdWarps;
            tokK[x] = g < kTileK / 2 ? tok_of(jr * kTileK + 2 * g + sub) : -1;
          }
        }
        for (int kv = 0; kv < 2 && ok; ++kv) {
          if (kv == 0 ? j == ntiles : j == 0) continue;
          const __nv_bfloat16* src = kv == 0 ? k : v;
          for (int c = 0; c < C::kChunks; ++c, ++u) {
            const int s = (int)(u % kStages);
            if (!(ok = W.wait(empty(s), ((u / kStages) & 1u) ^ 1u))) break;
            const uint32_t st = sStage + s * kStageBytes + a16 * 16384;
#pragma unroll
            for (int x = 0; x < kRowsPerLane; ++x) {
              const int g = pw + x * kProdWarps;
              if (g >= kTileK / 2) continue;
              const int r = 2 * g + sub;
              const int32_t tok = kv == 0 ? tokK[x] : tokV[x];
              const __nv_bfloat16* sp =
                  src + (int64_t)(tok >= 0 ? tok : 0) * D + c * 128 + c16 * 8;
              const uint32_t dst = st + r * 128 + ((ch8 ^ (r & 7)) << 4);
              // inside the ring, and no key after the query
              if (DSA_IN_BOUNDS(dst - sStage < (uint32_t)(kStages * kStageBytes) && tok <= t,
                                status))
                cp_async16(dst, sp, tok >= 0 ? 16u : 0u);
            }
            cp_async_mbar_arrive(full(s));
          }
        }
      }
      if (!ok) break;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == C::kMmaWarp) {
    // ================================================== MMA issuer
    if (lane == 0) {
      uint32_t u = 0, ntile_all = 0, nq = 0;
      int qi = 0;
      bool issued = false, ok = true;
      for (;; ++qi) {
        const int buf = qi & 1;
        if (!(ok = W.wait(toks_full(buf), (qi >> 1) & 1))) break;
        if (item_s[buf] >= n_items) break;
        const int n = ntok[buf];
        const int ntiles = (n + kTileK - 1) / kTileK;
        if (ntiles == 0) continue;
        if (!(ok = W.wait(q_full, nq & 1u))) break;
        // step j: S^T of tile j (if any), then O^T += V^T P^T of tile j-1
        for (int j = 0; j <= ntiles && ok; ++j) {
          if (j < ntiles) {
            const uint32_t T = ntile_all + (uint32_t)j;
            const int b = (int)(T & 1u);
            // the softmax has read this buffer's S^T of tile T-2
            if (!(ok = W.wait(s_free(b), ((T >> 1) & 1u) ^ 1u))) break;
            tc_fence_after();
            // ---- S^T = K_tile Q^T (accumulated over the D/128 slices)
            for (int c = 0; c < C::kChunks; ++c, ++u) {
              const int s = (int)(u % kStages);
              if (!(ok = W.wait(full(s), (u / kStages) & 1u))) break;
              fence_proxy_async();  // cp.async (generic) -> tensor core (async)
              tc_fence_after();
              const uint32_t st = sStage + s * kStageBytes;
#pragma unroll
              for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int kin = 0; kin < 4; ++kin) {
                  const uint64_t ad = sdesc_sw128(st + a * 16384 + kin * 32, 16, 1024);
                  const uint64_t bd =
                      sdesc_sw128(sQ + (2 * c + a) * (NH * 128) + kin * 32, 16, 1024);
                  tc_mma(tS + b * NH, ad, bd, IDESC_S, (c | a | kin) != 0 ? 1u : 0u);
                }
              issued = true;
              tc_commit(empty(s));
            }
            if (!ok) break;
            if (j == ntiles - 1) tc_commit(q_empty);
            tc_commit(s_full(b));
          }
          if (j >= 1) {
            const int jp = j - 1;
            const uint32_t T = ntile_all + (uint32_t)jp;
            // ---- O^T += V_tile^T P^T
            if (!(ok = W.wait(p_full, T & 1u))) break;
            if (jp == 0 && !(ok = W.wait(o_empty, (nq & 1u) ^ 1u))) break;
            tc_fence_after();
            for (int c = 0; c < C::kChunks; ++c, ++u) {
              const int s = (int)(u % kStages);
              if (!(ok = W.wait(full(s), (u / kStages) & 1u))) break;
              fence_proxy_async();
              tc_fence_after();
              const uint32_t st = sStage + s * kStageBytes;
#pragma unroll
              for (int ks = 0; ks < kTileK / 16; ++ks) {
                // A = V^T [128 dv x 16 keys], MN-major: two 64-dv atoms 16 KB
                // apart (LBO), 8-key groups 1024 B apart (SBO)
                const uint64_t ad = sdesc_sw128(st + ks * 2048, 16384, 1024);
                // B = P^T [NH heads x 16 keys]: rows of 64 heads per key
                // (MN-major) or rows of 128 keys per head (K-major)
                const uint64_t bd =
                    C::kPRows
                        ? sdesc_sw128(sP + ks * 2048, 16, 1024)
                        : sdesc_sw128(sP + (ks >> 2) * (NH * 128) + (ks & 3) * 32, 16, 1024);
                tc_mma(tO + c * NH, ad, bd, IDESC_O, (jp | ks) != 0 ? 1u : 0u);
              }
              tc_commit(empty(s));
            }
            if (!ok) break;
            tc_commit(p_done);
            if (jp == ntiles - 1) tc_commit(pv_done);
          }
        }
        ntile_all += (uint32_t)ntiles;
        ++nq;
      }
      if (issued) {
        tc_commit(done_bar);
        drain(done_bar, 0, timeout_ns);
      }
    }
  } else {
    // ============================== softmax + epilogue (128 per group)
    const int i = tid & 127;  // key lane while scoring, dv lane in epilogue
    const int grp = tid >> 7;  // heads grp*HPG .. grp*HPG+HPG-1
    const int h0g = grp * HPG;
    const int wq = warp & 3;   // TMEM lane quadrant
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    GroupBar G{sm_grp, 0u};
    uint32_t ntile_all = 0, nq = 0;
    int qi = 0;
    // address pieces of P^T element (h, key i), K-major 128-byte rows
    const uint32_t p_off = (uint32_t)(i >> 6) * (NH * 128) + (uint32_t)(i & 7) * 2;
    const uint32_t p_chunk = (uint32_t)((i & 63) >> 3);
    for (;; ++qi) {
      const int buf = qi & 1;
      if (!W.wait(toks_full(buf), (qi >> 1) & 1)) break;
      const int64_t item = item_s[buf];
      if (item >= n_items) break;
      const int64_t r = t_hi - 1 - item / n_hblk - t_lo;  // row of o and lse
      const int hb = (int)(item % n_hblk);
      const int hcount = min(NH, H - hb * 64);
      const int n = ntok[buf];
      const int rot = rot_s[buf];
      const uint32_t* vm = vmask + buf * kMaskWords;
      const int ntiles = (n + kTileK - 1) / kTileK;
      __nv_bfloat16* orow = o + (r * H + hb * 64) * (int64_t)D;
      if (ntiles == 0) {  // empty key set: O = 0, LSE = -inf
        for (int e = tid; e < hcount * D; e += kSoftmaxThreads)
          orow[e] = __float2bfloat16_rn(0.f);
        if (tid < hcount) lse[r * H + hb * 64 + tid] = -INFINITY;
        mbar_arrive(toks_empty(buf));
        continue;
      }
      if (tid < NH) m_s[tid] = -INFINITY;
      // row-sum partials; the running maxima are m_s[] (shared, the same
      // for every thread of a head)
      float l[HPG];
#pragma unroll
      for (int h = 0; h < HPG; ++h) l[h] = 0.f;
      bool ok = true;
      for (int j = 0; j < ntiles; ++j, ++ntile_all) {
        const int sb = (int)(ntile_all & 1u);
        const uint32_t tSb = tS + sb * NH;
        if (!(ok = W.wait(s_full(sb), (ntile_all >> 1) & 1u))) break;
        tc_fence_after();
        const int jr = j + rot < ntiles ? j + rot : j + rot - ntiles;
        const int slot = jr * kTileK + i;
        const bool valid = (vm[slot >> 5] >> (slot & 31)) & 1u;
        // does any score beat its running max by more than 2^8?  (always
        // true on the first tile, which also avoids reading m_s before its
        // reset is visible; rare afterwards).  S^T is read from TMEM in
        // groups of 16 columns to keep few scores live.
        bool need = j == 0;
        if (j > 0) {
#pragma unroll
          for (int h0 = 0; h0 < HPG; h0 += 16) {
            uint32_t r[16];
            tmem_ld16(tSb + lane_base + h0g + h0, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float x = valid ? __uint_as_float(r[e]) * scale_log2 : -INFINITY;
              const float m = m_s[h0g + h0 + e];
              need |= x > m + kMaxSlack || (m == -INFINITY && x > m);
            }
          }
        }
        if (__any_sync(0xffffffffu, need) && lane == 0) atomicOr((int*)&flags[j & 1], 1);
        if (!(ok = G.sync(W))) break;
        if (tid == 0) flags[(j + 1) & 1] = 0;  // next tile's flag (read two syncs ago)
        // the previous PV product has completed: O^T is current and P's
        // buffer is free
        if (ntile_all > 0 && !(ok = W.wait(p_done, (ntile_all - 1u) & 1u))) break;
        tc_fence_after();
        if (flags[j & 1] != 0) {
          // ---- slow path: exact column maxima, raise the beaten maxima
#pragma unroll
          for (int h0 = 0; h0 < HPG; h0 += 16) {
            uint32_t r[16];
            tmem_ld16(tSb + lane_base + h0g + h0, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float x = valid ? __uint_as_float(r[e]) * scale_log2 : -INFINITY;
#pragma unroll
              for (int sh = 16; sh > 0; sh >>= 1)
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, sh));
              if (lane == 0) red[wq * NH + h0g + h0 + e] = x;
            }
          }
          if (!(ok = G.sync(W))) break;
          if (tid < NH) {
            const float tm = fmaxf(fmaxf(red[tid], red[NH + tid]),
                                   fmaxf(red[2 * NH + tid], red[3 * NH + tid]));
            const float mo = m_s[tid];
            const bool raise = tm > mo + kMaxSlack || (mo == -INFINITY && tm > mo);
            alpha_s[tid] = raise && mo != -INFINITY ? exp2f(mo - tm) : 1.f;
            if (raise) m_s[tid] = tm;
          }
          if (!(ok = G.sync(W))) break;
          bool rescale = false;
#pragma unroll
          for (int h = 0; h < HPG; ++h) {
            const float a = alpha_s[h0g + h];
            l[h] *= a;
            rescale |= a != 1.f;
          }
          if (j > 0 && __any_sync(0xffffffffu, rescale)) {
            // O^T columns of raised maxima (the previous PV has completed)
#pragma unroll 1
            for (int c = 0; c < C::kChunks; ++c) {
#pragma unroll
              for (int hh = 0; hh < HPG; hh += 16) {
                uint32_t r[16];
                const uint32_t ta = tO + lane_base + c * NH + h0g + hh;
                tmem_ld16(ta, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha_s[h0g + hh + e]);
                tmem_st16(ta, r);
              }
            }
            tmem_wait_st();
          }
        }
        // P = exp2(s - m) -> row sums and P (bf16) in shared memory
        uint32_t pk[HPG / 2];  // P of this thread's heads, bf16 pairs
#pragma unroll
        for (int h0 = 0; h0 < HPG; h0 += 16) {
          uint32_t r[16];
          tmem_ld16(tSb + lane_base + h0g + h0, r);
          tmem_wait_ld();
          float pv[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int h = h0 + e, hh = h0g + h;
            const float x = valid ? __uint_as_float(r[e]) * scale_log2 : -INFINITY;
            const float m = m_s[hh];
            pv[e] = exp2f(x - (m == -INFINITY ? 0.f : m));
            l[h] += pv[e];
          }
#pragma unroll
          for (int e = 0; e < 16; e += 2) pk[(h0 + e) >> 1] = pack_bf16(pv[e], pv[e + 1]);
        }
        tc_fence_before();
        mbar_arrive(s_free(sb));  // S^T of this tile fully read
        if constexpr (C::kPRows) {
          // row i: 64 heads = 8 chunks of 16 B, this group's 4 chunks
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t ch = (uint32_t)(grp * 4 + c);
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(
                             sP + (uint32_t)i * 128u + ((ch ^ (uint32_t)(i & 7)) << 4)),
                         "r"(pk[4 * c]), "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]),
                         "r"(pk[4 * c + 3])
                         : "memory");
          }
        } else {
#pragma unroll
          for (int h = 0; h < HPG; ++h) {
            const int hh = h0g + h;
            const uint32_t addr = sP + p_off + (uint32_t)hh * 128u +
                                  ((p_chunk ^ (uint32_t)(hh & 7)) << 4);
            const uint16_t b16 = (uint16_t)((h & 1) ? (pk[h >> 1] >> 16) : (pk[h >> 1] & 0xFFFFu));
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(b16) : "memory");
          }
        }
        fence_proxy_async();  // P^T writes -> tensor core reads
        tc_fence_before();
        mbar_arrive(p_full);
      }
      if (!ok) break;
      // ---- epilogue: last PV done -> row sums, LSE, O = O^T / l
      if (!W.wait(pv_done, nq & 1u)) break;
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < HPG; ++h) {
        float x = l[h];
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) x += __shfl_xor_sync(0xffffffffu, x, sh);
        if (lane == 0) red[wq * NH + h0g + h] = x;
      }
      if (!G.sync(W)) break;
      if (tid < NH) {
        const float lt =
            red[tid] + red[NH + tid] + red[2 * NH + tid] + red[3 * NH + tid];
        inv_s[tid] = lt > 0.f ? 1.f / lt : 0.f;
        if (tid < hcount)
          lse[r * H + hb * 64 + tid] =
              lt > 0.f ? (m_s[tid] + log2f(lt)) * kLn2 : -INFINITY;
      }
      if (!G.sync(W)) break;
#pragma unroll 1
      for (int c = 0; c < C::kChunks; ++c) {
        float ov[HPG];
        tmem_ld_row<HPG>(tO + lane_base + c * NH + h0g, ov);
        const int d = c * 128 + i;
#pragma unroll
        for (int h = 0; h < HPG; ++h)
          if (h0g + h < hcount)
            orow[(h0g + h) * (int64_t)D + d] = __float2bfloat16_rn(ov[h] * inv_s[h0g + h]);
      }
      tc_fence_before();
      mbar_arrive(o_empty);
      mbar_arrive(toks_empty(buf));
      ++nq;
    }
  }

  // ---- teardown: every role has left its loop, no MMA or copy in flight
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::kMmaWarp) tmem_dealloc(tmem, C::kTmemCols);
}

template <int D, int NH>
cudaError_t launch_t(const LaunchCtx& c, const AttnShape& s, const CUtensorMap& qm,
                     const __nv_bfloat16* k, const __nv_bfloat16* v,
                     const int32_t* idx, __nv_bfloat16* o, float* lse) {
  using C = TcFwdCfg<D, NH>;
  const uint32_t smem = C::smem(s.K_p);
  if (smem > 232448) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_kernel<D, NH>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_fwd_tc_kernel<D, NH>,
                                                    C::kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) {
    cudaFuncAttributes fa;
    cudaFuncGetAttributes(&fa, attn_fwd_tc_kernel<D, NH>);
    int dev = 0, optin = 0, per_smem = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaDeviceGetAttribute(&per_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    set_error_detail("attn_fwd_tc occupancy 0: regs=%d threads=%d static_smem=%zu "
                     "dyn_smem=%u optin=%d smem_per_sm=%d max_threads=%d",
                     fa.numRegs, C::kThreads, fa.sharedSizeBytes, smem, optin,
                     per_smem, fa.maxThreadsPerBlock);
    return cudaErrorLaunchOutOfResources;
  }
  const int n_hblk = (s.H + 63) / 64;
  const int64_t items = (s.t_hi - s.t_lo) * n_hblk;
  // the whole-sequence CTA count sets the tile rotation of every query
  const int64_t rot_div = (int64_t)c.num_sms < s.S * n_hblk ? c.num_sms : s.S * n_hblk;
  int64_t grid = c.num_sms;
  if (grid > items) grid = items;
  if (items <= 0) return cudaSuccess;
  // sched[0]: work counter (a workspace header word)
  uint32_t* sched = c.status + 32;
  e = cudaMemsetAsync(sched, 0, 2 * sizeof(uint32_t), c.stream);
  if (e != cudaSuccess) return e;
  attn_fwd_tc_kernel<D, NH><<<(unsigned)grid, C::kThreads, smem, c.stream>>>(
      qm, k, v, idx, o, lse, s.t_lo, s.t_hi, (s.S - s.t_hi) * n_hblk, (int)rot_div, s.H,
      s.K_p, s.n_loc, s.scale * kLog2e, n_hblk,
      c.status, c.timeout_ns, sched);
  return cudaGetLastError();
}

}  // namespace

int attn_tc_heads(int H) {
  const int hb = H >= 64 ? 64 : H;
  return hb <= 16 ? 16 : (hb <= 32 ? 32 : 64);
}

cudaError_t launch_attn_fwd_tc(const LaunchCtx& c, const AttnShape& s,
                               const CUtensorMap& q_map, const __nv_bfloat16* k,
                               const __nv_bfloat16* v, const int32_t* idx,
                               __nv_bfloat16* o, float* lse) {
  const int nh = attn_tc_heads(s.H);
#define DSA_TCF(DD, NN) \
  if (s.D == DD && nh == NN) return launch_t<DD, NN>(c, s, q_map, k, v, idx, o, lse);
  DSA_TCF(128, 16) DSA_TCF(128, 32) DSA_TCF(128, 64)
  DSA_TCF(256, 16) DSA_TCF(256, 32) DSA_TCF(256, 64)
  DSA_TCF(512, 16) DSA_TCF(512, 32) DSA_TCF(512, 64)
#undef DSA_TCF
  return cudaErrorInvalidValue;
}

}  // namespace dsa
