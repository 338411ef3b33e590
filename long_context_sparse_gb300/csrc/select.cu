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
// result is bit-identical to a stable sort on (score desc, index asc).  A
// cut placed from evenly spaced samples first shrinks a long row to the few
// thousand candidates that can matter (checked, not assumed: a row where
// fewer than K_p keys pass the cut is selected in full).
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
constexpr int kBins = 2048;     // 11-bit digits: bits 31-21, 20-10, 9-0
constexpr int kSub = 256;                 // candidate slots of one warp
constexpr int kCand = kSub * kTopkWarps;  // candidate (key, pool) slots of a row
constexpr int kSamples = 1024;            // evenly spaced keys that place the cut

// Digit d of the highest bins that holds the kk-th largest key; *above =
// number of keys in higher bins, *count = keys in bin d.  Warp 0 only: lane
// l first sums the 64 bins kBins-64(l+1) .. kBins-64l-1 (lane 0: the top
// 64), starting at its own offset l so that the 32 lanes read 32 different
// banks; a warp scan finds the lane whose range holds the kk-th key, then
// the whole warp scans that range two bins per lane, highest first.
__device__ __forceinline__ void find_digit(const uint32_t* hist, uint32_t kk,
                                           uint32_t* sel_digit, uint32_t* sel_above,
                                           uint32_t* sel_count) {
  const int lane = threadIdx.x & 31;
  const int base = kBins - 64 * (lane + 1);
  uint32_t s = 0u;
#pragma unroll 16
  for (int j = 0; j < 64; ++j) s += hist[base + ((j + lane) & 63)];
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
      *sel_count = c0;
    } else {
      *sel_digit = (uint32_t)(top - 2 * lane - 1);
      *sel_above = before + c0;
      *sel_count = c1;
    }
  }
}

// Shared state of one top-k CTA (static shared memory, ~45 KB; two CTAs of
// 16 warps per SM, so the 256 rows of a score chunk run in one wave).
// Candidates live in one sub-buffer per warp; warp w's sub-buffer holds
// keys of a contiguous stretch of the row that precedes warp w+1's, so the
// sub-buffers read in warp order are in pool order.
struct TopkShared {
  uint32_t hist[kBins];
  uint32_t ckey[kCand];
  int32_t cidx[kCand];
  uint32_t samp[kSamples];
  uint32_t cnt[kTopkWarps];  // entries of each sub-buffer
  uint32_t wcnt[2][kTopkWarps];
  uint32_t sel_digit, sel_above, sel_count;
};

// The kk-th largest of a set of keys by radix select.  visit(f) calls
// f(key) for each key this thread owns (every key exactly once over the
// CTA).  The bits every key shares (the common prefix of the set's minimum
// and maximum) are known at once; the rest are resolved in digits of up to
// 11 bits from the top, so the first histogram spreads over many bins
// (a set of close keys would otherwise pile onto one) and a narrow set
// takes fewer passes.  *T = that key, *ties = how many keys equal to T rank
// among the kk largest (ties broken by position).
//
// When every key of the chosen bin ranks among the kk largest, no further
// digit is needed: the kk largest are exactly the keys >= the bin's lower
// edge, returned as *T = edge - 1 with *ties = 0.
//
// With max_passes = 1 the result is only a cut: *T is the lower edge of the
// first digit's bin that holds the kk-th largest key (at least kk keys are
// >= *T); *ties is then meaningless.
template <class Visit>
__device__ void radix_kth(Visit visit, uint32_t kk, TopkShared& sm, uint32_t* T,
                          uint32_t* ties, int max_passes = 3) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t lo = 0xffffffffu, hi = 0u;
  visit([&](uint32_t key) {
    lo = min(lo, key);
    hi = max(hi, key);
  });
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  if (lane == 0) {
    sm.wcnt[0][warp] = lo;
    sm.wcnt[1][warp] = hi;
  }
  __syncthreads();
  for (int w = 0; w < kTopkWarps; ++w) {
    lo = min(lo, sm.wcnt[0][w]);
    hi = max(hi, sm.wcnt[1][w]);
  }
  const int L = hi == lo ? 32 : __clz(hi ^ lo);  // bits shared by every key
  uint32_t pmask = L == 32 ? 0xffffffffu : ~(0xffffffffu >> L);
  uint32_t prefix = hi & pmask;
  int start = 32 - L;  // bits start-1 .. 0 are still open
  bool whole_bin = false;
#pragma unroll 1
  for (int pass = 0; start > 0 && pass < max_passes && !whole_bin; ++pass) {
    const int shift = start > 11 ? start - 11 : 0;
    const uint32_t dmask = (1u << (start - shift)) - 1u;
    for (int i = tid; i < kBins; i += kTopkThreads) sm.hist[i] = 0u;
    __syncthreads();
    visit([&](uint32_t key) {
      if ((key & pmask) == prefix) atomicAdd(&sm.hist[(key >> shift) & dmask], 1u);
    });
    __syncthreads();
    if (warp == 0) find_digit(sm.hist, kk, &sm.sel_digit, &sm.sel_above, &sm.sel_count);
    __syncthreads();
    prefix |= sm.sel_digit << shift;
    pmask |= dmask << shift;
    kk -= sm.sel_above;
    start = shift;
    // (sel_count is rewritten only by the next pass's find_digit, after two
    // more barriers: every thread reads the same value here)
    whole_bin = max_passes > 1 && start > 0 && kk == sm.sel_count && (prefix & pmask) != 0u;
  }
  __syncthreads();  // every thread has read the bounds and the digits
  prefix &= pmask;  // (a cut: the bits below the resolved digits are zero)
  *T = whole_bin ? prefix - 1u : prefix;
  *ties = whole_bin ? 0u : kk;
}

// Index-ordered selection: keys above T, then the first `ties` keys equal
// to T, each handed to emit(position, i) with its rank in order.  Warp w
// owns the keys key_at(i), i in [b0, b1), a stretch that precedes warp
// w+1's: one counting sweep, one exclusive sum over the warps, one emitting
// sweep with ballots.
template <class KeyAt, class Emit>
__device__ void ordered_take(KeyAt key_at, int64_t b0, int64_t b1, uint32_t T,
                             uint32_t ties, TopkShared& sm, Emit emit) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t cg = 0u, ct = 0u;
  for (int64_t i = b0 + lane; i < b1; i += 32) {
    const uint32_t key = key_at(i);
    cg += key > T;
    ct += key == T;
  }
  cg = __reduce_add_sync(0xffffffffu, cg);
  ct = __reduce_add_sync(0xffffffffu, ct);
  if (lane == 0) {
    sm.wcnt[0][warp] = cg;
    sm.wcnt[1][warp] = ct;
  }
  __syncthreads();
  uint32_t g = 0u, t = 0u;
  for (int w = 0; w < warp; ++w) {
    g += sm.wcnt[0][w];
    t += sm.wcnt[1][w];
  }
  for (int64_t i0 = b0; i0 < b1; i0 += 32) {
    const int64_t i = i0 + lane;
    const uint32_t key = i < b1 ? key_at(i) : 0u;
    const bool gt = i < b1 && key > T, eq = i < b1 && key == T;
    const uint32_t bg = __ballot_sync(0xffffffffu, gt), bt = __ballot_sync(0xffffffffu, eq);
    const uint32_t g_before = g + __popc(bg & lt), t_before = t + __popc(bt & lt);
    if (gt) emit(g_before + min(t_before, ties), i);
    else if (eq && t_before < ties) emit(g_before + t_before, i);
    g += __popc(bg);
    t += __popc(bt);
  }
  __syncthreads();  // wcnt is reused by the next call
}

// One CTA per query row (several resident per SM).  Exact whatever the
// data: a cut T0 taken from evenly spaced samples keeps every key >= T0 as
// a candidate, in pool order; when at least K_p keys pass and they fit,
// the K_p-th largest key of the row is the K_p-th largest candidate and
// the answer is read off the candidates.  Otherwise (a flat or skewed row)
// the row is selected directly from global memory.
__global__ void __launch_bounds__(kTopkThreads, 2)
    topk_rows_kernel(const float* __restrict__ scores, int64_t ld, int64_t row0,
                     int64_t rows, int K_p, int32_t* __restrict__ out, uint32_t* status) {
  __shared__ TopkShared sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* my_key = sm.ckey + warp * kSub;
  int32_t* my_idx = sm.cidx + warp * kSub;

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
    auto row_key = [&](int64_t i) { return order_key(__ldg(row + i)); };
    bool ok = true;
    int cb0, cb1;  // this warp's candidates: sm.ckey / sm.cidx [cb0, cb1)
    if (n <= kCand) {
      // ---- the whole row is the candidate set: warp w takes a stretch of
      // at most kSub keys
      const int64_t per = (n + kTopkWarps - 1) / kTopkWarps;
      const int64_t b0 = warp * per < n ? warp * per : n;
      const int64_t b1 = b0 + per < n ? b0 + per : n;
      for (int64_t i = b0 + lane; i < b1; i += 32) {
        my_key[i - b0] = row_key(i);
        my_idx[i - b0] = (int32_t)i;
      }
      cb0 = warp * kSub;
      cb1 = cb0 + (int)(b1 - b0);
    } else {
      // ---- the cut: the lower edge of the first-digit bin that holds the
      // rank-th largest of kSamples evenly spaced keys, rank chosen so that
      // about K_p (1 + 4/sqrt(a)) + 4 n/kSamples keys pass, a = K_p
      // kSamples / n being the expected samples above the answer
      {
        float x[kSamples / kTopkThreads];
#pragma unroll
        for (int u = 0; u < kSamples / kTopkThreads; ++u)
          x[u] = __ldg(row + (int64_t)(tid + u * kTopkThreads) * n / kSamples);
#pragma unroll
        for (int u = 0; u < kSamples / kTopkThreads; ++u)
          sm.samp[tid + u * kTopkThreads] = order_key(x[u]);
      }
      const float a = (float)K_p * (float)kSamples / (float)n;
      uint32_t rank = (uint32_t)ceilf(a + 4.f * sqrtf(a) + 4.f);
      if (rank > (uint32_t)kSamples) rank = kSamples;
      uint32_t T0, ties0;
      radix_kth(
          [&](auto f) {
            for (int j = tid; j < kSamples; j += kTopkThreads) f(sm.samp[j]);
          },
          rank, sm, &T0, &ties0, 1);
      // ---- one sweep: warp w appends the keys >= T0 of its stretch (whole
      // 512-key blocks, four float4 loads in flight per lane) to its own
      // sub-buffer, in order.  A stretch with more than kSub of them (a band
      // of high scores in one place) is swept again once every warp's count
      // is known, straight into its exact place in the flat array.
      constexpr int kU = 4;
      const bool vec = ((reinterpret_cast<uintptr_t>(row) & 15u) == 0);
      const int64_t nblk = (n + 128 * kU - 1) / (128 * kU);
      const int64_t bpw = (nblk + kTopkWarps - 1) / kTopkWarps;
      const int64_t b0 = warp * bpw * 128 * kU < n ? warp * bpw * 128 * kU : n;
      const int64_t b1 = b0 + bpw * 128 * kU < n ? b0 + bpw * 128 * kU : n;
      // keys i0 + 128u + 4 lane + e of a 512-key block (zero past b1)
      auto load_block = [&](int64_t i0, float4 (&f)[kU]) {
        if (vec && i0 + 128 * kU <= b1) {
#pragma unroll
          for (int u = 0; u < kU; ++u)
            f[u] = __ldg(reinterpret_cast<const float4*>(row + i0 + 128 * u + 4 * lane));
        } else {
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            const int64_t i = i0 + 128 * u + 4 * lane;
            f[u].x = i < b1 ? __ldg(row + i) : 0.f;
            f[u].y = i + 1 < b1 ? __ldg(row + i + 1) : 0.f;
            f[u].z = i + 2 < b1 ? __ldg(row + i + 2) : 0.f;
            f[u].w = i + 3 < b1 ? __ldg(row + i + 3) : 0.f;
          }
        }
      };
      const uint32_t lt = (1u << lane) - 1u;
      // sweep 0 writes the first kSub passing keys of the stretch to the
      // warp's sub-buffer; sweep 1 (only after a spill) all of them to their
      // exact place in the flat array
      uint32_t dbase = (uint32_t)(warp * kSub), cap = kSub;
#pragma unroll 1
      for (int sweep = 0; sweep < 2; ++sweep) {
      uint32_t c = 0u;
      for (int64_t i0 = b0; i0 < b1; i0 += 128 * kU) {
        float4 cur[kU];
        load_block(i0, cur);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int64_t i = i0 + 128 * u + 4 * lane;
          const uint32_t k0 = order_key(cur[u].x), k1 = order_key(cur[u].y),
                         k2 = order_key(cur[u].z), k3 = order_key(cur[u].w);
          const bool p0 = i < b1 && k0 >= T0, p1 = i + 1 < b1 && k1 >= T0,
                     p2 = i + 2 < b1 && k2 >= T0, p3 = i + 3 < b1 && k3 >= T0;
          const uint32_t q0 = __ballot_sync(0xffffffffu, p0), q1 = __ballot_sync(0xffffffffu, p1),
                         q2 = __ballot_sync(0xffffffffu, p2), q3 = __ballot_sync(0xffffffffu, p3);
          if ((q0 | q1 | q2 | q3) == 0u) continue;  // the usual case: nothing passes
          // keys of earlier lanes first, then this lane's in order
          uint32_t pos = c + __popc(q0 & lt) + __popc(q1 & lt) + __popc(q2 & lt) +
                         __popc(q3 & lt);
          const uint32_t kk4[4] = {k0, k1, k2, k3};
          const bool pp4[4] = {p0, p1, p2, p3};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (pp4[e]) {
              if (pos < cap && DSA_IN_BOUNDS(dbase + pos < (uint32_t)kCand, status)) {
                sm.ckey[dbase + pos] = kk4[e];
                sm.cidx[dbase + pos] = (int32_t)(i + e);
              }
              ++pos;
            }
          }
          c += __popc(q0) + __popc(q1) + __popc(q2) + __popc(q3);
        }
      }
      if (sweep == 1) break;  // (c and the layout were set by sweep 0)
      if (lane == 0) sm.cnt[warp] = c;
      __syncthreads();
      uint32_t total = 0u, before = 0u;
      bool spill = false;
      for (int w = 0; w < kTopkWarps; ++w) {
        before += w < warp ? sm.cnt[w] : 0u;
        total += sm.cnt[w];
        spill = spill || sm.cnt[w] > (uint32_t)kSub;
      }
      // too few keys pass (the cut was too high) or too many: the full row
      ok = total >= (uint32_t)K_p && total <= (uint32_t)kCand;
      if (ok && spill) {  // (CTA-uniform)
        dbase = before;
        cap = c;
        cb0 = (int)before;
        cb1 = (int)(before + c);
      } else {
        cb0 = warp * kSub;
        cb1 = cb0 + (int)c;
        break;
      }
      }
    }
    __syncthreads();
    // (positions are < K_p by construction; the guards keep a row that
    // changed under the kernel from writing into its neighbour)
    uint32_t T, ties;
    if (ok) {  // each warp takes its own candidates, which follow the previous warp's
      radix_kth(
          [&](auto f) {
            for (int j = cb0 + lane; j < cb1; j += 32) f(sm.ckey[j]);
          },
          (uint32_t)K_p, sm, &T, &ties);
      ordered_take([&](int64_t j) { return sm.ckey[j]; }, cb0, cb1, T, ties, sm,
                   [&](uint32_t pos, int64_t j) {
                     if (pos < (uint32_t)K_p) o[pos] = sm.cidx[j];
                   });
    } else {
      radix_kth(
          [&](auto f) {
            for (int64_t i = tid; i < n; i += kTopkThreads) f(row_key(i));
          },
          (uint32_t)K_p, sm, &T, &ties);
      const int64_t per = (n + kTopkWarps - 1) / kTopkWarps;
      const int64_t b0 = warp * per < n ? warp * per : n;
      const int64_t b1 = b0 + per < n ? b0 + per : n;
      ordered_take(row_key, b0, b1, T, ties, sm, [&](uint32_t pos, int64_t i) {
        if (pos < (uint32_t)K_p) o[pos] = (int32_t)i;
      });
    }
  }
}

cudaError_t launch_topk(const LaunchCtx& c, const float* scores, int64_t ld,
                        int64_t row0, int64_t rows, int K_p, int32_t* out) {
  if (rows <= 0) return cudaSuccess;
  int64_t grid = rows;
  const int64_t cap = (int64_t)c.num_sms * 2;
  if (grid > cap) grid = cap;
  topk_rows_kernel<<<(unsigned)grid, kTopkThreads, 0, c.stream>>>(scores, ld, row0, rows,
                                                                  K_p, out, c.status);
  return cudaGetLastError();
}

}  // namespace dsa
