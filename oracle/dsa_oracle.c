/*
 * dsa_oracle.c -- plain, slow, single-threaded CPU oracle for the
 * DeepSeek-Sparse-Attention (DSA) hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path links, loads or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header or table with the CUDA
 * library.
 *
 * Sources followed (web pages, cited by title and section):
 *   [SkyRL]     "Scaling Training to 1M Token Context on GLM-5.3-Flash"
 *               - section "DeepSeek Sparse Attention (DSA) Optimizations":
 *                 a lightweight indexer scores every query against every
 *                 earlier pool of 4 tokens; attention then reads only the
 *                 2048 selected tokens.
 *               - section "Making Sparse Attention Actually Sparse": NoPE
 *                 q/k (no rotary channels) and the 2,051-key selection.
 *               - section "Splitting the DSA Indexer / Over Time: Chunking":
 *                 scoring and selection a few hundred queries at a time.
 *               - section "Across GPUs: Sharding": selected pool indices are
 *                 int32.
 *   [MTraining] "MTraining: Efficient Distributed Training for Ultra-Long
 *               Contexts via Dynamic Sparse Attention", section 3.2 (Eq. 1):
 *               every backward GEMM depends on the attention weights A.
 *
 * Indexer score (the DSA "lightning indexer"): for query t and pool p
 *     I[t,p] = sum_h w[t,h] * max(0, sum_d q_idx[t,h,d] * k_pool[p,d])
 * defined for complete earlier pools only, p < n_full(t) = floor((t+1)/4).
 *
 * Everything is fp64 except the key pooling, which follows the pooling
 * rounding rule fixed by the library contract (fp32 pairwise sum, times 0.25,
 * round to bf16 nearest-even) so both sides feed identical pooled keys into
 * the score contraction.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared -o liboracle.so
 *        dsa_oracle.c -lm
 * (-ffp-contract=off: the fp32 pooling must not be fused into FMAs.)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
float oracle_bf16_to_f32(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static double bf(uint16_t h) { return (double)oracle_bf16_to_f32(h); }

/* binary32 -> bf16, round to nearest, ties to even; NaN stays a quiet NaN. */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
    return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lower = u & 0xffffu;
  uint32_t upper = u >> 16;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return (uint16_t)upper;
}

/* ------------------------------------------------------------ pool (a1) */

/* Number of complete 4-token pools at or before query t: only these are
 * "earlier pools" ([SkyRL] "DeepSeek Sparse Attention (DSA) Optimizations");
 * a partial pool would mix in tokens after t. */
int64_t oracle_n_full(int64_t t) { return (t + 1) / 4; }

/* k_pool[p] = mean of indexer keys 4p..4p+3.  Rounding rule: fp32
 * ((k0 + k1) + (k2 + k3)) * 0.25, then bf16 nearest-even.  Pools do not
 * overlap and start at multiples of 4; the trailing S mod 4 tokens form no
 * pool. */
void oracle_pool(int64_t S, int32_t D_I, const uint16_t* k_idx,
                 uint16_t* k_pool) {
  int64_t P = S / 4;
  for (int64_t p = 0; p < P; ++p) {
    for (int32_t d = 0; d < D_I; ++d) {
      float k0 = oracle_bf16_to_f32(k_idx[(4 * p + 0) * D_I + d]);
      float k1 = oracle_bf16_to_f32(k_idx[(4 * p + 1) * D_I + d]);
      float k2 = oracle_bf16_to_f32(k_idx[(4 * p + 2) * D_I + d]);
      float k3 = oracle_bf16_to_f32(k_idx[(4 * p + 3) * D_I + d]);
      volatile float a = k0 + k1;
      volatile float b = k2 + k3;
      volatile float s = a + b;
      float m = s * 0.25f;
      k_pool[p * D_I + d] = oracle_f32_to_bf16(m);
    }
  }
}

/* Gated pooling ("Scaling Training to 1M Token Context on GLM-5.3-Flash",
 * section "DSA: Gather by Token Position": k-pool gate scores weight each
 * key within its pool), read as a softmax of the 4 gate scores:
 *   k_pool[p] = sum_j w_j k[4p+j],  w_j = exp(g_j) / sum_i exp(g_i)
 * computed in fp64 (exp of g_j - max g for range), then rounded to fp32
 * and to bf16 nearest-even.  Equal gates give the mean. */
void oracle_pool_gated(int64_t S, int32_t D_I, const uint16_t* k_idx,
                       const float* gate, uint16_t* k_pool) {
  int64_t P = S / 4;
  for (int64_t p = 0; p < P; ++p) {
    double g[4], m = -HUGE_VAL, e[4], den = 0.0;
    for (int j = 0; j < 4; ++j) {
      g[j] = (double)gate[4 * p + j];
      if (g[j] > m) m = g[j];
    }
    for (int j = 0; j < 4; ++j) {
      e[j] = exp(g[j] - m);
      den += e[j];
    }
    for (int32_t d = 0; d < D_I; ++d) {
      double acc = 0.0;
      for (int j = 0; j < 4; ++j) acc += (e[j] / den) * bf(k_idx[(4 * p + j) * D_I + d]);
      k_pool[p * D_I + d] = oracle_f32_to_bf16((float)acc);
    }
  }
}

/* ------------------------------------------------------- indexer (a2,a3) */

/* Scores of the listed query rows against every pool, fp64.
 *   q_idx  [nrows, H_I, D_I] bf16 and w [nrows, H_I] fp32 hold the listed
 *          rows (row r is query t = rows[r]); k_pool [P, D_I] bf16
 *   out    [nrows, P]: I[t,p] for p < n_full(t), -inf for later pools
 *          (those are never candidates). */
void oracle_index_scores(int64_t S, int32_t H_I, int32_t D_I,
                         const uint16_t* q_idx, const uint16_t* k_pool,
                         const float* w, int64_t nrows, const int64_t* rows,
                         double* out) {
  int64_t P = S / 4;
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t t = rows[r];
    int64_t nf = oracle_n_full(t);
    double* o = out + r * P;
    for (int64_t p = 0; p < P; ++p) {
      if (p >= nf) {
        o[p] = -INFINITY;
        continue;
      }
      double acc = 0.0;
      for (int32_t h = 0; h < H_I; ++h) {
        const uint16_t* qv = q_idx + (r * H_I + h) * D_I;
        const uint16_t* kv = k_pool + p * D_I;
        double dot = 0.0;
        for (int32_t d = 0; d < D_I; ++d) dot += bf(qv[d]) * bf(kv[d]);
        double relu = dot > 0.0 ? dot : 0.0;
        acc += (double)w[r * H_I + h] * relu;
      }
      o[p] = acc;
    }
  }
}

/* ------------------------------------------------------------ top-k (a4) */

typedef struct {
  double s;
  int64_t p;
} cand_t;

/* Order: higher score first; equal scores -> lower pool index first.
 * -0.0 and +0.0 compare equal here, as IEEE comparison says. */
static int cand_cmp(const void* a, const void* b) {
  const cand_t* x = (const cand_t*)a;
  const cand_t* y = (const cand_t*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->p < y->p) ? -1 : (x->p > y->p ? 1 : 0);
}

static int idx_cmp(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

/* One row: the min(K_p, n_valid) best of scores[0..n_valid) by the order
 * above, written in ascending pool index, the rest of the K_p slots -1. */
static void topk_row(const double* scores, int64_t n_valid, int32_t K_p,
                     int32_t* out, cand_t* buf) {
  for (int64_t p = 0; p < n_valid; ++p) {
    buf[p].s = scores[p];
    buf[p].p = p;
  }
  qsort(buf, (size_t)n_valid, sizeof(cand_t), cand_cmp);
  int64_t take = n_valid < K_p ? n_valid : K_p;
  for (int64_t i = 0; i < take; ++i) out[i] = (int32_t)buf[i].p;
  qsort(out, (size_t)take, sizeof(int32_t), idx_cmp);
  for (int64_t i = take; i < K_p; ++i) out[i] = -1;
}

/* Top-k over fp64 score rows (the oracle's own indexer output).
 *   scores [nrows, ld]; row r is query rows[r]; n_full(rows[r]) entries valid
 *   out    [nrows, K_p] int32 */
int oracle_topk_f64(int64_t nrows, int64_t ld, const double* scores,
                    const int64_t* rows, int32_t K_p, int32_t* out) {
  int64_t maxn = 0;
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t nf = oracle_n_full(rows[r]);
    if (nf > maxn) maxn = nf;
  }
  cand_t* buf = (cand_t*)malloc((size_t)(maxn > 0 ? maxn : 1) * sizeof(cand_t));
  if (!buf) return -1;
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t nf = oracle_n_full(rows[r]);
    if (nf > ld) nf = ld;
    topk_row(scores + r * ld, nf, K_p, out + r * K_p, buf);
  }
  free(buf);
  return 0;
}

/* Same selection over an fp32 score array (the bit-exact top-k check: both
 * sides read the same fp32 values; widening to fp64 keeps order and ties). */
int oracle_topk_f32(int64_t nrows, int64_t ld, const float* scores,
                    const int64_t* rows, int32_t K_p, int32_t* out) {
  double* row = (double*)malloc((size_t)(ld > 0 ? ld : 1) * sizeof(double));
  cand_t* buf = (cand_t*)malloc((size_t)(ld > 0 ? ld : 1) * sizeof(cand_t));
  if (!row || !buf) {
    free(row);
    free(buf);
    return -1;
  }
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t nf = oracle_n_full(rows[r]);
    if (nf > ld) nf = ld;
    for (int64_t p = 0; p < nf; ++p) row[p] = (double)scores[r * ld + p];
    topk_row(row, nf, K_p, out + r * K_p, buf);
  }
  free(row);
  free(buf);
  return 0;
}

/* ----------------------------------------------------- key set (a5) */

/* Token set K(t) attended by query t: tokens 4p..4p+3 of every selected pool
 * p (idx_row holds K_p entries, -1 = empty slot), plus, when n_loc == 3, the
 * query's own most recent tokens {t-2, t-1, t} clipped to [0, t] ([SkyRL]
 * "Making Sparse Attention Actually Sparse": 2,051 = 2,048 pooled keys + 3).
 * A token is counted once.  Returned ascending; result count is returned.
 * keys must hold 4*K_p + n_loc entries. */
int64_t oracle_key_set(int64_t t, int32_t K_p, int32_t n_loc,
                       const int32_t* idx_row, int64_t* keys) {
  int64_t n = 0;
  for (int32_t i = 0; i < K_p; ++i) {
    int32_t p = idx_row[i];
    if (p < 0) continue;
    for (int j = 0; j < 4; ++j) keys[n++] = 4 * (int64_t)p + j;
  }
  for (int32_t j = n_loc - 1; j >= 0; --j) {
    int64_t s = t - j;
    if (s < 0) continue;
    int dup = 0;
    for (int64_t i = 0; i < n; ++i)
      if (keys[i] == s) {
        dup = 1;
        break;
      }
    if (!dup) keys[n++] = s;
  }
  /* insertion sort: small and obviously correct */
  for (int64_t i = 1; i < n; ++i) {
    int64_t v = keys[i], j = i - 1;
    while (j >= 0 && keys[j] > v) {
      keys[j + 1] = keys[j];
      --j;
    }
    keys[j + 1] = v;
  }
  return n;
}

/* ------------------------------------------------- attention fwd (a6) */

/* For each listed query row t and head h:
 *   s_j   = scale * q[t,h] . k_j            for j in K(t)
 *   O     = sum_j softmax_j(s) v_j,  LSE = log sum_j exp(s_j)
 * An empty key set gives O = 0 and LSE = -inf.
 * q [nrows,H,d_qk] bf16 holds the listed rows (row r is query t = rows[r]);
 * k [S,d_qk], v [S,d_v] bf16 (one K and one V shared by all heads);
 * topk_idx [S,K_p] int32; o [nrows,H,d_v], lse [nrows,H] fp64. */
int oracle_attn_fwd(int64_t S, int32_t H, int32_t d_qk, int32_t d_v,
                    int32_t K_p, int32_t n_loc, double scale,
                    const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    const int32_t* topk_idx, int64_t nrows,
                    const int64_t* rows, double* o, double* lse) {
  (void)S;
  int64_t cap = 4 * (int64_t)K_p + n_loc + 1;
  int64_t* keys = (int64_t*)malloc((size_t)cap * sizeof(int64_t));
  double* s = (double*)malloc((size_t)cap * sizeof(double));
  if (!keys || !s) {
    free(keys);
    free(s);
    return -1;
  }
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t t = rows[r];
    int64_t n = oracle_key_set(t, K_p, n_loc, topk_idx + t * K_p, keys);
    for (int32_t h = 0; h < H; ++h) {
      double* orow = o + (r * H + h) * d_v;
      for (int32_t e = 0; e < d_v; ++e) orow[e] = 0.0;
      if (n == 0) {
        lse[r * H + h] = -INFINITY;
        continue;
      }
      const uint16_t* qv = q + (r * H + h) * (int64_t)d_qk;
      double mx = -INFINITY;
      for (int64_t i = 0; i < n; ++i) {
        const uint16_t* kv = k + keys[i] * d_qk;
        double dot = 0.0;
        for (int32_t d = 0; d < d_qk; ++d) dot += bf(qv[d]) * bf(kv[d]);
        s[i] = scale * dot;
        if (s[i] > mx) mx = s[i];
      }
      double sum = 0.0;
      for (int64_t i = 0; i < n; ++i) sum += exp(s[i] - mx);
      for (int64_t i = 0; i < n; ++i) {
        double pw = exp(s[i] - mx) / sum;
        const uint16_t* vv = v + keys[i] * d_v;
        for (int32_t e = 0; e < d_v; ++e) orow[e] += pw * bf(vv[e]);
      }
      lse[r * H + h] = mx + log(sum);
    }
  }
  free(keys);
  free(s);
  return 0;
}

/* ------------------------------------------------ attention bwd (a7,a8) */

/* Analytic gradients of L = sum_{t in rows} sum_h <dO[t,h], O[t,h]>, i.e.
 * the backward with upstream gradient dO on the listed rows and zero on all
 * others.  Per row t and head h (P recomputed here in fp64):
 *   P_j   = exp(s_j - LSE)
 *   dP_j  = dO . v_j
 *   delta = sum_j P_j dP_j            (= dO . O)
 *   dS_j  = P_j (dP_j - delta)
 *   dQ   += scale * sum_j dS_j k_j
 *   dK_j += scale * dS_j q[t,h]
 *   dV_j += P_j dO
 * ([MTraining] section 3.2: every backward GEMM depends on A = P.)
 * q [nrows,H,d_qk] and dO [nrows,H,d_v] bf16 hold the listed rows;
 * dq [nrows,H,d_qk].  dk [n_slots,d_qk] and
 * dv [n_slots,d_v] are overwritten with the contributions of the listed rows:
 * token j lands in row key_slot[j] (skipped when -1), or in row j when
 * key_slot is NULL (then n_slots = S).  Only the addressing differs. */
int oracle_attn_bwd(int64_t S, int32_t H, int32_t d_qk, int32_t d_v,
                    int32_t K_p, int32_t n_loc, double scale,
                    const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    const uint16_t* dO, const int32_t* topk_idx,
                    int64_t nrows, const int64_t* rows, const int64_t* key_slot,
                    int64_t n_slots, double* dq, double* dk, double* dv) {
  int64_t cap = 4 * (int64_t)K_p + n_loc + 1;
  int64_t* keys = (int64_t*)malloc((size_t)cap * sizeof(int64_t));
  double* s = (double*)malloc((size_t)cap * sizeof(double));
  double* dp = (double*)malloc((size_t)cap * sizeof(double));
  if (!keys || !s || !dp) {
    free(keys);
    free(s);
    free(dp);
    return -1;
  }
  if (!key_slot) n_slots = S;
  memset(dk, 0, (size_t)n_slots * d_qk * sizeof(double));
  memset(dv, 0, (size_t)n_slots * d_v * sizeof(double));
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t t = rows[r];
    int64_t n = oracle_key_set(t, K_p, n_loc, topk_idx + t * K_p, keys);
    for (int32_t h = 0; h < H; ++h) {
      double* dqrow = dq + (r * H + h) * (int64_t)d_qk;
      for (int32_t d = 0; d < d_qk; ++d) dqrow[d] = 0.0;
      if (n == 0) continue;
      const uint16_t* qv = q + (r * H + h) * (int64_t)d_qk;
      const uint16_t* gv = dO + (r * H + h) * (int64_t)d_v;
      double mx = -INFINITY;
      for (int64_t i = 0; i < n; ++i) {
        const uint16_t* kv = k + keys[i] * d_qk;
        double dot = 0.0;
        for (int32_t d = 0; d < d_qk; ++d) dot += bf(qv[d]) * bf(kv[d]);
        s[i] = scale * dot;
        if (s[i] > mx) mx = s[i];
      }
      double sum = 0.0;
      for (int64_t i = 0; i < n; ++i) sum += exp(s[i] - mx);
      double lse = mx + log(sum);
      double delta = 0.0;
      for (int64_t i = 0; i < n; ++i) {
        const uint16_t* vv = v + keys[i] * d_v;
        double g = 0.0;
        for (int32_t e = 0; e < d_v; ++e) g += bf(gv[e]) * bf(vv[e]);
        dp[i] = g;
        delta += exp(s[i] - lse) * g;
      }
      for (int64_t i = 0; i < n; ++i) {
        double pw = exp(s[i] - lse);
        double ds = pw * (dp[i] - delta);
        const uint16_t* kv = k + keys[i] * d_qk;
        int64_t slot = key_slot ? key_slot[keys[i]] : keys[i];
        for (int32_t d = 0; d < d_qk; ++d) dqrow[d] += scale * ds * bf(kv[d]);
        if (slot < 0) continue;
        double* dkrow = dk + slot * d_qk;
        double* dvrow = dv + slot * d_v;
        for (int32_t d = 0; d < d_qk; ++d) dkrow[d] += scale * ds * bf(qv[d]);
        for (int32_t e = 0; e < d_v; ++e) dvrow[e] += pw * bf(gv[e]);
      }
    }
  }
  free(keys);
  free(s);
  free(dp);
  return 0;
}

/* ---------------------------------------- dense masked attention (check) */

/* Textbook dense attention under an explicit S x S 0/1 mask (mask[t*S+j]
 * = 1 when query t may attend to token j).  A separate code path from the
 * key-set route above; used to cross-check it.  Rows with no allowed key
 * give O = 0, LSE = -inf. */
void oracle_dense_masked_attn(int64_t S, int32_t H, int32_t d_qk, int32_t d_v,
                              double scale, const uint16_t* q,
                              const uint16_t* k, const uint16_t* v,
                              const uint8_t* mask, double* o, double* lse) {
  for (int64_t t = 0; t < S; ++t)
    for (int32_t h = 0; h < H; ++h) {
      const uint16_t* qv = q + (t * H + h) * (int64_t)d_qk;
      double* orow = o + (t * H + h) * (int64_t)d_v;
      double mx = -INFINITY;
      for (int64_t j = 0; j < S; ++j) {
        if (!mask[t * S + j]) continue;
        double dot = 0.0;
        for (int32_t d = 0; d < d_qk; ++d) dot += bf(qv[d]) * bf(k[j * d_qk + d]);
        if (scale * dot > mx) mx = scale * dot;
      }
      for (int32_t e = 0; e < d_v; ++e) orow[e] = 0.0;
      if (mx == -INFINITY) {
        lse[t * H + h] = -INFINITY;
        continue;
      }
      double sum = 0.0;
      for (int64_t j = 0; j < S; ++j) {
        if (!mask[t * S + j]) continue;
        double dot = 0.0;
        for (int32_t d = 0; d < d_qk; ++d) dot += bf(qv[d]) * bf(k[j * d_qk + d]);
        double e = exp(scale * dot - mx);
        sum += e;
        for (int32_t c = 0; c < d_v; ++c) orow[c] += e * bf(v[j * d_v + c]);
      }
      for (int32_t c = 0; c < d_v; ++c) orow[c] /= sum;
      lse[t * H + h] = mx + log(sum);
    }
}
