/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DeepSeek-Sparse-Attention hot path.
 *
 * The method is the DSA layer of "Scaling Training to 1M Token Context on
 * GLM-5.3-Flash" (sections "DeepSeek Sparse Attention (DSA) Optimizations",
 * "Making Sparse Attention Actually Sparse", "Splitting the DSA Indexer"):
 *
 *   1. pool     k_pool[p] = mean of indexer keys 4p..4p+3 (pools of 4 tokens)
 *   2. score    I[t,p] = sum_h w[t,h] * max(0, q_idx[t,h,:] . k_pool[p,:])
 *               for every complete earlier pool p < n_full(t) = (t+1)/4
 *   3. chunk    queries are scored a few hundred at a time ("Over Time:
 *               Chunking") so the S x S/4 score matrix never exists at once
 *   4. select   the K_p best pools per query, ties to the lower pool index,
 *               emitted as int32 ("Across GPUs: Sharding": int32 indices)
 *   5. attend   softmax attention of each query head over the tokens of the
 *               selected pools (4*K_p = 2048 keys), plus, when n_local = 3,
 *               the query's own 3 most recent tokens (2,051 keys), with one
 *               NoPE K and one V shared by all heads
 *   6. backward recompute P, scatter dK/dV ("MTraining: Efficient
 *               Distributed Training for Ultra-Long Contexts via Dynamic
 *               Sparse Attention", section 3.2: every backward GEMM depends
 *               on the attention weights)
 *
 * Conventions for every entry point:
 *  - Ownership: the caller owns every buffer, the workspace included.  The
 *    library allocates no device or host memory and keeps no state between
 *    calls (a per-process cache of device attributes aside).
 *  - Pointers: device pointers unless stated.  Dense, row-major, contiguous.
 *    Every tensor pointer must be 16-byte aligned, else DSA_ERR_MISALIGNED.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy
 *    default stream).  Calls are asynchronous on that stream; argument
 *    errors are returned before anything is launched; launch failures return
 *    DSA_ERR_CUDA.  Errors found by a kernel (a bounded wait that ran out, an
 *    out-of-range index) are latched in the workspace status word and read
 *    back with dsa_get_device_status().
 *  - No fallback: a shape the kernels do not support returns
 *    DSA_ERR_UNSUPPORTED_SHAPE.  There is no dense or CPU path.
 *  - bf16 = IEEE bfloat16; fp32 = IEEE binary32.
 */
#ifndef DSA_GB300_H
#define DSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_ABI_VERSION 1

#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

typedef enum dsa_status {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad value */
  DSA_ERR_UNSUPPORTED_SHAPE = 2, /* valid, but not a shape the kernels run */
  DSA_ERR_WORKSPACE_TOO_SMALL = 3,
  DSA_ERR_MISALIGNED = 4,        /* a pointer is not 16-byte aligned */
  DSA_ERR_CUDA = 5,              /* a CUDA runtime/driver call failed */
  DSA_ERR_DEVICE_TIMEOUT = 6,    /* a kernel's bounded wait ran out */
  DSA_ERR_DEVICE_BAD_INDEX = 7,  /* a kernel read an out-of-range pool index */
  DSA_ERR_SCRATCH_CAP = 8,       /* one score chunk would exceed scratch_cap */
  DSA_ERR_DEVICE_CHECK = 9       /* debug build (DSA_CHECKS) only: a kernel computed an
                                    out-of-range shared-memory, TMEM or global offset; the
                                    access was skipped */
} dsa_status_t;

/* Problem description (one sequence per call; batch = 1).
 * Layout is fixed for foreign callers: 56 bytes, natural alignment. */
typedef struct dsa_config {
  int64_t seq_len;     /* S >= 1 */
  int32_t pool_size;   /* tokens per pool; must be 4 */
  int32_t topk_pools;  /* K_p, selected pools per query: 1..2048 */
  int32_t n_local;     /* 0 (4*K_p keys) or 3 (4*K_p + 3 keys) */
  int32_t idx_heads;   /* H_I in {1,2,4,8,16,32,64} */
  int32_t idx_dim;     /* D_I in {64,128} */
  int32_t attn_heads;  /* H, 1..128 */
  int32_t d_qk;        /* NoPE q/k dim in {128,256,512} */
  int32_t d_v;         /* must equal d_qk */
  int32_t chunk_q;     /* C, queries scored per indexer chunk, >= 1 */
  float sm_scale;      /* softmax scale; 0 -> 1/sqrt(d_qk) */
  uint64_t scratch_cap;/* max bytes of one [C, ld] fp32 score chunk */
} dsa_config_t;

/* Workspace kinds for dsa_workspace_size(). */
#define DSA_WS_INDEX 0 /* dsa_index_scores_topk */
#define DSA_WS_FWD 1   /* dsa_sparse_attn_fwd */
#define DSA_WS_BWD 2   /* dsa_sparse_attn_bwd */
#define DSA_WS_STATUS 3 /* dsa_index_scores, dsa_topk_from_scores */
#define DSA_WS_STREAM 4 /* dsa_index_topk_streaming */
#define DSA_WS_BWD_ROWS 5 /* dsa_sparse_attn_bwd_range */
#define DSA_WS_STEP 6   /* dsa_step, dsa_step_host */

/* Bytes of device workspace the call `which` needs for `cfg`.  Every
 * workspace begins with a 256-byte header holding the device status word;
 * zero it once with dsa_workspace_init() before first use. */
DSA_API dsa_status_t dsa_workspace_size(const dsa_config_t* cfg, int32_t which,
                                size_t* bytes);

/* Zero the workspace header (status word) on `stream`. */
DSA_API dsa_status_t dsa_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Step 1 alone.  k_idx [S, D_I] bf16 -> k_pool [S/4, D_I] bf16.
 * k_pool[p,d] = bf16_rne(((k[4p,d] + k[4p+1,d]) + (k[4p+2,d] + k[4p+3,d]))
 *               * 0.25) in fp32.  The S mod 4 trailing tokens form no pool. */
DSA_API dsa_status_t dsa_pool_keys(const dsa_config_t* cfg, const void* k_idx,
                           void* k_pool, void* stream);

/* Step 1 with gated pools ("Scaling Training to 1M Token Context on
 * GLM-5.3-Flash", section "DSA: Gather by Token Position": k-pool gate
 * scores weight each key within its pool), read as a softmax over the
 * pool's four gate scores, in fp32:
 *   w_j = exp(g_j - m) / ((e_0 + e_1) + (e_2 + e_3)),  m = max_j g_j,
 *   k_pool[p,d] = bf16_rne((w_0 k[4p,d] + w_1 k[4p+1,d])
 *                          + (w_2 k[4p+2,d] + w_3 k[4p+3,d])).
 * k_gate [S] fp32 (finite), 16-byte aligned.  Equal gates give the mean
 * pooling of dsa_pool_keys.  Forward only: the pages do not say how the
 * gates are trained. */
DSA_API dsa_status_t dsa_pool_keys_gated(const dsa_config_t* cfg, const void* k_idx,
                                 const float* k_gate, void* k_pool,
                                 void* stream);

/* Step 2 for one block of queries t0 .. t0+rows-1 (rows <= 4096):
 *   scores[r*ld + p] = I[t0 + r, p]  (fp32, tensor-core bf16 products,
 *   fp32 accumulation) for p < n_full(t0 + r).  Entries with p >= n_full(t)
 *   and p < ld may be overwritten with unspecified values.
 * q_idx [S, H_I, D_I] bf16; k_pool [S/4, D_I] bf16; w [S, H_I] fp32;
 * ld >= n_full(t0+rows-1), ld % 4 == 0.  ws: DSA_WS_STATUS. */
DSA_API dsa_status_t dsa_index_scores(const dsa_config_t* cfg, const void* q_idx,
                              const void* k_pool, const float* w, int64_t t0,
                              int64_t rows, float* scores, int64_t ld,
                              void* ws, size_t ws_bytes, void* stream);

/* Step 4 alone (the bit-exact selection check).  Row r of scores [rows, ld]
 * fp32 belongs to query t = row0 + r; its candidates are entries
 * 0 .. n_full(t)-1.  topk_idx[r*K_p ..] receives the min(K_p, n_full(t))
 * best pools (larger score first, equal scores -> lower pool index; -0.0 ==
 * +0.0) in ascending pool order, then -1.  Scores must not be NaN.
 * ws: DSA_WS_STATUS. */
DSA_API dsa_status_t dsa_topk_from_scores(const dsa_config_t* cfg,
                                  const float* scores, int64_t ld,
                                  int64_t row0, int64_t rows,
                                  int32_t* topk_idx, void* ws,
                                  size_t ws_bytes, void* stream);

/* Steps 1-4: pool, then per chunk of C queries score and select.
 * q_idx [S, H_I, D_I] bf16, k_idx [S, D_I] bf16, w [S, H_I] fp32 ->
 * topk_idx [S, K_p] int32 (as dsa_topk_from_scores).  The workspace holds
 * the pooled keys and one [C, ld] fp32 score chunk (ld = S/4 rounded up to
 * 128); C * ld * 4 > scratch_cap returns DSA_ERR_SCRATCH_CAP.
 * ws: DSA_WS_INDEX. */
DSA_API dsa_status_t dsa_index_scores_topk(const dsa_config_t* cfg,
                                   const void* q_idx, const void* k_idx,
                                   const float* w, int32_t* topk_idx,
                                   void* ws, size_t ws_bytes, void* stream);

/* Steps 1-4 for the query rows t_begin .. t_end-1 only, with mean pooling
 * (k_gate NULL) or gated pooling (k_gate [S] fp32, as dsa_pool_keys_gated):
 * the share of one
 * rank when the indexer is split by query, each rank scoring its queries
 * against all earlier pools and the int32 selections being gathered
 * afterwards ("Scaling Training to 1M Token Context on GLM-5.3-Flash",
 * section "Across GPUs: Sharding").  The selection of every row is exactly
 * the one dsa_index_scores_topk gives that row.
 * q_idx [t_end-t_begin, H_I, D_I] bf16 and w [t_end-t_begin, H_I] fp32 hold
 * the range's rows (row r <-> query t_begin + r); k_idx [S, D_I] bf16 holds
 * every key -> topk_idx [t_end-t_begin, K_p] int32.  0 <= t_begin <= t_end
 * <= S, else DSA_ERR_INVALID_ARG; an empty range does nothing.
 * ws: DSA_WS_INDEX (pooled keys of all S tokens plus one score chunk). */
DSA_API dsa_status_t dsa_index_scores_topk_range(
    const dsa_config_t* cfg, const void* q_idx, const void* k_idx, const float* k_gate,
    const float* w, int64_t t_begin, int64_t t_end, int32_t* topk_idx, void* ws,
    size_t ws_bytes, void* stream);

/* Steps 1-4 with the selection fused into the indexer: no score is ever
 * stored (the chunking of "Scaling Training to 1M Token Context on
 * GLM-5.3-Flash", section "Splitting the DSA Indexer / Over Time: Chunking",
 * taken to the end: each query's running selection lives in on-chip
 * memory while the pools stream past).  Same arguments and result, row for
 * row bit-identical, as dsa_index_scores_topk_range; the workspace holds
 * only the pooled keys (DSA_WS_STREAM), so there is no scratch cap.
 * Supported: H_I in {32, 64}, D_I in {64, 128}, K_p <= 768; otherwise
 * DSA_ERR_UNSUPPORTED_SHAPE (use dsa_index_scores_topk_range). */
DSA_API dsa_status_t dsa_index_topk_streaming(
    const dsa_config_t* cfg, const void* q_idx, const void* k_idx, const float* k_gate,
    const float* w, int64_t t_begin, int64_t t_end, int32_t* topk_idx, void* ws,
    size_t ws_bytes, void* stream);

/* Step 5, forward.  For every query t and head h, over the key set K(t):
 *   O[t,h]   = sum_j softmax_j(scale * q[t,h] . k_j) v_j
 *   LSE[t,h] = log sum_j exp(scale * q[t,h] . k_j)      (natural log)
 * K(t) = tokens 4p..4p+3 of every selected pool (topk_idx[t,:] >= 0, each
 * must be < n_full(t), else DSA_ERR_DEVICE_BAD_INDEX is latched and the row
 * skips that pool), plus {t-2, t-1, t} clipped to >= 0 when n_local = 3, each
 * token counted once.  An empty K(t) gives O = 0 and LSE = -inf.
 * q [S, H, d_qk], k [S, d_qk], v [S, d_v] bf16; topk_idx [S, K_p] int32 ->
 * o [S, H, d_v] bf16, lse [S, H] fp32.  ws: DSA_WS_FWD. */
DSA_API dsa_status_t dsa_sparse_attn_fwd(const dsa_config_t* cfg, const void* q,
                                 const void* k, const void* v,
                                 const int32_t* topk_idx, void* o, float* lse,
                                 void* ws, size_t ws_bytes, void* stream);

/* Step 6, backward of step 5 for upstream gradient dO [S, H, d_v] bf16, with
 * o and lse from dsa_sparse_attn_fwd on the same inputs:
 *   P = exp(scale q.k_j - LSE), dP = dO . v_j, delta = dO . O,
 *   dS = P (dP - delta), dq = scale sum_j dS k_j,
 *   dk_j = scale sum_{t,h} dS q[t,h], dv_j = sum_{t,h} P dO[t,h].
 * dk/dv are accumulated in fp32 in the workspace and written once as bf16.
 * dq [S, H, d_qk], dk [S, d_qk], dv [S, d_v] bf16 are overwritten.
 * ws: DSA_WS_BWD. */
DSA_API dsa_status_t dsa_sparse_attn_bwd(const dsa_config_t* cfg, const void* q,
                                 const void* k, const void* v, const void* o,
                                 const float* lse, const void* dO,
                                 const int32_t* topk_idx, void* dq, void* dk,
                                 void* dv, void* ws, size_t ws_bytes,
                                 void* stream);

/* Steps 5 and 6 with K = V: one tensor kv [S, d] (d = d_qk = d_v) serves as
 * both keys and values, as the shared latent of multi-head latent attention
 * does ("shared NoPE K/V" read as one tensor; the backward gathers each key
 * row once for both products and sums dK and dV per row before a single
 * scatter).  Results are those of dsa_sparse_attn_fwd / _bwd with k = v = kv,
 * except that dkv [S, d] bf16 = dK + dV (one fp32 accumulator).
 * ws: DSA_WS_FWD / DSA_WS_BWD. */
DSA_API dsa_status_t dsa_sparse_attn_fwd_kv(const dsa_config_t* cfg, const void* q,
                                    const void* kv, const int32_t* topk_idx, void* o,
                                    float* lse, void* ws, size_t ws_bytes,
                                    void* stream);
DSA_API dsa_status_t dsa_sparse_attn_bwd_kv(const dsa_config_t* cfg, const void* q,
                                    const void* kv, const void* o, const float* lse,
                                    const void* dO, const int32_t* topk_idx, void* dq,
                                    void* dkv, void* ws, size_t ws_bytes,
                                    void* stream);

/* Step 5 for the queries [t_begin, t_end) only: the form a rank takes when
 * attention is split by query across GPUs ("Scaling Training to 1M Token
 * Context on GLM-5.3-Flash", section "Across GPUs: Sharding"), and the unit
 * dsa_step_host pipelines.  q [n, H, d_qk], topk_idx [n, K_p], o [n, H, d_v]
 * and lse [n, H] hold the range's rows (n = t_end - t_begin, row r <->
 * query t_begin + r); k, v [S, d] hold every key.  Every row is
 * bit-identical to the same row of dsa_sparse_attn_fwd.  0 <= t_begin <=
 * t_end <= S, else DSA_ERR_INVALID_ARG; an empty range does nothing.
 * ws: DSA_WS_FWD. */
DSA_API dsa_status_t dsa_sparse_attn_fwd_range(const dsa_config_t* cfg, const void* q,
                                       const void* k, const void* v,
                                       const int32_t* topk_idx, int64_t t_begin,
                                       int64_t t_end, void* o, float* lse, void* ws,
                                       size_t ws_bytes, void* stream);

/* Step 6 for the queries [t_begin, t_end) only.  q, o, lse, dO, topk_idx
 * and dq hold the range's rows (as in dsa_sparse_attn_fwd_range); k, v
 * every key.  dq rows are bit-identical to dsa_sparse_attn_bwd's.  The
 * range's contributions to dK and dV are ADDED into the caller's fp32
 * accumulators dk_acc, dv_acc [S, d]: zero them before the first range and
 * convert them with dsa_accum_to_bf16 after the last (across GPUs, reduce
 * them first).  Over ranges that partition [0, S) the sums equal the
 * accumulators of dsa_sparse_attn_bwd up to the order of the fp32
 * additions, which the atomic scatter leaves unspecified in every case.
 * dv_acc == NULL requires v == k (K = V): dk_acc then receives dK + dV.
 * ws: DSA_WS_BWD_ROWS (the range's delta rows). */
DSA_API dsa_status_t dsa_sparse_attn_bwd_range(const dsa_config_t* cfg, const void* q,
                                       const void* k, const void* v, const void* o,
                                       const float* lse, const void* dO,
                                       const int32_t* topk_idx, int64_t t_begin,
                                       int64_t t_end, void* dq, float* dk_acc,
                                       float* dv_acc, void* ws, size_t ws_bytes,
                                       void* stream);

/* out[i] = bf16_rne(acc[i]) for n fp32 values, n a multiple of 4 (acc
 * 16-byte aligned, out 8-byte aligned). */
DSA_API dsa_status_t dsa_accum_to_bf16(const float* acc, void* out, int64_t n,
                               void* stream);

/* The tensors of one whole step (steps 1-6), all [S, ...] rows, dense:
 *   inputs : q_idx [S,H_I,D_I] bf16, k_idx [S,D_I] bf16, w [S,H_I] fp32,
 *            k_gate [S] fp32 or NULL (mean pools; else gated pools as in
 *            dsa_pool_keys_gated), q [S,H,d_qk] bf16, k [S,d_qk] bf16,
 *            v [S,d_v] bf16 (v == k: K = V, as in dsa_sparse_attn_fwd_kv),
 *            dO [S,H,d_v] bf16 or NULL (forward only);
 *   outputs: topk_idx [S,K_p] int32, o [S,H,d_v] bf16, lse [S,H] fp32, and
 *            with dO: dq [S,H,d_qk] bf16, dk [S,d_qk] bf16 (K = V: dK + dV),
 *            dv [S,d_v] bf16 (unused when K = V). */
typedef struct dsa_step_tensors {
  void* q_idx;
  void* k_idx;
  float* w;
  float* k_gate;
  void* q;
  void* k;
  void* v;
  void* dO;
  int32_t* topk_idx;
  void* o;
  float* lse;
  void* dq;
  void* dk;
  void* dv;
} dsa_step_tensors_t;

/* One whole step on device-resident tensors `dev`: dsa_index_scores_topk
 * (or the gated range call over every query), dsa_sparse_attn_fwd, and when
 * dO != NULL dsa_sparse_attn_bwd, in that order on `stream`, with one
 * workspace (ws: DSA_WS_STEP) and one status word.  Results equal those
 * calls'. */
DSA_API dsa_status_t dsa_step(const dsa_config_t* cfg, const dsa_step_tensors_t* dev,
                      void* ws, size_t ws_bytes, void* stream);

/* dsa_step with the inputs in and the outputs out of HOST memory: `host`
 * holds host pointers (page-locked, e.g. cudaHostAlloc, for the copies to
 * overlap anything), `dev` device buffers of the same shapes, which the call
 * fills and uses.  The queries are cut into n_chunks ranges (1..64) and
 * the copies run on h2d_stream and d2h_stream while the kernels run on
 * `stream`: the indexer inputs and K, V go first, then for each range its
 * q and dO rows; the forward and the backward of a range start as soon as
 * its rows have landed, and its o, lse and dq rows are copied back as soon
 * as they are final (the top-k indices after the indexer, dK and dV after
 * the last range).  The call orders itself after work already queued on
 * `stream`, and work queued on `stream` after it waits for the
 * last copy back, so synchronising `stream` makes every host output
 * valid.  Results equal dsa_step's, up to the order of dK/dV's fp32
 * additions.  The three streams must be distinct.  CUDA events are created
 * and released inside the call; no memory is allocated.  Argument errors
 * return before anything is queued; after DSA_ERR_CUDA part of the step may
 * already be queued on the three streams: synchronise them before reusing
 * any buffer.  ws: DSA_WS_STEP. */
DSA_API dsa_status_t dsa_step_host(const dsa_config_t* cfg,
                           const dsa_step_tensors_t* host,
                           const dsa_step_tensors_t* dev, int32_t n_chunks, void* ws,
                           size_t ws_bytes, void* stream, void* h2d_stream,
                           void* d2h_stream);

/* Allocation-free variant of dsa_index_scores_topk (the pages have no
 * counterpart: it exists for callers that cannot allocate device memory,
 * such as a plugin whose host application has reserved all device memory
 * for its own pool, or a service that forbids allocation after start-up).
 * The workspace is a fixed DSA_STATIC_SCRATCH_BYTES array inside the
 * library, held by every GPU that loads the library until the process
 * exits; problems whose DSA_WS_INDEX workspace exceeds it return
 * DSA_ERR_WORKSPACE_TOO_SMALL before anything is launched.  The first call
 * on a device looks up the array's device address (cudaGetSymbolAddress)
 * and caches it.  Every call shares the array: calls whose work overlaps on the GPU race, so
 * serialise them (one stream, or events).  The status-word header is
 * cleared at the start of each call; device-side errors that a call's
 * kernels latch there are read with dsa_static_device_status.  Results
 * equal dsa_index_scores_topk's.  No device memory is allocated by the
 * call.  A device ordinal of 64 or more returns DSA_ERR_UNSUPPORTED_SHAPE. */
#define DSA_STATIC_SCRATCH_BYTES (32u << 20)
DSA_API dsa_status_t dsa_index_scores_topk_static(const dsa_config_t* cfg,
                                                  const void* q_idx,
                                                  const void* k_idx,
                                                  const float* w,
                                                  int32_t* topk_idx,
                                                  void* stream);

/* dsa_get_device_status for the array of dsa_index_scores_topk_static on
 * the current device: synchronise `stream` (the stream of the static calls),
 * read the status word that their kernels latch into *device_status
 * (DSA_OK if nothing was latched) and clear it.  Allocates nothing. */
DSA_API dsa_status_t dsa_static_device_status(void* stream, uint32_t* device_status);

/* Synchronise `stream`, read the workspace status word into *device_status
 * (a dsa_status_t value, DSA_OK if nothing was latched) and clear it. */
DSA_API dsa_status_t dsa_get_device_status(void* ws, void* stream,
                                   uint32_t* device_status);

/* Check on this device that a bounded wait ends: one kernel thread waits,
 * through the waiter every kernel of the library uses, on an mbarrier that
 * nothing arrives on, for timeout_ms (1..10000) milliseconds, then latches
 * DSA_ERR_DEVICE_TIMEOUT in the workspace status word (any workspace; read
 * it with dsa_get_device_status) and returns.  Nothing faults or hangs and
 * the context stays usable. */
DSA_API dsa_status_t dsa_check_wait_timeout(void* ws, size_t ws_bytes, uint32_t timeout_ms,
                                    void* stream);

/* Static, human-readable name of a status code. */
DSA_API const char* dsa_status_string(dsa_status_t status);

/* DSA_ABI_VERSION of the loaded library. */
DSA_API int32_t dsa_abi_version(void);

/* Name of the CUDA runtime error behind the calling thread's most recent
 * DSA_ERR_CUDA (static string; "no error" if there was none). */
DSA_API const char* dsa_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* DSA_GB300_H */
