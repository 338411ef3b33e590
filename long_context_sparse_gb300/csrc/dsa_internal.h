// dsa_internal.h -- launchers shared between the C-ABI layer and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dsa {

// Record a printf-style detail for the calling thread's next DSA_ERR_CUDA
// (returned by dsa_last_cuda_error).
void set_error_detail(const char* fmt, ...);

struct LaunchCtx {
  cudaStream_t stream;
  uint32_t* status;     // device status word (workspace header)
  uint64_t timeout_ns;  // bounded-wait limit for every spin in the kernels
  int num_sms;
};

// a1: k_pool[p] = bf16(((k0 + k1) + (k2 + k3)) * 0.25), fp32.
cudaError_t launch_pool(const LaunchCtx& c, const __nv_bfloat16* k_idx,
                        __nv_bfloat16* k_pool, int64_t S, int D_I);

// a1 with gates: softmax of gate[4p..4p+3] weights the pool's keys (fp32),
// then bf16 RNE.  gate [S] fp32, 16-byte aligned.
cudaError_t launch_pool_gated(const LaunchCtx& c, const __nv_bfloat16* k_idx,
                              const float* gate, __nv_bfloat16* k_pool, int64_t S,
                              int D_I);

// a2 + a4 fused: the indexer whose epilogue keeps each query's selection
// in shared memory (no score is stored).  q_map over the range's rows
// [n_q*H_I, D_I] box {64, 256}; w [n_q, H_I]; out [n_q, K_p].
bool indexer_topk_supported(int H_I, int D_I, int K_p);
cudaError_t launch_indexer_topk(const LaunchCtx& c, const CUtensorMap& q_map,
                                const CUtensorMap& k_map, const float* w, int H_I,
                                int D_I, int64_t t_begin, int64_t t_end, int K_p,
                                int32_t* out);

// a4: per-row top-k over fp32 scores (row r <-> query row0 + r).
cudaError_t launch_topk(const LaunchCtx& c, const float* scores, int64_t ld,
                        int64_t row0, int64_t rows, int K_p, int32_t* out);

// a2: indexer scores for queries t0 .. t0+rows-1 against pools < p_lim.
// q_map: q_idx viewed as [rows_q*H_I, D_I] bf16, box {64, 256}, and w
// [rows_q, H_I], whose row 0 is query q0 (q0 = 0 for whole-sequence
// tensors); k_map: k_pool [P, D_I] bf16, box {64, 128}.
cudaError_t launch_indexer(const LaunchCtx& c, const CUtensorMap& q_map,
                           const CUtensorMap& k_map, const float* w, int H_I,
                           int D_I, int64_t t0, int64_t q0, int64_t rows,
                           int64_t p_lim, float* scores, int64_t ld);

struct AttnShape {
  int64_t S;
  int H;
  int D;        // d_qk == d_v
  int K_p;
  int n_loc;
  float scale;
  // queries [t_lo, t_hi) of the call; the per-query buffers (q, idx, o,
  // lse, dO, dq, delta) hold those rows only, row r <-> query t_lo + r
  int64_t t_lo = 0;
  int64_t t_hi = 0;
};

// Heads per tensor-core tile (N) of the attention kernels: H, or 64 per
// head block, rounded up to 16, 32 or 64.
int attn_tc_heads(int H);

// a5 + a6: sparse attention forward (tcgen05) for queries s.t_lo ..
// s.t_hi - 1.  q_map: the call's q rows viewed as [(t_hi - t_lo)*H, D]
// bf16, box {64, attn_tc_heads(H)}, 128-byte swizzle; idx, o, lse hold the
// call's rows too.
cudaError_t launch_attn_fwd_tc(const LaunchCtx& c, const AttnShape& s,
                               const CUtensorMap& q_map, const __nv_bfloat16* k,
                               const __nv_bfloat16* v, const int32_t* idx,
                               __nv_bfloat16* o, float* lse);

// a7 for the call's query rows: delta = rowsum(dO * O); also restarts the
// backward's work counter.
cudaError_t launch_attn_bwd_delta(const LaunchCtx& c, const AttnShape& s,
                                  const __nv_bfloat16* o, const __nv_bfloat16* dO,
                                  float* delta);

// Zero the fp32 dK/dV accumulators of all S keys (dv_acc may be nullptr).
cudaError_t launch_attn_bwd_zero(const LaunchCtx& c, const AttnShape& s, float* dk_acc,
                                 float* dv_acc);

// a8: sparse attention backward on tcgen05 (dQ direct, dK/dV fp32 scatter)
// for queries s.t_lo .. s.t_hi - 1.  q_map / g_map: the call's q and dO
// rows viewed as [(t_hi - t_lo)*H, D] bf16, box {64, 64}; lse, delta, idx
// and dq hold the call's rows; dk_acc / dv_acc span every key.
// dv_acc == nullptr: K and V are one tensor; dk_acc receives dK + dV.
cudaError_t launch_attn_bwd_tc(const LaunchCtx& c, const AttnShape& s,
                               const CUtensorMap& q_map, const CUtensorMap& g_map,
                               const __nv_bfloat16* k, const __nv_bfloat16* v,
                               const float* lse, const float* delta,
                               const int32_t* idx, __nv_bfloat16* dq, float* dk_acc,
                               float* dv_acc);

// a9 on n values (n a multiple of 4, 16-byte aligned): bf16 round to nearest even.
cudaError_t launch_f32_to_bf16(const LaunchCtx& c, const float* a, __nv_bfloat16* out,
                               int64_t n);

// a9: fp32 accumulators -> bf16 dK, dV.
cudaError_t launch_attn_bwd_finalize(const LaunchCtx& c, const AttnShape& s,
                                     const float* dk_acc, const float* dv_acc,
                                     __nv_bfloat16* dk, __nv_bfloat16* dv);

}  // namespace dsa
