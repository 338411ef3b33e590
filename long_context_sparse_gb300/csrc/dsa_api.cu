// dsa_api.cu -- the C ABI declared in include/dsa.h: argument validation,
// workspace carving, the chunked indexer loop and kernel launches.  Host
// code only; every step of the path runs in this library's kernels.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

// NVTX range over the launches of one host step (a profiler shows it on the
// CPU timeline; without a tool attached it costs a call through a null hook).
// `value` (e.g. a chunk's first query) is attached as the range's payload.
class NvtxRange {
 public:
  NvtxRange(const char* name, int64_t value) {
    nvtxEventAttributes_t a = {};
    a.version = NVTX_VERSION;
    a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    a.messageType = NVTX_MESSAGE_TYPE_ASCII;
    a.message.ascii = name;
    a.payloadType = NVTX_PAYLOAD_TYPE_INT64;
    a.payload.llValue = value;
    nvtxRangePushEx(&a);
  }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr size_t kHeader = 256;        // status word + padding
constexpr int64_t kPoolTile = 128;     // score row pitch granularity
constexpr int kMaxDevices = 64;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Name of the CUDA error behind the last DSA_ERR_CUDA of this thread.
thread_local const char* t_last_cuda_error = "no error";
thread_local char t_detail[512] = "";
thread_local bool t_detail_set = false;

struct DeviceInfo {
  int num_sms = 0;
  int cc_major = 0, cc_minor = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

dsa_status_t device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return DSA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.num_sms == 0) {
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) !=
            cudaSuccess) {
      d.num_sms = 0;
      return DSA_ERR_CUDA;
    }
  }
  *out = d;
  return DSA_OK;
}

dsa_status_t get_encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p) {
      t_last_cuda_error = "cudaGetDriverEntryPointByVersion";
      return DSA_ERR_CUDA;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  *fn = g_encode;
  return DSA_OK;
}

// 2D bf16 row-major [rows, cols] tensor, box {64 cols, box_rows}, 128B swizzle.
dsa_status_t encode_2d(CUtensorMap* map, const void* base, uint64_t rows,
                       uint64_t cols, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  dsa_status_t st = get_encoder(&fn);
  if (st != DSA_OK) return st;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    t_last_cuda_error = "cuTensorMapEncodeTiled";
    return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

uint64_t timeout_ns() {
  static uint64_t v = [] {
    const char* e = getenv("DSA_WAIT_TIMEOUT_MS");
    double ms = e ? atof(e) : 2000.0;
    if (!(ms > 0)) ms = 2000.0;
    return (uint64_t)(ms * 1e6);
  }();
  return v;
}

bool is_pow2_upto(int x, int hi) { return x >= 1 && x <= hi && (x & (x - 1)) == 0; }

// Shape checks common to every entry point.  Values outside the problem
// statement are INVALID_ARG; valid values the kernels do not run are
// UNSUPPORTED_SHAPE (never a fallback).
dsa_status_t check_cfg(const dsa_config_t* c, bool need_index, bool need_attn) {
  if (!c) return DSA_ERR_INVALID_ARG;
  if (c->seq_len < 1 || c->pool_size < 1 || c->topk_pools < 1 || c->chunk_q < 1 ||
      c->n_local < 0 || c->idx_heads < 1 || c->idx_dim < 1 || c->attn_heads < 1 ||
      c->d_qk < 1 || c->d_v < 1 || !(c->sm_scale >= 0.f) || isinf(c->sm_scale))
    return DSA_ERR_INVALID_ARG;
  if (c->seq_len > (int64_t)1 << 26) return DSA_ERR_UNSUPPORTED_SHAPE;
  if (c->pool_size != 4) return DSA_ERR_UNSUPPORTED_SHAPE;
  if (c->topk_pools > 2048) return DSA_ERR_UNSUPPORTED_SHAPE;
  if (c->n_local != 0 && c->n_local != 3) return DSA_ERR_UNSUPPORTED_SHAPE;
  if (need_index) {
    if (!is_pow2_upto(c->idx_heads, 64)) return DSA_ERR_UNSUPPORTED_SHAPE;
    if (c->idx_dim != 64 && c->idx_dim != 128) return DSA_ERR_UNSUPPORTED_SHAPE;
    if (c->seq_len * (int64_t)c->idx_heads > ((int64_t)1 << 31) - 512)
      return DSA_ERR_UNSUPPORTED_SHAPE;
    if (c->chunk_q > 4096) return DSA_ERR_UNSUPPORTED_SHAPE;
  }
  if (need_attn) {
    if (c->attn_heads > 128) return DSA_ERR_UNSUPPORTED_SHAPE;
    if (c->d_qk != 128 && c->d_qk != 256 && c->d_qk != 512)
      return DSA_ERR_UNSUPPORTED_SHAPE;
    if (c->d_v != c->d_qk) return DSA_ERR_UNSUPPORTED_SHAPE;
  }
  return DSA_OK;
}

int64_t score_ld(const dsa_config_t* c) {
  int64_t P = c->seq_len / 4;
  if (P < 1) P = 1;
  return (int64_t)round_up((size_t)P, kPoolTile);
}

int64_t chunk_rows(const dsa_config_t* c) {
  return c->chunk_q < c->seq_len ? c->chunk_q : c->seq_len;
}

size_t ws_bytes_for(const dsa_config_t* c, int which) {
  const int64_t S = c->seq_len;
  switch (which) {
    case DSA_WS_INDEX: {
      const size_t kp = round_up((size_t)(S / 4) * c->idx_dim * 2, 256);
      const size_t sc = (size_t)chunk_rows(c) * score_ld(c) * 4;
      return kHeader + kp + sc;
    }
    case DSA_WS_FWD:
    case DSA_WS_STATUS:
      return kHeader;
    case DSA_WS_STREAM:  // pooled keys only: no score is stored
      return kHeader + round_up((size_t)(S / 4) * c->idx_dim * 2, 256);
    case DSA_WS_BWD: {
      const size_t dl = round_up((size_t)S * c->attn_heads * 4, 256);
      const size_t acc = round_up((size_t)S * c->d_qk * 4, 256);
      return kHeader + dl + 2 * acc;
    }
    case DSA_WS_BWD_ROWS:  // delta rows only: the accumulators are the caller's
      return kHeader + round_up((size_t)S * c->attn_heads * 4, 256);
    case DSA_WS_STEP:  // one header, the indexer's regions, then the backward's
      return ws_bytes_for(c, DSA_WS_INDEX) + ws_bytes_for(c, DSA_WS_BWD) - kHeader;
    default:
      return 0;
  }
}

dsa_status_t make_ctx(void* ws, void* stream, LaunchCtx* ctx) {
  DeviceInfo d;
  dsa_status_t st = device_info(&d);
  if (st != DSA_OK) return st;
  ctx->stream = reinterpret_cast<cudaStream_t>(stream);
  ctx->status = reinterpret_cast<uint32_t*>(ws);
  ctx->timeout_ns = timeout_ns();
  ctx->num_sms = d.num_sms;
  return DSA_OK;
}

dsa_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DSA_OK;
  if (t_detail_set) {
    t_last_cuda_error = t_detail;
    t_detail_set = false;
  } else {
    t_last_cuda_error = cudaGetErrorName(e);
  }
  return DSA_ERR_CUDA;
}

dsa_status_t check_ws(const dsa_config_t* cfg, int which, void* ws, size_t ws_bytes) {
  if (!ws) return DSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return DSA_ERR_MISALIGNED;
  if (ws_bytes < ws_bytes_for(cfg, which)) return DSA_ERR_WORKSPACE_TOO_SMALL;
  return DSA_OK;
}

AttnShape attn_shape(const dsa_config_t* c) {
  AttnShape s;
  s.S = c->seq_len;
  s.H = c->attn_heads;
  s.D = c->d_qk;
  s.K_p = c->topk_pools;
  s.n_loc = c->n_local;
  s.scale = c->sm_scale > 0.f ? c->sm_scale : 1.0f / sqrtf((float)c->d_qk);
  s.t_lo = 0;
  s.t_hi = c->seq_len;
  return s;
}

}  // namespace

void set_error_detail(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_detail, sizeof t_detail, fmt, ap);
  va_end(ap);
  t_detail_set = true;
}

namespace {

// One thread waits, through the same bounded waiter every kernel uses, on an
// mbarrier that nothing arrives on: the wait must run out after timeout_ns,
// latch DSA_ERR_DEVICE_TIMEOUT and return.
__global__ void wait_timeout_kernel(uint32_t* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  const Waiter W{&abort_flag, status, timeout_ns};
  if (threadIdx.x == 0) W.wait(smem_u32(&bar), 0);
}

}  // namespace

}  // namespace dsa

using namespace dsa;

extern "C" {

int32_t dsa_abi_version(void) { return DSA_ABI_VERSION; }

const char* dsa_last_cuda_error(void) { return t_last_cuda_error; }

const char* dsa_status_string(dsa_status_t s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED_SHAPE: return "DSA_ERR_UNSUPPORTED_SHAPE";
    case DSA_ERR_WORKSPACE_TOO_SMALL: return "DSA_ERR_WORKSPACE_TOO_SMALL";
    case DSA_ERR_MISALIGNED: return "DSA_ERR_MISALIGNED";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_DEVICE_TIMEOUT: return "DSA_ERR_DEVICE_TIMEOUT";
    case DSA_ERR_DEVICE_BAD_INDEX: return "DSA_ERR_DEVICE_BAD_INDEX";
    case DSA_ERR_SCRATCH_CAP: return "DSA_ERR_SCRATCH_CAP";
    case DSA_ERR_DEVICE_CHECK: return "DSA_ERR_DEVICE_CHECK";
  }
  return "DSA_ERR_UNKNOWN";
}

dsa_status_t dsa_workspace_size(const dsa_config_t* cfg, int32_t which, size_t* bytes) {
  if (!bytes) return DSA_ERR_INVALID_ARG;
  if (which < DSA_WS_INDEX || which > DSA_WS_STEP) return DSA_ERR_INVALID_ARG;
  dsa_status_t st = check_cfg(
      cfg, which == DSA_WS_INDEX || which == DSA_WS_STREAM || which == DSA_WS_STEP,
      which == DSA_WS_FWD || which == DSA_WS_BWD || which == DSA_WS_BWD_ROWS ||
          which == DSA_WS_STEP);
  if (st != DSA_OK) return st;
  *bytes = ws_bytes_for(cfg, which);
  return DSA_OK;
}

dsa_status_t dsa_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < kHeader) return DSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return DSA_ERR_MISALIGNED;
  return cuda_status(
      cudaMemsetAsync(ws, 0, kHeader, reinterpret_cast<cudaStream_t>(stream)));
}

dsa_status_t dsa_pool_keys(const dsa_config_t* cfg, const void* k_idx, void* k_pool,
                           void* stream) {
  dsa_status_t st = check_cfg(cfg, true, false);
  if (st != DSA_OK) return st;
  if (!k_idx || (!k_pool && cfg->seq_len >= 4)) return DSA_ERR_INVALID_ARG;
  if (!aligned16(k_idx) || !aligned16(k_pool)) return DSA_ERR_MISALIGNED;
  LaunchCtx ctx;
  st = make_ctx(nullptr, stream, &ctx);
  if (st != DSA_OK) return st;
  return cuda_status(launch_pool(ctx, static_cast<const __nv_bfloat16*>(k_idx),
                                 static_cast<__nv_bfloat16*>(k_pool), cfg->seq_len,
                                 cfg->idx_dim));
}

dsa_status_t dsa_pool_keys_gated(const dsa_config_t* cfg, const void* k_idx,
                                 const float* k_gate, void* k_pool, void* stream) {
  dsa_status_t st = check_cfg(cfg, true, false);
  if (st != DSA_OK) return st;
  if (!k_idx || !k_gate || (!k_pool && cfg->seq_len >= 4)) return DSA_ERR_INVALID_ARG;
  if (!aligned16(k_idx) || !aligned16(k_gate) || !aligned16(k_pool))
    return DSA_ERR_MISALIGNED;
  LaunchCtx ctx;
  st = make_ctx(nullptr, stream, &ctx);
  if (st != DSA_OK) return st;
  return cuda_status(launch_pool_gated(ctx, static_cast<const __nv_bfloat16*>(k_idx),
                                       k_gate, static_cast<__nv_bfloat16*>(k_pool),
                                       cfg->seq_len, cfg->idx_dim));
}

dsa_status_t dsa_index_scores(const dsa_config_t* cfg, const void* q_idx,
                              const void* k_pool, const float* w, int64_t t0,
                              int64_t rows, float* scores, int64_t ld, void* ws,
                              size_t ws_bytes, void* stream) {
  dsa_status_t st = check_cfg(cfg, true, false);
  if (st != DSA_OK) return st;
  if (!q_idx || !w || !scores || t0 < 0 || rows < 0 || t0 + rows > cfg->seq_len ||
      ld < 1 || (ld & 3) != 0)
    return DSA_ERR_INVALID_ARG;
  if (rows > 4096) return DSA_ERR_UNSUPPORTED_SHAPE;
  if ((st = check_ws(cfg, DSA_WS_STATUS, ws, ws_bytes)) != DSA_OK) return st;
  if (rows == 0) return DSA_OK;
  const int64_t p_lim = n_full(t0 + rows - 1);
  if (p_lim > ld) return DSA_ERR_INVALID_ARG;
  if (p_lim == 0) return DSA_OK;
  if (!k_pool) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_pool) || !aligned16(w) || !aligned16(scores))
    return DSA_ERR_MISALIGNED;
  LaunchCtx ctx;
  if ((st = make_ctx(ws, stream, &ctx)) != DSA_OK) return st;
  CUtensorMap qm, km;
  const int64_t S = cfg->seq_len;
  if ((st = encode_2d(&qm, q_idx, (uint64_t)(S * cfg->idx_heads), cfg->idx_dim, 256)) !=
      DSA_OK)
    return st;
  if ((st = encode_2d(&km, k_pool, (uint64_t)(S / 4), cfg->idx_dim, 128)) != DSA_OK)
    return st;
  return cuda_status(launch_indexer(ctx, qm, km, w, cfg->idx_heads, cfg->idx_dim, t0,
                                    0, rows, p_lim, scores, ld));
}

dsa_status_t dsa_topk_from_scores(const dsa_config_t* cfg, const float* scores,
                                  int64_t ld, int64_t row0, int64_t rows,
                                  int32_t* topk_idx, void* ws, size_t ws_bytes,
                                  void* stream) {
  dsa_status_t st = check_cfg(cfg, false, false);
  if (st != DSA_OK) return st;
  if (!scores || !topk_idx || ld < 1 || row0 < 0 || rows < 0 ||
      row0 + rows > cfg->seq_len)
    return DSA_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, DSA_WS_STATUS, ws, ws_bytes)) != DSA_OK) return st;
  if (!aligned16(scores) || !aligned16(topk_idx)) return DSA_ERR_MISALIGNED;
  if (rows == 0) return DSA_OK;
  LaunchCtx ctx;
  if ((st = make_ctx(ws, stream, &ctx)) != DSA_OK) return st;
  return cuda_status(
      launch_topk(ctx, scores, ld, row0, rows, cfg->topk_pools, topk_idx));
}

namespace {

// Steps 1-4 for the query rows [t_begin, t_end) on validated arguments: pool
// every key into k_pool, then one indexer + one top-k launch per chunk of C
// queries through the score chunk `scores`.  q_idx / w / topk_idx hold the
// range's rows only (row r <-> query t_begin + r).
dsa_status_t index_rows(const LaunchCtx& ctx, const dsa_config_t* cfg, const void* q_idx,
                        const void* k_idx, const float* k_gate, const float* w,
                        int64_t t_begin, int64_t t_end, int32_t* topk_idx,
                        __nv_bfloat16* k_pool, float* scores) {
  const int64_t S = cfg->seq_len, P = S / 4, C = chunk_rows(cfg), ld = score_ld(cfg);
  const int64_t n_q = t_end - t_begin;
  if (n_q == 0) return DSA_OK;
  dsa_status_t st;
  CUtensorMap qm, km;
  if (P > 0) {
    const __nv_bfloat16* kb = static_cast<const __nv_bfloat16*>(k_idx);
    cudaError_t e = k_gate ? launch_pool_gated(ctx, kb, k_gate, k_pool, S, cfg->idx_dim)
                           : launch_pool(ctx, kb, k_pool, S, cfg->idx_dim);
    if (e != cudaSuccess) return cuda_status(e);
    if ((st = encode_2d(&qm, q_idx, (uint64_t)(n_q * cfg->idx_heads), cfg->idx_dim,
                        256)) != DSA_OK)
      return st;
    if ((st = encode_2d(&km, k_pool, (uint64_t)P, cfg->idx_dim, 128)) != DSA_OK)
      return st;
  }
  for (int64_t t0 = t_begin; t0 < t_end; t0 += C) {
    const NvtxRange range("dsa.index_chunk", t0);
    const int64_t rows = (t_end - t0) < C ? (t_end - t0) : C;
    const int64_t p_lim = n_full(t0 + rows - 1);
    if (p_lim > cfg->topk_pools) {  // some row has more pools than K_p: score
      cudaError_t e = launch_indexer(ctx, qm, km, w, cfg->idx_heads, cfg->idx_dim, t0,
                                     t_begin, rows, p_lim, scores, ld);
      if (e != cudaSuccess) return cuda_status(e);
    }
    cudaError_t e = launch_topk(ctx, scores, ld, t0, rows, cfg->topk_pools,
                                topk_idx + (t0 - t_begin) * cfg->topk_pools);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return DSA_OK;
}

// The indexer's payload regions (after a header): pooled keys, score chunk.
__nv_bfloat16* index_k_pool(uint8_t* payload) {
  return reinterpret_cast<__nv_bfloat16*>(payload);
}
float* index_scores(const dsa_config_t* cfg, uint8_t* payload) {
  return reinterpret_cast<float*>(
      payload + round_up((size_t)(cfg->seq_len / 4) * cfg->idx_dim * 2, 256));
}

// Steps 1-4 for the query rows [t_begin, t_end), arguments checked.
dsa_status_t index_topk_rows(const dsa_config_t* cfg, const void* q_idx,
                             const void* k_idx, const float* k_gate, const float* w,
                             int64_t t_begin, int64_t t_end, int32_t* topk_idx,
                             void* ws, size_t ws_bytes, void* stream) {
  dsa_status_t st = check_cfg(cfg, true, false);
  if (st != DSA_OK) return st;
  if (t_begin < 0 || t_end < t_begin || t_end > cfg->seq_len) return DSA_ERR_INVALID_ARG;
  if (t_end == t_begin) return DSA_OK;  // nothing is read or written
  if (!q_idx || !k_idx || !w || !topk_idx) return DSA_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, DSA_WS_INDEX, ws, ws_bytes)) != DSA_OK) return st;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(w) || !aligned16(topk_idx) ||
      (k_gate && !aligned16(k_gate)))
    return DSA_ERR_MISALIGNED;
  const int64_t C = chunk_rows(cfg), ld = score_ld(cfg);
  if ((uint64_t)C * (uint64_t)ld * 4u > cfg->scratch_cap) return DSA_ERR_SCRATCH_CAP;
  LaunchCtx ctx;
  if ((st = make_ctx(ws, stream, &ctx)) != DSA_OK) return st;
  uint8_t* payload = static_cast<uint8_t*>(ws) + kHeader;
  return index_rows(ctx, cfg, q_idx, k_idx, k_gate, w, t_begin, t_end, topk_idx,
                    index_k_pool(payload), index_scores(cfg, payload));
}

}  // namespace

dsa_status_t dsa_index_scores_topk(const dsa_config_t* cfg, const void* q_idx,
                                   const void* k_idx, const float* w, int32_t* topk_idx,
                                   void* ws, size_t ws_bytes, void* stream) {
  if (!cfg) return DSA_ERR_INVALID_ARG;
  return index_topk_rows(cfg, q_idx, k_idx, nullptr, w, 0, cfg->seq_len, topk_idx, ws,
                         ws_bytes, stream);
}

dsa_status_t dsa_index_scores_topk_range(const dsa_config_t* cfg, const void* q_idx,
                                         const void* k_idx, const float* k_gate,
                                         const float* w, int64_t t_begin, int64_t t_end,
                                         int32_t* topk_idx, void* ws, size_t ws_bytes,
                                         void* stream) {
  return index_topk_rows(cfg, q_idx, k_idx, k_gate, w, t_begin, t_end, topk_idx, ws,
                         ws_bytes, stream);
}

dsa_status_t dsa_index_topk_streaming(const dsa_config_t* cfg, const void* q_idx,
                                      const void* k_idx, const float* k_gate,
                                      const float* w, int64_t t_begin, int64_t t_end,
                                      int32_t* topk_idx, void* ws, size_t ws_bytes,
                                      void* stream) {
  dsa_status_t st = check_cfg(cfg, true, false);
  if (st != DSA_OK) return st;
  if (!indexer_topk_supported(cfg->idx_heads, cfg->idx_dim, cfg->topk_pools))
    return DSA_ERR_UNSUPPORTED_SHAPE;
  if (t_begin < 0 || t_end < t_begin || t_end > cfg->seq_len) return DSA_ERR_INVALID_ARG;
  if (t_end == t_begin) return DSA_OK;  // nothing is read or written
  if (!q_idx || !k_idx || !w || !topk_idx) return DSA_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, DSA_WS_STREAM, ws, ws_bytes)) != DSA_OK) return st;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(w) || !aligned16(topk_idx) ||
      (k_gate && !aligned16(k_gate)))
    return DSA_ERR_MISALIGNED;
  LaunchCtx ctx;
  if ((st = make_ctx(ws, stream, &ctx)) != DSA_OK) return st;
  const int64_t S = cfg->seq_len, P = S / 4, n_q = t_end - t_begin;
  __nv_bfloat16* k_pool = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(ws) +
                                                           kHeader);
  const __nv_bfloat16* kb = static_cast<const __nv_bfloat16*>(k_idx);
  cudaError_t e = k_gate ? launch_pool_gated(ctx, kb, k_gate, k_pool, S, cfg->idx_dim)
                         : launch_pool(ctx, kb, k_pool, S, cfg->idx_dim);
  if (e != cudaSuccess) return cuda_status(e);
  CUtensorMap qm, km;
  if ((st = encode_2d(&qm, q_idx, (uint64_t)(n_q * cfg->idx_heads), cfg->idx_dim, 256)) !=
      DSA_OK)
    return st;
  if ((st = encode_2d(&km, P > 0 ? (const void*)k_pool : k_idx, (uint64_t)(P > 0 ? P : 1),
                      cfg->idx_dim, 128)) != DSA_OK)
    return st;
  e = launch_indexer_topk(ctx, qm, km, w, cfg->idx_heads, cfg->idx_dim, t_begin, t_end,
                          cfg->topk_pools, topk_idx);
  return cuda_status(e);
}

namespace {

bool valid_range(const dsa_config_t* cfg, int64_t t_begin, int64_t t_end) {
  return t_begin >= 0 && t_begin <= t_end && t_end <= cfg->seq_len;
}

// Step 5 for the queries s.t_lo .. s.t_hi - 1; q, idx, o and lse hold those
// rows (row r <-> query s.t_lo + r), k and v every key.
dsa_status_t fwd_rows(const LaunchCtx& ctx, const AttnShape& s, const void* q,
                      const void* k, const void* v, const int32_t* idx, void* o,
                      float* lse) {
  const int64_t n = s.t_hi - s.t_lo;
  if (n == 0) return DSA_OK;
  const NvtxRange range("dsa.attn_fwd", s.t_lo);
  CUtensorMap qm;
  dsa_status_t st = encode_2d(&qm, q, (uint64_t)(n * s.H), (uint64_t)s.D,
                              (uint32_t)attn_tc_heads(s.H));
  if (st != DSA_OK) return st;
  cudaError_t e = launch_attn_fwd_tc(ctx, s, qm, static_cast<const __nv_bfloat16*>(k),
                                     static_cast<const __nv_bfloat16*>(v), idx,
                                     static_cast<__nv_bfloat16*>(o), lse);
  return e == cudaErrorInvalidValue ? DSA_ERR_UNSUPPORTED_SHAPE : cuda_status(e);
}

// a7-a8 for the queries s.t_lo .. s.t_hi - 1 (row-indexed buffers as in
// fwd_rows; delta holds the rows too): dq rows, and the rows' dK/dV
// contributions added into dk_acc / dv_acc (dv_acc == nullptr: K = V,
// dk_acc receives dK + dV).
dsa_status_t bwd_rows(const LaunchCtx& ctx, const AttnShape& s, const void* q,
                      const void* k, const void* v, const void* o, const float* lse,
                      const void* dO, const int32_t* idx, void* dq, float* delta,
                      float* dk_acc, float* dv_acc) {
  const int64_t n = s.t_hi - s.t_lo;
  if (n == 0) return DSA_OK;
  const NvtxRange range("dsa.attn_bwd", s.t_lo);
  cudaError_t e = launch_attn_bwd_delta(ctx, s, static_cast<const __nv_bfloat16*>(o),
                                        static_cast<const __nv_bfloat16*>(dO), delta);
  if (e != cudaSuccess) return cuda_status(e);
  CUtensorMap qm, gm;
  dsa_status_t st;
  if ((st = encode_2d(&qm, q, (uint64_t)(n * s.H), (uint64_t)s.D, 64)) != DSA_OK)
    return st;
  if ((st = encode_2d(&gm, dO, (uint64_t)(n * s.H), (uint64_t)s.D, 64)) != DSA_OK)
    return st;
  e = launch_attn_bwd_tc(ctx, s, qm, gm, static_cast<const __nv_bfloat16*>(k),
                         static_cast<const __nv_bfloat16*>(v), lse, delta, idx,
                         static_cast<__nv_bfloat16*>(dq), dk_acc, dv_acc);
  if (e == cudaErrorInvalidValue) return DSA_ERR_UNSUPPORTED_SHAPE;
  return cuda_status(e);
}

// Payload regions of a backward workspace (after the header).
struct BwdRegions {
  float* delta;
  float* dk_acc;
  float* dv_acc;
};
BwdRegions bwd_regions(const dsa_config_t* cfg, uint8_t* payload, bool kv) {
  const int64_t S = cfg->seq_len;
  BwdRegions r;
  r.delta = reinterpret_cast<float*>(payload);
  r.dk_acc = reinterpret_cast<float*>(payload +
                                      round_up((size_t)S * cfg->attn_heads * 4, 256));
  r.dv_acc = kv ? nullptr : r.dk_acc + round_up((size_t)S * cfg->d_qk * 4, 256) / 4;
  return r;
}

dsa_status_t fwd_checked(const dsa_config_t* cfg, const void* q, const void* k,
                         const void* v, const int32_t* topk_idx, int64_t t_begin,
                         int64_t t_end, void* o, float* lse, void* ws, size_t ws_bytes,
                         void* stream) {
  dsa_status_t st = check_cfg(cfg, false, true);
  if (st != DSA_OK) return st;
  if (!valid_range(cfg, t_begin, t_end)) return DSA_ERR_INVALID_ARG;
  if (t_end == t_begin) return DSA_OK;  // nothing is read or written
  if (!q || !k || !v || !topk_idx || !o || !lse) return DSA_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, DSA_WS_FWD, ws, ws_bytes)) != DSA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(topk_idx) ||
      !aligned16(o) || !aligned16(lse))
    return DSA_ERR_MISALIGNED;
  LaunchCtx ctx;
  if ((st = make_ctx(ws, stream, &ctx)) != DSA_OK) return st;
  AttnShape s = attn_shape(cfg);
  s.t_lo = t_begin;
  s.t_hi = t_end;
  return fwd_rows(ctx, s, q, k, v, topk_idx, o, lse);
}

// a7-a9 over every query.  kv: K and V are the one tensor k; dk receives
// dK + dV (dv unused).
dsa_status_t attn_bwd(const dsa_config_t* cfg, const void* q, const void* k,
                      const void* v, const void* o, const float* lse, const void* dO,
                      const int32_t* topk_idx, void* dq, void* dk, void* dv, bool kv,
                      void* ws, size_t ws_bytes, void* stream) {
  dsa_status_t st = check_cfg(cfg, false, true);
  if (st != DSA_OK) return st;
  if (!q || !k || !v || !o || !lse || !dO || !topk_idx || !dq || !dk || !dv)
    return DSA_ERR_INVALID_ARG;
  if ((st = check_ws(cfg, DSA_WS_BWD, ws, ws_bytes)) != DSA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      !aligned16(lse) || !aligned16(dO) || !aligned16(topk_idx) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv))
    return DSA_ERR_MISALIGNED;
  LaunchCtx ctx;
  if ((st = make_ctx(ws, stream, &ctx)) != DSA_OK) return st;
  const AttnShape s = attn_shape(cfg);
  const BwdRegions r = bwd_regions(cfg, static_cast<uint8_t*>(ws) + kHeader, kv);
  cudaError_t e = launch_attn_bwd_zero(ctx, s, r.dk_acc, r.dv_acc);
  if (e != cudaSuccess) return cuda_status(e);
  if ((st = bwd_rows(ctx, s, q, k, v, o, lse, dO, topk_idx, dq, r.delta, r.dk_acc,
                     r.dv_acc)) != DSA_OK)
    return st;
  e = launch_attn_bwd_finalize(ctx, s, r.dk_acc, r.dv_acc, static_cast<__nv_bfloat16*>(dk),
                               static_cast<__nv_bfloat16*>(dv));
  return cuda_status(e);
}

}  // namespace

dsa_status_t dsa_sparse_attn_fwd(const dsa_config_t* cfg, const void* q, const void* k,
                                 const void* v, const int32_t* topk_idx, void* o,
                                 float* lse, void* ws, size_t ws_bytes, void* stream) {
  if (!cfg) return DSA_ERR_INVALID_ARG;
  return fwd_checked(cfg, q, k, v, topk_idx, 0, cfg->seq_len, o, lse, ws, ws_bytes,
                     stream);
}

dsa_status_t dsa_sparse_attn_fwd_range(const dsa_config_t* cfg, const void* q,
                                       const void* k, const void* v,
                                       const int32_t* topk_idx, int64_t t_begin,
                                       int64_t t_end, void* o, float* lse, void* ws,
                                       size_t ws_bytes, void* stream) {
  return fwd_checked(cfg, q, k, v, topk_idx, t_begin, t_end, o, lse, ws, ws_bytes,
                     stream);
}

dsa_status_t dsa_sparse_attn_fwd_kv(const dsa_config_t* cfg, const void* q, const void* kv,
                                    const int32_t* topk_idx, void* o, float* lse, void* ws,
                                    size_t ws_bytes, void* stream) {
  return dsa_sparse_attn_fwd(cfg, q, kv, kv, topk_idx, o, lse, ws, ws_bytes, stream);
}

dsa_status_t dsa_sparse_attn_bwd(const dsa_config_t* cfg, const void* q, const void* k,
                                 const void* v, const void* o, const float* lse,
                                 const void* dO, const int32_t* topk_idx, void* dq,
                                 void* dk, void* dv, void* ws, size_t ws_bytes,
                                 void* stream) {
  return attn_bwd(cfg, q, k, v, o, lse, dO, topk_idx, dq, dk, dv, false, ws, ws_bytes,
                  stream);
}

dsa_status_t dsa_sparse_attn_bwd_kv(const dsa_config_t* cfg, const void* q, const void* kv,
                                    const void* o, const float* lse, const void* dO,
                                    const int32_t* topk_idx, void* dq, void* dkv, void* ws,
                                    size_t ws_bytes, void* stream) {
  return attn_bwd(cfg, q, kv, kv, o, lse, dO, topk_idx, dq, dkv, dkv, true, ws, ws_bytes,
                  stream);
}

dsa_status_t dsa_sparse_attn_bwd_range(const dsa_config_t* cfg, const void* q,
                                       const void* k, const void* v, const void* o,
                                       const float* lse, const void* dO,
                                       const int32_t* topk_idx, int64_t t_begin,
                                       int64_t t_end, void* dq, float* dk_acc,
                                       float* dv_acc, void* ws, size_t ws_bytes,
                                       void* stream) {
  dsa_status_t st = check_cfg(cfg, false, true);
  if (st != DSA_OK) return st;
  if (!valid_range(cfg, t_begin, t_end)) return DSA_ERR_INVALID_ARG;
  if (t_end == t_begin) return DSA_OK;  // nothing is read or written
  if (!q || !k || !v || !o || !lse || !dO || !topk_idx || !dq || !dk_acc)
    return DSA_ERR_INVALID_ARG;
  if (!dv_acc && v != k) return DSA_ERR_INVALID_ARG;  // one accumulator: K = V only
  if ((st = check_ws(cfg, DSA_WS_BWD_ROWS, ws, ws_bytes)) != DSA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      !aligned16(lse) || !aligned16(dO) || !aligned16(topk_idx) || !aligned16(dq) ||
      !aligned16(dk_acc) || (dv_acc && !aligned16(dv_acc)))
    return DSA_ERR_MISALIGNED;
  LaunchCtx ctx;
  if ((st = make_ctx(ws, stream, &ctx)) != DSA_OK) return st;
  AttnShape s = attn_shape(cfg);
  s.t_lo = t_begin;
  s.t_hi = t_end;
  float* delta = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kHeader);
  return bwd_rows(ctx, s, q, k, v, o, lse, dO, topk_idx, dq, delta, dk_acc, dv_acc);
}

dsa_status_t dsa_accum_to_bf16(const float* acc, void* out, int64_t n, void* stream) {
  if (n < 0 || (n & 3) != 0) return DSA_ERR_INVALID_ARG;
  if (n == 0) return DSA_OK;
  if (!acc || !out) return DSA_ERR_INVALID_ARG;
  if (!aligned16(acc) || (reinterpret_cast<uintptr_t>(out) & 7u) != 0)
    return DSA_ERR_MISALIGNED;
  LaunchCtx ctx;
  dsa_status_t st = make_ctx(nullptr, stream, &ctx);
  if (st != DSA_OK) return st;
  return cuda_status(launch_f32_to_bf16(ctx, acc, static_cast<__nv_bfloat16*>(out), n));
}

namespace {

// Which optional parts a step has, from its tensor set.
struct StepKind {
  bool kv;     // v == k: one tensor as keys and values
  bool bwd;    // dO given: run the backward
  bool gated;  // k_gate given: gated pools
};

dsa_status_t check_step_tensors(const dsa_step_tensors_t* t, bool device, StepKind* kind) {
  if (!t) return DSA_ERR_INVALID_ARG;
  if (!t->q_idx || !t->k_idx || !t->w || !t->q || !t->k || !t->v || !t->topk_idx ||
      !t->o || !t->lse)
    return DSA_ERR_INVALID_ARG;
  kind->kv = t->v == t->k;
  kind->bwd = t->dO != nullptr;
  kind->gated = t->k_gate != nullptr;
  if (kind->bwd && (!t->dq || !t->dk || (!kind->kv && !t->dv))) return DSA_ERR_INVALID_ARG;
  if (device) {
    const void* ps[] = {t->q_idx, t->k_idx, t->w, t->k_gate, t->q, t->k, t->v, t->dO,
                        t->topk_idx, t->o, t->lse, t->dq, t->dk, t->dv};
    for (const void* p : ps)
      if (p && !aligned16(p)) return DSA_ERR_MISALIGNED;
  }
  return DSA_OK;
}

// Regions of a DSA_WS_STEP workspace: one header, then the indexer's
// payload (pooled keys, score chunk), then the backward's (delta, dK, dV).
struct StepRegions {
  __nv_bfloat16* k_pool;
  float* scores;
  BwdRegions bwd;
};
StepRegions step_regions(const dsa_config_t* cfg, void* ws, bool kv) {
  uint8_t* payload = static_cast<uint8_t*>(ws) + kHeader;
  StepRegions r;
  r.k_pool = index_k_pool(payload);
  r.scores = index_scores(cfg, payload);
  r.bwd = bwd_regions(cfg, payload + (ws_bytes_for(cfg, DSA_WS_INDEX) - kHeader), kv);
  return r;
}

dsa_status_t check_step_common(const dsa_config_t* cfg, void* ws, size_t ws_bytes) {
  dsa_status_t st = check_cfg(cfg, true, true);
  if (st != DSA_OK) return st;
  if ((uint64_t)chunk_rows(cfg) * (uint64_t)score_ld(cfg) * 4u > cfg->scratch_cap)
    return DSA_ERR_SCRATCH_CAP;
  return check_ws(cfg, DSA_WS_STEP, ws, ws_bytes);
}

// Events of one call, released when the call returns (a recorded event
// that is still pending is released by CUDA once it completes).
struct EventPool {
  cudaEvent_t ev[6 * 64 + 8];  // 6 per query range + 4 (at most 64 ranges)
  int n = 0;
  ~EventPool() {
    for (int i = 0; i < n; ++i) cudaEventDestroy(ev[i]);
  }
  // Record a new event on `from` and make `to` wait for it.
  cudaError_t link(cudaStream_t from, cudaStream_t to) {
    if (n == (int)(sizeof ev / sizeof ev[0])) return cudaErrorInvalidValue;
    cudaError_t e = cudaEventCreateWithFlags(&ev[n], cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
    cudaEvent_t x = ev[n++];
    if ((e = cudaEventRecord(x, from)) != cudaSuccess) return e;
    return cudaStreamWaitEvent(to, x, 0);
  }
};

}  // namespace

dsa_status_t dsa_step(const dsa_config_t* cfg, const dsa_step_tensors_t* dev, void* ws,
                      size_t ws_bytes, void* stream) {
  dsa_status_t st = check_step_common(cfg, ws, ws_bytes);
  if (st != DSA_OK) return st;
  StepKind kind;
  if ((st = check_step_tensors(dev, true, &kind)) != DSA_OK) return st;
  LaunchCtx ctx;
  if ((st = make_ctx(ws, stream, &ctx)) != DSA_OK) return st;
  const StepRegions r = step_regions(cfg, ws, kind.kv);
  const int64_t S = cfg->seq_len;
  if ((st = index_rows(ctx, cfg, dev->q_idx, dev->k_idx, dev->k_gate, dev->w, 0, S,
                       dev->topk_idx, r.k_pool, r.scores)) != DSA_OK)
    return st;
  const AttnShape s = attn_shape(cfg);
  if ((st = fwd_rows(ctx, s, dev->q, dev->k, dev->v, dev->topk_idx, dev->o, dev->lse)) !=
      DSA_OK)
    return st;
  if (!kind.bwd) return DSA_OK;
  cudaError_t e = launch_attn_bwd_zero(ctx, s, r.bwd.dk_acc, r.bwd.dv_acc);
  if (e != cudaSuccess) return cuda_status(e);
  if ((st = bwd_rows(ctx, s, dev->q, dev->k, dev->v, dev->o, dev->lse, dev->dO,
                     dev->topk_idx, dev->dq, r.bwd.delta, r.bwd.dk_acc, r.bwd.dv_acc)) !=
      DSA_OK)
    return st;
  return cuda_status(launch_attn_bwd_finalize(ctx, s, r.bwd.dk_acc, r.bwd.dv_acc,
                                              static_cast<__nv_bfloat16*>(dev->dk),
                                              static_cast<__nv_bfloat16*>(dev->dv)));
}

dsa_status_t dsa_step_host(const dsa_config_t* cfg, const dsa_step_tensors_t* host,
                           const dsa_step_tensors_t* dev, int32_t n_chunks, void* ws,
                           size_t ws_bytes, void* stream, void* h2d_stream,
                           void* d2h_stream) {
  dsa_status_t st = check_step_common(cfg, ws, ws_bytes);
  if (st != DSA_OK) return st;
  StepKind kh, kd;
  if ((st = check_step_tensors(host, false, &kh)) != DSA_OK) return st;
  if ((st = check_step_tensors(dev, true, &kd)) != DSA_OK) return st;
  if (kh.kv != kd.kv || kh.bwd != kd.bwd || kh.gated != kd.gated)
    return DSA_ERR_INVALID_ARG;  // the two tensor sets describe different steps
  if (n_chunks < 1 || n_chunks > 64) return DSA_ERR_INVALID_ARG;
  if (stream == h2d_stream || stream == d2h_stream || h2d_stream == d2h_stream)
    return DSA_ERR_INVALID_ARG;
  LaunchCtx ctx;
  if ((st = make_ctx(ws, stream, &ctx)) != DSA_OK) return st;
  const StepRegions r = step_regions(cfg, ws, kd.kv);
  const cudaStream_t cs = ctx.stream;
  const cudaStream_t hs = reinterpret_cast<cudaStream_t>(h2d_stream);
  const cudaStream_t ds = reinterpret_cast<cudaStream_t>(d2h_stream);
  const int64_t S = cfg->seq_len, H = cfg->attn_heads, D = cfg->d_qk;
  const int64_t HI = cfg->idx_heads, DI = cfg->idx_dim, Kp = cfg->topk_pools;
  const size_t q_row = (size_t)H * D * 2, lse_row = (size_t)H * 4;
  // query ranges: equal shares rounded to multiples of 4 rows, which keeps
  // every row-offset pointer 16-byte aligned
  int64_t per = (S + n_chunks - 1) / n_chunks;
  per = (per + 3) / 4 * 4;
  EventPool ev;
  cudaError_t e;
  auto up = [&](void* d, const void* h, size_t bytes) {
    return cudaMemcpyAsync(d, h, bytes, cudaMemcpyHostToDevice, hs);
  };
  auto down = [&](void* h, const void* d, size_t bytes) {
    return cudaMemcpyAsync(h, d, bytes, cudaMemcpyDeviceToHost, ds);
  };
#define DSA_TRY(x)                                  \
  do {                                              \
    if ((e = (x)) != cudaSuccess) return cuda_status(e); \
  } while (0)
  // everything queued on `stream` before the call comes first
  DSA_TRY(ev.link(cs, hs));
  DSA_TRY(ev.link(cs, ds));
  if (kd.bwd) DSA_TRY(launch_attn_bwd_zero(ctx, attn_shape(cfg), r.bwd.dk_acc, r.bwd.dv_acc));
  // ---- the indexer, range by range as each range's q_idx rows land (the
  // keys and weights first: every range pools all keys)
  DSA_TRY(up(dev->k_idx, host->k_idx, (size_t)S * DI * 2));
  DSA_TRY(up(dev->w, host->w, (size_t)S * HI * 4));
  if (kd.gated) DSA_TRY(up(dev->k_gate, host->k_gate, (size_t)S * 4));
  const size_t qi_row = (size_t)HI * DI * 2;
  for (int64_t t0 = 0; t0 < S; t0 += per) {
    const int64_t t1 = t0 + per < S ? t0 + per : S, n = t1 - t0;
    DSA_TRY(up(static_cast<uint8_t*>(dev->q_idx) + t0 * qi_row,
               static_cast<const uint8_t*>(host->q_idx) + t0 * qi_row, n * qi_row));
    DSA_TRY(ev.link(hs, cs));  // keys, weights and this range's q_idx
    if ((st = index_rows(ctx, cfg, static_cast<const uint8_t*>(dev->q_idx) + t0 * qi_row,
                         dev->k_idx, dev->k_gate, dev->w + t0 * HI, t0, t1,
                         dev->topk_idx + t0 * Kp, r.k_pool, r.scores)) != DSA_OK)
      return st;
    DSA_TRY(ev.link(cs, ds));  // this range's selection is final
    DSA_TRY(down(host->topk_idx + t0 * Kp, dev->topk_idx + t0 * Kp, n * Kp * 4));
  }
  DSA_TRY(up(dev->k, host->k, (size_t)S * D * 2));
  if (!kd.kv) DSA_TRY(up(dev->v, host->v, (size_t)S * D * 2));
  // ---- per query range: q (and dO) up, forward (and backward), rows down
  for (int64_t t0 = 0; t0 < S; t0 += per) {
    const int64_t t1 = t0 + per < S ? t0 + per : S, n = t1 - t0;
    AttnShape s = attn_shape(cfg);
    s.t_lo = t0;
    s.t_hi = t1;
    uint8_t* dq_rows = static_cast<uint8_t*>(dev->q) + t0 * q_row;
    uint8_t* do_rows = kd.bwd ? static_cast<uint8_t*>(dev->dO) + t0 * q_row : nullptr;
    uint8_t* o_rows = static_cast<uint8_t*>(dev->o) + t0 * q_row;
    float* lse_rows = dev->lse + t0 * H;
    int32_t* idx_rows = dev->topk_idx + t0 * Kp;
    DSA_TRY(up(dq_rows, static_cast<const uint8_t*>(host->q) + t0 * q_row, n * q_row));
    DSA_TRY(ev.link(hs, cs));  // K, V (first range) and this range's q
    if ((st = fwd_rows(ctx, s, dq_rows, dev->k, dev->v, idx_rows, o_rows, lse_rows)) !=
        DSA_OK)
      return st;
    DSA_TRY(ev.link(cs, ds));  // o and lse rows are final
    DSA_TRY(down(static_cast<uint8_t*>(host->o) + t0 * q_row, o_rows, n * q_row));
    DSA_TRY(down(host->lse + t0 * H, lse_rows, n * lse_row));
    if (!kd.bwd) continue;
    DSA_TRY(up(do_rows, static_cast<const uint8_t*>(host->dO) + t0 * q_row, n * q_row));
    DSA_TRY(ev.link(hs, cs));  // this range's dO
    uint8_t* dqr = static_cast<uint8_t*>(dev->dq) + t0 * q_row;
    if ((st = bwd_rows(ctx, s, dq_rows, dev->k, dev->v, o_rows, lse_rows, do_rows,
                       idx_rows, dqr, r.bwd.delta, r.bwd.dk_acc, r.bwd.dv_acc)) != DSA_OK)
      return st;
    DSA_TRY(ev.link(cs, ds));  // dq rows are final
    DSA_TRY(down(static_cast<uint8_t*>(host->dq) + t0 * q_row, dqr, n * q_row));
  }
  if (kd.bwd) {
    DSA_TRY(launch_attn_bwd_finalize(ctx, attn_shape(cfg), r.bwd.dk_acc, r.bwd.dv_acc,
                                     static_cast<__nv_bfloat16*>(dev->dk),
                                     static_cast<__nv_bfloat16*>(dev->dv)));
    DSA_TRY(ev.link(cs, ds));
    DSA_TRY(down(host->dk, dev->dk, (size_t)S * D * 2));
    if (!kd.kv) DSA_TRY(down(host->dv, dev->dv, (size_t)S * D * 2));
  }
  // work queued on `stream` after the call waits for the last copy back
  DSA_TRY(ev.link(ds, cs));
#undef DSA_TRY
  return DSA_OK;
}

dsa_status_t dsa_check_wait_timeout(void* ws, size_t ws_bytes, uint32_t timeout_ms,
                                    void* stream) {
  if (!ws || ws_bytes < kHeader || timeout_ms < 1 || timeout_ms > 10000)
    return DSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return DSA_ERR_MISALIGNED;
  LaunchCtx ctx;
  dsa_status_t st = make_ctx(ws, stream, &ctx);
  if (st != DSA_OK) return st;
  wait_timeout_kernel<<<1, 32, 0, ctx.stream>>>(ctx.status, (uint64_t)timeout_ms * 1000000u);
  return cuda_status(cudaGetLastError());
}

dsa_status_t dsa_get_device_status(void* ws, void* stream, uint32_t* device_status) {
  if (!ws || !device_status) return DSA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DSA_ERR_CUDA;
  if (cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof v, s) != cudaSuccess) return DSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DSA_ERR_CUDA;
  *device_status = v;
  return DSA_OK;
}

}  // extern "C"
