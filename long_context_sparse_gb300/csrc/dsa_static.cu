// dsa_static.cu -- dsa_index_scores_topk_static: the indexer + top-k entry
// point for callers that cannot allocate device memory.
//
// Some callers own no allocator of their own: a plugin running inside a host
// application that has already reserved all device memory for its own pool,
// or a service that forbids any allocation after start-up so that its memory
// footprint stays fixed.  They can pass inputs and outputs they already hold,
// but not a workspace.  This entry point takes its scratch from a fixed array
// in the library's own device memory instead: every GPU that loads the
// library holds DSA_STATIC_SCRATCH_BYTES of it until the process exits.
//
// Host code cannot use the array's name as a device address, so the address
// is looked up once per device with cudaGetSymbolAddress (with that device
// current) and cached.  All calls share the one array and it keeps the last
// call's contents; the status-word header is cleared on the stream at the
// start of every call, and dsa_static_device_status reads (and clears) what
// a call's kernels latched there.  Calls whose work overlaps on the GPU race
// on the array.
#include <mutex>

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_static_scratch[DSA_STATIC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// The array's device address on the current device, looked up once per
// device (with that device current) and cached.
dsa_status_t static_scratch_address(void** out) {
  int dev = 0;
  const cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess) {
    dsa::set_error_detail("cudaGetDevice: %s", cudaGetErrorName(ge));
    return DSA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    dsa::set_error_detail("device ordinal %d: the static scratch serves ordinals below %d",
                          dev, kMaxDevices);
    return DSA_ERR_UNSUPPORTED_SHAPE;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p) {
      dsa::set_error_detail("cudaGetSymbolAddress: %s", cudaGetErrorName(e));
      return DSA_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return DSA_OK;
}

}  // namespace

extern "C" DSA_API dsa_status_t dsa_index_scores_topk_static(
    const dsa_config_t* cfg, const void* q_idx, const void* k_idx, const float* w,
    int32_t* topk_idx, void* stream) {
  size_t need = 0;
  dsa_status_t st = dsa_workspace_size(cfg, DSA_WS_INDEX, &need);
  if (st != DSA_OK) return st;
  if (need > DSA_STATIC_SCRATCH_BYTES) return DSA_ERR_WORKSPACE_TOO_SMALL;
  if (!q_idx || !k_idx || !w || !topk_idx) return DSA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  if ((st = static_scratch_address(&scratch)) != DSA_OK) return st;
  st = dsa_workspace_init(scratch, DSA_STATIC_SCRATCH_BYTES, stream);
  if (st != DSA_OK) return st;
  return dsa_index_scores_topk(cfg, q_idx, k_idx, w, topk_idx, scratch,
                               DSA_STATIC_SCRATCH_BYTES, stream);
}

extern "C" DSA_API dsa_status_t dsa_static_device_status(void* stream,
                                                         uint32_t* device_status) {
  if (!device_status) return DSA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const dsa_status_t st = static_scratch_address(&scratch);
  if (st != DSA_OK) return st;
  return dsa_get_device_status(scratch, stream, device_status);
}
