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
// start of every call.  Calls whose work overlaps on the GPU race on the
// array.
#include <mutex>

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_static_scratch[DSA_STATIC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

extern "C" DSA_API dsa_status_t dsa_index_scores_topk_static(
    const dsa_config_t* cfg, const void* q_idx, const void* k_idx, const float* w,
    int32_t* topk_idx, void* stream) {
  size_t need = 0;
  dsa_status_t st = dsa_workspace_size(cfg, DSA_WS_INDEX, &need);
  if (st != DSA_OK) return st;
  if (need > DSA_STATIC_SCRATCH_BYTES) return DSA_ERR_WORKSPACE_TOO_SMALL;
  if (!q_idx || !k_idx || !w || !topk_idx) return DSA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return DSA_ERR_CUDA;
  void* scratch = nullptr;
  {
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
    scratch = g_scratch_addr[dev];
  }
  st = dsa_workspace_init(scratch, DSA_STATIC_SCRATCH_BYTES, stream);
  if (st != DSA_OK) return st;
  return dsa_index_scores_topk(cfg, q_idx, k_idx, w, topk_idx, scratch,
                               DSA_STATIC_SCRATCH_BYTES, stream);
}
