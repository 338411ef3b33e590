// attn_bwd.cu -- the streaming steps around the sparse attention backward:
// delta = rowsum(dO * O) (the softmax-gradient correction term, "MTraining:
// Efficient Distributed Training for Ultra-Long Contexts via Dynamic Sparse
// Attention", section 3.2), zeroing of the fp32 dK/dV accumulators, and the
// final fp32 -> bf16 rounding of dK/dV.  The main backward is
// attn_bwd_tc.cu.
#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

// ------------------------------------------------------- a7 preprocess
// delta[t,h] = sum_d dO[t,h,d] O[t,h,d] (fp32), one warp per (t,h) row.
__global__ void __launch_bounds__(256) bwd_delta_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dO,
    float* __restrict__ delta, int64_t n_rows, int D, uint32_t* sched) {
  // the backward's work counter restarts at zero every call
  if (blockIdx.x == 0 && threadIdx.x < 2 && sched) sched[threadIdx.x] = 0u;
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t r = w0; r < n_rows; r += nw) {
    const uint4* a = reinterpret_cast<const uint4*>(o + r * D);
    const uint4* b = reinterpret_cast<const uint4*>(dO + r * D);
    float acc = 0.f;
    for (int i = lane; i < D / 8; i += 32) {
      const uint4 x = __ldg(a + i), y = __ldg(b + i);
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc = fmaf(bf16_lo(xs[j]), bf16_lo(ys[j]), acc);
        acc = fmaf(bf16_hi(xs[j]), bf16_hi(ys[j]), acc);
      }
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) delta[r] = acc;
  }
}

__global__ void __launch_bounds__(256) zero_kernel(float4* __restrict__ a, int64_t n4) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x)
    a[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void __launch_bounds__(256) finalize_kernel(const float4* __restrict__ a,
                                                       uint2* __restrict__ out,
                                                       int64_t n4) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 x = __ldg(a + i);
    out[i] = make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
  }
}

int64_t grid_for(const LaunchCtx& c, int64_t n) {
  int64_t g = (n + 255) / 256;
  const int64_t cap = (int64_t)c.num_sms * 8;
  return g < 1 ? 1 : (g > cap ? cap : g);
}

}  // namespace

cudaError_t launch_attn_bwd_delta(const LaunchCtx& c, const AttnShape& s,
                                  const __nv_bfloat16* o, const __nv_bfloat16* dO,
                                  float* delta) {
  const int64_t rows = (s.t_hi - s.t_lo) * s.H;  // the call's query rows
  bwd_delta_kernel<<<(unsigned)grid_for(c, rows * 32), 256, 0, c.stream>>>(
      o, dO, delta, rows, s.D, c.status ? c.status + 32 : nullptr);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_zero(const LaunchCtx& c, const AttnShape& s, float* dk_acc,
                                 float* dv_acc) {
  const int64_t n4 = s.S * s.D / 4;
  zero_kernel<<<(unsigned)grid_for(c, n4), 256, 0, c.stream>>>(
      reinterpret_cast<float4*>(dk_acc), n4);
  if (dv_acc)  // (no second accumulator when K and V are one tensor)
    zero_kernel<<<(unsigned)grid_for(c, n4), 256, 0, c.stream>>>(
        reinterpret_cast<float4*>(dv_acc), n4);
  return cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const LaunchCtx& c, const float* a, __nv_bfloat16* out,
                               int64_t n) {
  const int64_t n4 = n / 4;
  if (n4 == 0) return cudaSuccess;
  finalize_kernel<<<(unsigned)grid_for(c, n4), 256, 0, c.stream>>>(
      reinterpret_cast<const float4*>(a), reinterpret_cast<uint2*>(out), n4);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_finalize(const LaunchCtx& c, const AttnShape& s,
                                     const float* dk_acc, const float* dv_acc,
                                     __nv_bfloat16* dk, __nv_bfloat16* dv) {
  const int64_t n4 = s.S * s.D / 4;
  finalize_kernel<<<(unsigned)grid_for(c, n4), 256, 0, c.stream>>>(
      reinterpret_cast<const float4*>(dk_acc), reinterpret_cast<uint2*>(dk), n4);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !dv_acc) return e;
  finalize_kernel<<<(unsigned)grid_for(c, n4), 256, 0, c.stream>>>(
      reinterpret_cast<const float4*>(dv_acc), reinterpret_cast<uint2*>(dv), n4);
  return cudaGetLastError();
}

}  // namespace dsa
