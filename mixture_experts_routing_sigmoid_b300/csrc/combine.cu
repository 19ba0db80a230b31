// Weighted combine back to token order plus the shared experts' output
// ("从零构建DeepSeekMoE", section 2.2 forward: shared experts' sum + routed output):
//   out[t] = sum_k [slot_row(t,k) >= 0] w[t,k] * y[slot_row(t,k)] + y_shared[t]
// One warp per token, 16-byte loads of every contributing row, fp32 accumulation in slot order.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

template <typename T>
__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
  constexpr int V = Vec<T>::N;
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int chunks = a.H / V;
  const T* y = static_cast<const T*>(a.y);
  const T* ys = static_cast<const T*>(a.ys);
  T* out = static_cast<T*>(a.out);
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < a.T; t += warps) {
    const int my_row = lane < a.K ? a.slot_row[(size_t)t * a.K + lane] : -1;
    const float my_w = lane < a.K ? a.w[(size_t)t * a.K + lane] : 0.0f;
    int rows[16];
    float ws[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      rows[k] = __shfl_sync(FULL_MASK, my_row, k);
      ws[k] = __shfl_sync(FULL_MASK, my_w, k);
    }
    for (int c = lane; c < chunks; c += 32) {
      float acc[V];
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = 0.0f;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        if (k < a.K && rows[k] >= 0) {
          float v[V];
          Vec<T>::unpack(ld_nc_v4(y + (size_t)rows[k] * a.H + (size_t)c * V), v);
#pragma unroll
          for (int i = 0; i < V; ++i) acc[i] = fmaf(ws[k], v[i], acc[i]);
        }
      }
      if (ys != nullptr) {
        float v[V];
        Vec<T>::unpack(ld_nc_v4(ys + (size_t)t * a.H + (size_t)c * V), v);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] += v[i];
      }
      st_v4(out + (size_t)t * a.H + (size_t)c * V, Vec<T>::pack(acc));
    }
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, int num_sms, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  int blocks = (a.T + 7) / 8;
  if (blocks > num_sms * 16) blocks = num_sms * 16;
  if (a.dtype == 1)
    combine_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(a);
  else
    combine_kernel<float><<<blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
