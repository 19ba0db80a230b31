// Weighted combine back to token order plus the shared experts' output
// ("从零构建DeepSeekMoE", section 2.2 forward: shared experts' sum + routed output):
//   out[t] = sum_k [slot_row(t,k) >= 0] w[t,k] * y[slot_row(t,k)] + y_shared[t]
// One warp per token, fp32 accumulation in slot order. Each lane owns 16-byte chunks of the
// row; for two chunks at a time it issues the loads of all K contributing rows (and the shared
// row) before the first FMA, so 2 (K + 1) independent loads are in flight per lane. A dropped
// slot (row -1) is not read and adds nothing.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

// acc = sum_k w[k] * v[k] (slot order, fp32) + shared row
template <typename T, int KM>
__device__ __forceinline__ const float* weighted_sum_impl(const uint4 (&v)[KM],
                                                          const float (&w)[KM], int K,
                                                          const uint4& vs, float* acc) {
  constexpr int V = Vec<T>::N;
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.0f;
#pragma unroll
  for (int k = 0; k < KM; ++k) {
    if (k < K) {
      float f[V];
      Vec<T>::unpack(v[k], f);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(w[k], f[i], acc[i]);
    }
  }
  float f[V];
  Vec<T>::unpack(vs, f);
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] += f[i];
  return acc;
}

template <typename T>
struct Acc {
  float a[Vec<T>::N];
};

template <typename T, int KM>
__device__ __forceinline__ Acc<T> weighted_sum(const uint4 (&v)[KM], const float (&w)[KM], int K,
                                               const uint4& vs) {
  Acc<T> r;
  weighted_sum_impl<T, KM>(v, w, K, vs, r.a);
  return r;
}

template <typename T, int KC>  // KC = top_k (compile time), or 0 for any K <= 16
__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
  constexpr int V = Vec<T>::N;
  constexpr int KM = KC > 0 ? KC : 16;
  const int K = KC > 0 ? KC : a.K;
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int chunks = a.H / V;
  const T* y = static_cast<const T*>(a.y);
  const T* ys = static_cast<const T*>(a.ys);
  T* out = static_cast<T*>(a.out);
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < a.T; t += warps) {
    const int my_row = lane < K ? a.slot_row[(size_t)t * K + lane] : -1;
    const float my_w = lane < K ? a.w[(size_t)t * K + lane] : 0.0f;
    const T* src[KM];
    float ws[KM];
    uint32_t live = 0;
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      const int r = __shfl_sync(FULL_MASK, my_row, k);
      const float wk = __shfl_sync(FULL_MASK, my_w, k);
      const bool on = k < K && r >= 0;
      live |= (on ? 1u : 0u) << k;
      src[k] = y + (size_t)(on ? r : 0) * a.H;
      ws[k] = on ? wk : 0.0f;
    }
    const T* srow = ys != nullptr ? ys + (size_t)t * a.H : nullptr;
    T* orow = out + (size_t)t * a.H;
    // two chunks per lane and iteration: 2 (K + 1) independent 16-byte loads in flight
    for (int c0 = lane; c0 < chunks; c0 += 64) {
      const int c1 = c0 + 32;
      const bool two = c1 < chunks;
      uint4 v0[KM], v1[KM];
#pragma unroll
      for (int k = 0; k < KM; ++k) {
        if (k < K) {
          const bool on = (live >> k) & 1u;
          v0[k] = on ? ld_nc_v4(src[k] + (size_t)c0 * V) : make_uint4(0u, 0u, 0u, 0u);
          v1[k] = (on && two) ? ld_nc_v4(src[k] + (size_t)c1 * V) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      uint4 s0 = make_uint4(0u, 0u, 0u, 0u), s1 = s0;
      if (srow != nullptr) {
        s0 = ld_nc_v4(srow + (size_t)c0 * V);
        if (two) s1 = ld_nc_v4(srow + (size_t)c1 * V);
      }
      st_v4(orow + (size_t)c0 * V, Vec<T>::pack(weighted_sum<T, KM>(v0, ws, K, s0).a));
      if (two) st_v4(orow + (size_t)c1 * V, Vec<T>::pack(weighted_sum<T, KM>(v1, ws, K, s1).a));
    }
  }
}

template <typename T>
void launch_typed(const CombineArgs& a, int blocks, cudaStream_t st) {
  switch (a.K) {
    case 4: combine_kernel<T, 4><<<blocks, 256, 0, st>>>(a); break;
    case 6: combine_kernel<T, 6><<<blocks, 256, 0, st>>>(a); break;
    case 8: combine_kernel<T, 8><<<blocks, 256, 0, st>>>(a); break;
    default: combine_kernel<T, 0><<<blocks, 256, 0, st>>>(a); break;
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, int num_sms, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  int blocks = (a.T + 7) / 8;
  if (blocks > num_sms * 16) blocks = num_sms * 16;
  if (a.dtype == 1)
    launch_typed<__nv_bfloat16>(a, blocks, st);
  else
    launch_typed<float>(a, blocks, st);
  return cudaGetLastError();
}

}  // namespace moe
