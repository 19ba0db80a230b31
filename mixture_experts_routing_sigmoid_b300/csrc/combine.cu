// Weighted combine back to token order plus the shared experts' output
// ("从零构建DeepSeekMoE", section 2.2 forward: shared experts' sum + routed output):
//   out[t] = sum_k [slot_row(t,k) >= 0] w[t,k] * y[slot_row(t,k)] + y_shared[t]
// One thread per 16-byte chunk of an output row: it issues the loads of all K contributing
// rows' chunks (and the shared row's) before the first FMA, then accumulates in fp32 in slot
// order. Consecutive threads take consecutive chunks of a row, so each warp reads contiguous
// runs of every source row; a few-token batch still spreads over the whole GPU. A dropped
// slot (row -1) is not read and adds nothing.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

template <typename T, int KC>  // KC = top_k (compile time), or 0 for any K <= 16
__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
  pdl_wait();
  pdl_trigger();
  constexpr int V = Vec<T>::N;
  constexpr int KM = KC > 0 ? KC : 16;
  const int K = KC > 0 ? KC : a.K;
  const int chunks = a.H / V;
  const size_t n = (size_t)a.T * chunks;
  const T* y = static_cast<const T*>(a.y);
  const T* ys = static_cast<const T*>(a.ys);
  T* out = static_cast<T*>(a.out);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / chunks);
    const int c = (int)(i - (size_t)t * chunks);
    // row indices and weights first, then every row load, then the arithmetic
    int r[KM];
    float wk[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      r[k] = k < K ? __ldg(a.slot_row + (size_t)t * K + k) : -1;
      if (kChecks && (r[k] < -1 || r[k] >= a.rows)) {
        set_error(a.err, ERR_DEVICE_CHECK);  // not a row of y: skip it
        r[k] = -1;
      }
      wk[k] = k < K ? __ldg(a.w + (size_t)t * K + k) : 0.0f;
    }
    uint4 v[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      const uint4* src = reinterpret_cast<const uint4*>(y + (size_t)max(r[k], 0) * a.H) + c;
      v[k] = r[k] >= 0 ? __ldg(src) : make_uint4(0u, 0u, 0u, 0u);
    }
    const uint4 vs = ys != nullptr
                         ? __ldg(reinterpret_cast<const uint4*>(ys + (size_t)t * a.H) + c)
                         : make_uint4(0u, 0u, 0u, 0u);
    float acc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = 0.0f;
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      if (k < K && r[k] >= 0) {
        float f[V];
        Vec<T>::unpack(v[k], f);
#pragma unroll
        for (int j = 0; j < V; ++j) acc[j] = fmaf(wk[k], f[j], acc[j]);
      }
    }
    if (ys != nullptr) {
      float f[V];
      Vec<T>::unpack(vs, f);
#pragma unroll
      for (int j = 0; j < V; ++j) acc[j] += f[j];
    }
    st_v4(out + (size_t)t * a.H + (size_t)c * V, Vec<T>::pack(acc));
  }
}

template <typename T>
cudaError_t launch_typed(const CombineArgs& a, int blocks, cudaStream_t st) {
  switch (a.K) {
    case 4: return launch_pdl(combine_kernel<T, 4>, dim3(blocks), dim3(256), 0, st, a);
    case 6: return launch_pdl(combine_kernel<T, 6>, dim3(blocks), dim3(256), 0, st, a);
    case 8: return launch_pdl(combine_kernel<T, 8>, dim3(blocks), dim3(256), 0, st, a);
    default: return launch_pdl(combine_kernel<T, 0>, dim3(blocks), dim3(256), 0, st, a);
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, int num_sms, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  const int V = a.dtype == 1 ? 8 : 4;
  const size_t n = (size_t)a.T * (a.H / V);
  size_t blocks = (n + 255) / 256;
  if (blocks > (size_t)num_sms * 16) blocks = (size_t)num_sms * 16;
  return a.dtype == 1 ? launch_typed<__nv_bfloat16>(a, (int)blocks, st)
                      : launch_typed<float>(a, (int)blocks, st);
}

}  // namespace moe
