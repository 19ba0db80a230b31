// Load balancing from the batch's expert counts and scores.
//
// Auxiliary-loss-free bias update ("DeepSeek MoE：从v1到v3的演进", DeepSeek-v3, 无辅助损失负载
// 均衡): every expert's selection bias moves by a constant rate u against its load,
//   e_i = c_bar - c_i,  b_i <- b_i + u * sign(e_i),  c_bar = mean_j c_j.
// The sign is decided exactly in integers: sign(c_bar - c_i) = sign(sum_j c_j - N c_i). The
// update is one fp32 addition per expert (the bias is kept in fp32).
//
// Sequence-wise balance loss (same page, DeepSeek-v3, sequence粒度的负载均衡loss): the
// expert-level balance loss of the ST-MoE section computed within each sequence of the batch
// and averaged over sequences (the page prints no formula; this is the plain reading):
//   L_b = N sum_e f_e^b P_e^b,  f_e^b = c_e^b / (L K),  P_e^b = sum_{t in b} s_te / sum_{t in b} sum_j s_tj
//   L_seq = (1/B) sum_b L_b,  B = T / L sequences of L consecutive tokens.
// Three launches: per (sequence, chunk of 64+ tokens) partial score sums (fp32, warp per token)
// and counts; per sequence a fixed-order fp64 reduction of its chunks; the mean over sequences.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

__global__ void __launch_bounds__(256) bias_update_kernel(BiasUpdateArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ long long part[8];
  long long s = 0;
  for (int e = threadIdx.x; e < a.N; e += blockDim.x) s += a.counts[e];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(FULL_MASK, s, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
  __syncthreads();
  long long total = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) total += part[w];
  for (int e = threadIdx.x; e < a.N; e += blockDim.x) {
    const long long d = total - (long long)a.N * a.counts[e];  // N (c_bar - c_e)
    const float step = d > 0 ? a.rate : (d < 0 ? -a.rate : 0.0f);
    a.bias[e] = a.bias[e] + step;
  }
}

constexpr int MAXJ = 8;  // experts per lane (N <= 256)

__global__ void __launch_bounds__(256) seq_partial_kernel(SeqLossArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[8][256];
  __shared__ int cnt[256];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int b = blockIdx.x, ch = blockIdx.y;
  const int J = (a.N + 31) >> 5;
  const int per = (a.L + a.cps - 1) / a.cps;
  const int t_begin = b * a.L + ch * per;
  const int t_end = min(b * a.L + a.L, t_begin + per);
  for (int e = threadIdx.x; e < 256; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  float acc[MAXJ];
#pragma unroll
  for (int j = 0; j < MAXJ; ++j) acc[j] = 0.0f;
  for (int t = t_begin + wid; t < t_end; t += 8) {
    const float* ut = a.u + (size_t)t * a.N;
    float u[MAXJ];
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) {
      const int e = j * 32 + lane;
      u[j] = (j < J && e < a.N) ? ut[e] : -INFINITY;
    }
    if (a.score_fn == 1) {
#pragma unroll
      for (int j = 0; j < MAXJ; ++j)
        if (j < J && j * 32 + lane < a.N) acc[j] += 1.0f / (1.0f + expf(-u[j]));
    } else {
      float m = u[0];
#pragma unroll
      for (int j = 1; j < MAXJ; ++j) m = fmaxf(m, u[j]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL_MASK, m, o));
      float ex[MAXJ], z = 0.0f;
#pragma unroll
      for (int j = 0; j < MAXJ; ++j) { ex[j] = expf(u[j] - m); z += ex[j]; }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(FULL_MASK, z, o);
#pragma unroll
      for (int j = 0; j < MAXJ; ++j) acc[j] += ex[j] / z;
    }
    if (lane < a.K) {
      const int e = a.idx[(size_t)t * a.K + lane];
      if (e >= 0 && e < a.N) atomicAdd(&cnt[e], 1);
      else set_error(a.err, ERR_DEVICE_CHECK);
    }
  }
#pragma unroll
  for (int j = 0; j < MAXJ; ++j) {
    const int e = j * 32 + lane;
    if (e < 256) red[wid][e] = (j < J && e < a.N) ? acc[j] : 0.0f;
  }
  __syncthreads();
  const size_t row = (size_t)(b * a.cps + ch) * a.N;
  for (int e = threadIdx.x; e < a.N; e += blockDim.x) {
    float sum = 0.0f;
    for (int w = 0; w < 8; ++w) sum += red[w][e];
    a.part_s[row + e] = sum;
    a.part_c[row + e] = cnt[e];
  }
}

__global__ void __launch_bounds__(256) seq_final_kernel(SeqLossArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ double colsum[256];
  __shared__ double fp[256];
  const int b = blockIdx.x, e = threadIdx.x;
  double cs = 0.0;
  long long c = 0;
  if (e < a.N)
    for (int ch = 0; ch < a.cps; ++ch) {
      const size_t row = (size_t)(b * a.cps + ch) * a.N;
      cs += (double)a.part_s[row + e];
      c += a.part_c[row + e];
    }
  colsum[e] = cs;
  __syncthreads();
  if (e == 0) {
    double tot = 0.0;
    for (int i = 0; i < a.N; ++i) tot += colsum[i];
    fp[0] = tot;
  }
  __syncthreads();
  const double total = fp[0];
  __syncthreads();
  fp[e] = (e < a.N) ? ((double)c / ((double)a.L * a.K)) * (colsum[e] / total) : 0.0;
  __syncthreads();
  if (e == 0) {
    double lb = 0.0;
    for (int i = 0; i < a.N; ++i) lb += fp[i];
    lb *= a.N;
    a.seq_lb[b] = lb;
    if (a.per_seq) a.per_seq[b] = (float)lb;
  }
}

__global__ void seq_mean_kernel(SeqLossArgs a) {
  pdl_wait();
  pdl_trigger();
  double s = 0.0;
  for (int b = 0; b < a.B; ++b) s += a.seq_lb[b];
  a.mean[0] = (float)(s / a.B);
}

}  // namespace

int seq_loss_chunks(int L) {
  int c = (L + 63) / 64;
  return c < 1 ? 1 : (c > 64 ? 64 : c);
}

cudaError_t launch_seq_loss(const SeqLossArgs& a, cudaStream_t st) {
  if (a.B <= 0) return cudaSuccess;
  cudaError_t e = launch_pdl(seq_partial_kernel, dim3(a.B, a.cps), dim3(256), 0, st, a);
  if (e == cudaSuccess) e = launch_pdl(seq_final_kernel, dim3(a.B), dim3(256), 0, st, a);
  if (e == cudaSuccess) e = launch_pdl(seq_mean_kernel, dim3(1), dim3(1), 0, st, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_bias_update(const BiasUpdateArgs& a, cudaStream_t st) {
  return launch_pdl(bias_update_kernel, dim3(1), dim3(256), 0, st, a);
}

}  // namespace moe
