// fp32 grouped GEMMs on CUDA cores (the MOE_F32 path: small layers held to 1e-5).
//   MODE_GATE: u[t, e]  = x[t] . W_g[e] + gate_bias[e]                       (router linear)
//   MODE_UP:   h[r, j]  = silu(A[r] . W13_p[j]) * (A[r] . W13_p[I + j])       (SwiGLU up)
//   MODE_DOWN: y[r, o]  = h[r] . W2_p[o]                                      (down projection)
// A problem p < n_routed is expert p's segment rows offsets[p] .. offsets[p+1]-1 of the routed
// tensors; p == n_routed is the shared experts over all T rows, stacked so that S shared
// experts act as one expert of intermediate size S*I ("从零构建DeepSeekMoE", section 2.2:
// shared experts always active, their outputs summed).
// 64x64 output tile per 256-thread block, 4x4 per thread, K staged 16 at a time in shared
// memory. Accumulation order is plain ascending k in fp32.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int TM = 64, TN = 64, TK = 16;

struct Prob {
  int row0, rows, shared;
};

__device__ __forceinline__ Prob get_prob(const GemmArgs& a, int p) {
  Prob q;
  if (a.mode == MODE_GATE) { q.row0 = 0; q.rows = a.T; q.shared = 0; return q; }
  if (p < a.n_routed) {
    q.row0 = a.offsets[p];
    q.rows = a.offsets[p + 1] - q.row0;
    q.shared = 0;
  } else {
    q.row0 = 0; q.rows = a.T; q.shared = 1;
  }
  return q;
}

// Weight element W(o, k) of problem p for output column o and reduction index k.
__device__ __forceinline__ float wval(const GemmArgs& a, int p, bool shared, int o, int k,
                                      bool up_half) {
  const float* b0 = static_cast<const float*>(a.b0);
  const float* b1 = static_cast<const float*>(a.b1);
  const size_t H = a.H, I = a.I;
  if (a.mode == MODE_GATE) return b0[(size_t)o * H + k];
  if (a.mode == MODE_UP) {
    if (!shared) return b0[((size_t)p * 2 * I + (up_half ? I : 0) + o) * H + k];
    const size_t s = o / I, j = o % I;
    return b1[(s * 2 * I + (up_half ? I : 0) + j) * H + k];
  }
  // MODE_DOWN
  if (!shared) return b0[((size_t)p * H + o) * I + k];
  const size_t s = k / I, kk = k % I;
  return b1[(s * H + o) * I + kk];
}

__global__ void __launch_bounds__(256) simt_gemm_kernel(GemmArgs a) {
  pdl_wait();
  pdl_trigger();
  const int p = blockIdx.z;
  Prob q = get_prob(a, p);
  if (kChecks && a.mode != MODE_GATE && p < a.n_routed &&
      (q.row0 < 0 || q.rows < 0 || q.row0 + q.rows > a.rows_cap)) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) set_error(a.err, ERR_DEVICE_CHECK);
    return;  // a segment outside the rows: skip the problem
  }
  const int m0 = blockIdx.y * TM;
  if (m0 >= q.rows) return;
  const bool up = a.mode == MODE_UP;
  int ncols, kdim, lda;
  const float* A;
  if (a.mode == MODE_GATE) { ncols = a.N; kdim = a.H; lda = a.H; A = (const float*)a.a0; }
  else if (up) {
    ncols = q.shared ? a.S * a.I : a.I; kdim = a.H; lda = a.H;
    A = (const float*)(q.shared ? a.a1 : a.a0);
  } else {
    ncols = a.H; kdim = q.shared ? a.S * a.I : a.I; lda = kdim;
    A = (const float*)(q.shared ? a.a1 : a.a0);
  }
  const int n0 = blockIdx.x * TN;
  if (n0 >= ncols) return;

  __shared__ float As[TK][TM + 1];
  __shared__ float Bs[TK][TN + 1];
  __shared__ float Us[TK][TN + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4], accu[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) { acc[i][j] = 0.0f; accu[i][j] = 0.0f; }

  for (int k0 = 0; k0 < kdim; k0 += TK) {
    for (int i = threadIdx.x; i < TK * TM; i += 256) {
      const int r = i / TK, kk = i % TK;
      const int gr = m0 + r, gk = k0 + kk;
      As[kk][r] = (gr < q.rows && gk < kdim) ? A[(size_t)(q.row0 + gr) * lda + gk] : 0.0f;
    }
    for (int i = threadIdx.x; i < TK * TN; i += 256) {
      const int c = i / TK, kk = i % TK;
      const int gc = n0 + c, gk = k0 + kk;
      const bool ok = gc < ncols && gk < kdim;
      Bs[kk][c] = ok ? wval(a, p, q.shared, gc, gk, false) : 0.0f;
      if (up) Us[kk][c] = ok ? wval(a, p, q.shared, gc, gk, true) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float av[4], bv[4], uv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) { bv[j] = Bs[kk][tx * 4 + j]; uv[j] = up ? Us[kk][tx * 4 + j] : 0.f; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
          if (up) accu[i][j] = fmaf(av[i], uv[j], accu[i][j]);
        }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = m0 + ty * 4 + i;
    if (r >= q.rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = n0 + tx * 4 + j;
      if (c >= ncols) continue;
      if (a.mode == MODE_GATE) {
        float v = acc[i][j] + (a.gate_bias ? a.gate_bias[c] : 0.0f);
        static_cast<float*>(a.out0)[(size_t)r * a.N + c] = v;
      } else if (up) {
        const float g = acc[i][j];
        const float h = g / (1.0f + expf(-g)) * accu[i][j];
        float* o = static_cast<float*>(q.shared ? a.out1 : a.out0);
        o[(size_t)(q.row0 + r) * ncols + c] = h;
      } else {
        float* o = static_cast<float*>(q.shared ? a.out1 : a.out0);
        o[(size_t)(q.row0 + r) * a.H + c] = acc[i][j];
      }
    }
  }
}

}  // namespace

cudaError_t launch_gemm_simt(const GemmArgs& a, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  int ncols_max, probs;
  if (a.mode == MODE_GATE) { ncols_max = a.N; probs = 1; }
  else {
    probs = a.n_routed + (a.has_shared ? 1 : 0);
    if (a.mode == MODE_UP) ncols_max = (a.has_shared ? a.S : 1) * a.I;
    else ncols_max = a.H;
    if (a.mode == MODE_UP && a.I > ncols_max) ncols_max = a.I;
  }
  if (probs == 0) return cudaSuccess;
  // routed rows of one expert never exceed T (a token picks an expert at most once)
  dim3 grid((ncols_max + TN - 1) / TN, (a.T + TM - 1) / TM, probs);
  return launch_pdl(simt_gemm_kernel, grid, dim3(256), 0, st, a);
}

}  // namespace moe
