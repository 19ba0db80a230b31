// Token permutation by expert, with the DeepSeek-v2 device-level drop.
//
// Kept (token, slot) assignments are laid out as one contiguous segment per expert, experts in
// ascending order, rows inside a segment in ascending token order (the dispatch that expert
// parallelism implies: "DeepSeek MoE：从v1到v3的演进", GShard expert parallelism;
// "DeepSeek-V3的Group-Limited Expert Routing与负载均衡优化实践", section 5, all-to-all).
// Deterministic, no atomics-order dependence:
//   1. per 256-token block, a bitmask per expert of the block's tokens that chose it;
//   2. one CTA scans counts over blocks and experts -> segment offsets, per-block bases;
//   3. a token's row = base + number of earlier tokens of its block in the expert's mask;
//   4. one thread per 16-byte chunk of x[t] copies it once to each of the token's rows.
// Drop ("DeepSeek MoE：从v1到v3的演进", DeepSeek-v2 device-level token drop): device d of the G
// virtual devices keeps its C = ceil(T K / G) best assignments by (fp32 weight desc, token asc,
// slot asc). One CTA per device radix-selects the C-th largest 64-bit key
// (weight bits << 32 | ~(t K + k)); an assignment is kept iff its key is >= that threshold.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int PB = 256;  // tokens per permutation block

__device__ __forceinline__ unsigned long long drop_key(float w, long long a) {
  const uint32_t wb = (w > 0.0f) ? __float_as_uint(w) : 0u;  // weights are >= 0
  return (static_cast<unsigned long long>(wb) << 32) |
         static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(a));
}

// One CTA per device: radix select, 8 bits per pass from the top, of the C-th largest key among
// the device's assignments. A first pass over all assignments (loads batched so that many are in
// flight) collects the device's keys into shared memory, up to DROP_SMEM_KEYS of them; each radix
// pass then histograms the keys that match the bits chosen so far, every warp into a histogram
// of its own (no contention between warps), and a parallel suffix scan over the 256 bins picks
// the bin holding the C-th key. A device with more keys than fit streams them from global memory
// on every pass instead (same arithmetic).
constexpr int DROP_THREADS = 1024;
constexpr int DROP_WARPS = DROP_THREADS / 32;
constexpr int DROP_SMEM_KEYS = 20480;  // 160 KB of 64-bit keys
constexpr int DROP_BATCH = 8;          // assignments per thread per load batch

__global__ void __launch_bounds__(DROP_THREADS) drop_threshold_kernel(PermuteArgs p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ unsigned long long skey[];          // [DROP_SMEM_KEYS]
  __shared__ unsigned int whist[DROP_WARPS][256];       // per-warp histograms
  __shared__ unsigned int wsum[8];
  __shared__ unsigned long long s_prefix;
  __shared__ long long s_remaining;
  __shared__ unsigned int s_count;
  const int d = blockIdx.x;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int per = p.N / p.D;
  const long long A = (long long)p.T * p.K;
  const long long C = (A + p.D - 1) / p.D;
  if (threadIdx.x == 0) s_count = 0;
  __syncthreads();
  // ---- collect this device's keys (every lane runs the same number of iterations)
  const long long step = (long long)DROP_THREADS * DROP_BATCH;
  for (long long a0 = 0; a0 < A; a0 += step) {
    int e[DROP_BATCH];
#pragma unroll
    for (int i = 0; i < DROP_BATCH; ++i) {
      const long long a = a0 + (long long)i * DROP_THREADS + threadIdx.x;
      e[i] = a < A ? __ldg(p.idx + a) : -1;
    }
#pragma unroll
    for (int i = 0; i < DROP_BATCH; ++i) {
      const long long a = a0 + (long long)i * DROP_THREADS + threadIdx.x;
      const bool mine = e[i] >= 0 && e[i] / per == d;
      const unsigned int bal = __ballot_sync(FULL_MASK, mine);
      unsigned int base = 0;
      if (lane == 0 && bal != 0u) base = atomicAdd(&s_count, (unsigned int)__popc(bal));
      base = __shfl_sync(FULL_MASK, base, 0);
      if (mine) {
        const unsigned int pos = base + __popc(bal & ((1u << lane) - 1u));
        if (pos < (unsigned int)DROP_SMEM_KEYS) skey[pos] = drop_key(__ldg(p.w + a), a);
      }
    }
  }
  __syncthreads();
  const long long n = s_count;
  if (n <= C) {
    if (threadIdx.x == 0) p.thr[d] = 0ull;  // every key is >= 0: keep all
    return;
  }
  const bool in_smem = n <= DROP_SMEM_KEYS;
  if (threadIdx.x == 0) { s_prefix = 0ull; s_remaining = C; }
  unsigned int* hist = whist[wid];
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    const unsigned long long hi_mask = (pass == 0) ? 0ull : (~0ull << (shift + 8));
    for (int i = threadIdx.x; i < DROP_WARPS * 256; i += DROP_THREADS) (&whist[0][0])[i] = 0;
    __syncthreads();
    const unsigned long long prefix = s_prefix;
    const long long rem = s_remaining;
    if (in_smem) {
      for (long long i = threadIdx.x; i < n; i += DROP_THREADS) {
        const unsigned long long key = skey[i];
        if ((key & hi_mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
    } else {
      for (long long a = threadIdx.x; a < A; a += DROP_THREADS) {
        if (__ldg(p.idx + a) / per != d) continue;
        const unsigned long long key = drop_key(__ldg(p.w + a), a);
        if ((key & hi_mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
    }
    __syncthreads();
    // thread t < 256 takes bin 255 - t (summed over the warps' histograms): an inclusive scan
    // over t gives the keys in bins >= it
    unsigned int v = 0, incl = 0;
    if (threadIdx.x < 256) {
      const int bin = 255 - threadIdx.x;
      for (int w = 0; w < DROP_WARPS; ++w) v += whist[w][bin];
      incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned int x = __shfl_up_sync(FULL_MASK, incl, o);
        if (lane >= o) incl += x;
      }
      if (lane == 31) wsum[wid] = incl;
    }
    __syncthreads();
    if (threadIdx.x < 256) {
      for (int w = 0; w < wid; ++w) incl += wsum[w];
      const long long above = (long long)(incl - v);  // keys in the bins above this one
      if (above < rem && (long long)incl >= rem) {     // the C-th key lies in this bin
        s_prefix = prefix | (static_cast<unsigned long long>(255 - threadIdx.x) << shift);
        s_remaining = rem - above;
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) p.thr[d] = s_prefix;
}

__device__ __forceinline__ bool is_kept(const PermuteArgs& p, long long a, int e) {
  if (!p.capacity_drop) return true;
  const int per = p.N / p.D;
  return drop_key(p.w[a], a) >= p.thr[e / per];
}

__global__ void __launch_bounds__(PB) perm_hist_kernel(PermuteArgs p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t sm[];  // [N][8]
  for (int i = threadIdx.x; i < p.N * 8; i += PB) sm[i] = 0;
  __syncthreads();
  const int t = blockIdx.x * PB + threadIdx.x;
  if (t < p.T) {
    for (int k = 0; k < p.K; ++k) {
      const long long a = (long long)t * p.K + k;
      const int e = p.idx[a];
      if (e < 0 || e >= p.N) { set_error(p.err, ERR_DEVICE_CHECK); continue; }
      if (is_kept(p, a, e)) atomicOr(&sm[e * 8 + (threadIdx.x >> 5)], 1u << (threadIdx.x & 31));
    }
  }
  __syncthreads();
  uint32_t* gm = p.masks + (size_t)blockIdx.x * p.N * 8;
  for (int i = threadIdx.x; i < p.N * 8; i += PB) gm[i] = sm[i];
  for (int e = threadIdx.x; e < p.N; e += PB) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) c += __popc(sm[e * 8 + w]);
    p.cnt[(size_t)blockIdx.x * p.N + e] = c;
  }
}

__global__ void __launch_bounds__(256) perm_scan_kernel(PermuteArgs p, int nb) {
  pdl_wait();
  pdl_trigger();
  __shared__ int wtot[8];
  const int e = threadIdx.x, lane = e & 31, wid = e >> 5;
  // base[b][e]: expert e's rows in the blocks before b (the scatter adds the expert's offset);
  // eight blocks' counts are loaded before they are added
  int running = 0;
  if (e < p.N) {
    for (int b0 = 0; b0 < nb; b0 += 8) {
      int c[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = b0 + i < nb ? p.cnt[(size_t)(b0 + i) * p.N + e] : 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (b0 + i < nb) p.base[(size_t)(b0 + i) * p.N + e] = running;
        running += c[i];
      }
    }
  }
  // exclusive scan of the experts' totals: warp scans, then the warp totals
  int incl = e < p.N ? running : 0;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wtot[wid] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < wid; ++w) before += wtot[w];
  if (e < p.N) p.offsets[e] = before + incl - running;
  if (e == p.N - 1) p.offsets[p.N] = before + incl;
  if (blockIdx.x == 0 && p.sched_zero != nullptr)
    for (int i = e; i < kSchedInts; i += blockDim.x) p.sched_zero[i] = 0;
}

__global__ void __launch_bounds__(PB) perm_scatter_kernel(PermuteArgs p) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x * PB + threadIdx.x;
  if (t >= p.T) return;
  const int wi = threadIdx.x >> 5;
  const uint32_t below = (1u << (threadIdx.x & 31)) - 1u;
  for (int k = 0; k < p.K; ++k) {
    const long long a = (long long)t * p.K + k;
    const int e = p.idx[a];
    if (e < 0 || e >= p.N || !is_kept(p, a, e)) { p.slot_row[a] = -1; continue; }
    const uint32_t* m = p.masks + ((size_t)blockIdx.x * p.N + e) * 8;
    int rank = __popc(m[wi] & below);
    for (int i = 0; i < wi; ++i) rank += __popc(m[i]);
    const int row = p.offsets[e] + p.base[(size_t)blockIdx.x * p.N + e] + rank;
    p.slot_row[a] = row;
    p.row_token[row] = t;
    if (p.row_w != nullptr) p.row_w[row] = p.w[a];
  }
}

// Batches of at most SB_MAX_T tokens: one kernel, SB_CTAS CTAs of one thread per token (at least
// one per expert). Every CTA counts the kept assignments of all experts in shared memory and scans
// the counts (so every CTA knows every segment's offset), then places the assignments of its own
// experts (experts cta * epb .. + epb - 1): a token's rank inside its expert is the number of
// earlier tokens in that expert's bitmask ([epb][W] words, W = ceil(T / 32)). Same arithmetic as
// the three-kernel path above; the work is spread so that no CTA walks a long serial chain.
constexpr int SB_MAX_T = 1024;
constexpr int SB_CTAS = 32;
__global__ void __launch_bounds__(SB_MAX_T) perm_small_kernel(PermuteArgs p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t sm[];  // [epb][W] masks, [N] counts, [N + 1] exclusive offsets
  __shared__ int wsum[SB_MAX_T / 32];
  const int W = (p.T + 31) >> 5;
  const int epb = (p.N + gridDim.x - 1) / gridDim.x;
  const int e0 = blockIdx.x * epb;
  int* cnt = reinterpret_cast<int*>(sm + epb * W);
  int* excl = cnt + p.N;
  for (int i = threadIdx.x; i < epb * W; i += blockDim.x) sm[i] = 0;
  for (int i = threadIdx.x; i < p.N; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int t = threadIdx.x;
  if (t < p.T) {
    for (int k = 0; k < p.K; ++k) {
      const long long a = (long long)t * p.K + k;
      const int e = p.idx[a];
      if (e < 0 || e >= p.N) {
        if (blockIdx.x == 0) set_error(p.err, ERR_DEVICE_CHECK);
        continue;
      }
      if (!is_kept(p, a, e)) continue;
      atomicAdd(&cnt[e], 1);
      if (e >= e0 && e < e0 + epb) atomicOr(&sm[(e - e0) * W + (t >> 5)], 1u << (t & 31));
    }
  }
  __syncthreads();
  {
    // exclusive scan of the per-expert counts (N <= blockDim): warp scans, then warp totals
    const int e = threadIdx.x, lane = e & 31, wi = e >> 5;
    const int c = e < p.N ? cnt[e] : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(FULL_MASK, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[wi] = incl;
    __syncthreads();
    int before = 0;
    for (int i = 0; i < wi; ++i) before += wsum[i];
    if (e < p.N) excl[e] = before + incl - c;
    if (e == p.N - 1) excl[p.N] = before + incl;
    if (blockIdx.x == 0) {
      if (e < p.N) p.offsets[e] = before + incl - c;
      if (e == p.N - 1) p.offsets[p.N] = before + incl;
    }
  }
  if (blockIdx.x == 0 && p.sched_zero != nullptr)
    for (int i = threadIdx.x; i < kSchedInts; i += blockDim.x) p.sched_zero[i] = 0;
  __syncthreads();
  if (t < p.T) {
    const int wi = t >> 5;
    const uint32_t below = (1u << (t & 31)) - 1u;
    for (int k = 0; k < p.K; ++k) {
      const long long a = (long long)t * p.K + k;
      const int e = p.idx[a];
      if (e < 0 || e >= p.N) {
        if (blockIdx.x == 0) p.slot_row[a] = -1;
        continue;
      }
      if (e < e0 || e >= e0 + epb) continue;  // another CTA's expert
      if (!is_kept(p, a, e)) { p.slot_row[a] = -1; continue; }
      const uint32_t* m = sm + (e - e0) * W;
      int rank = __popc(m[wi] & below);
      for (int i = 0; i < wi; ++i) rank += __popc(m[i]);
      const int row = excl[e] + rank;
      p.slot_row[a] = row;
      p.row_token[row] = t;
      if (p.row_w != nullptr) p.row_w[row] = p.w[a];
    }
  }
}

// One thread per 16-byte chunk of a token's row: read it once, write it to each kept row of
// the token. Consecutive threads take consecutive chunks of a row, so every warp reads and
// writes contiguous runs; a batch of a few tokens still spreads over the whole GPU.
__global__ void __launch_bounds__(256) dispatch_rows_kernel(PermuteArgs p) {
  pdl_wait();
  pdl_trigger();
  const size_t row_bytes = (size_t)p.H * p.elem_bytes;
  const int chunks = (int)(row_bytes / 16);
  const size_t n = (size_t)p.T * chunks;
  const char* src = static_cast<const char*>(p.x);
  char* dst = static_cast<char*>(p.x_perm);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / chunks);
    const int c = (int)(i - (size_t)t * chunks);
    const uint4 v = ld_nc_v4(src + (size_t)t * row_bytes + (size_t)c * 16);
    const int32_t* sr = p.slot_row + (size_t)t * p.K;
    for (int k = 0; k < p.K; ++k) {
      const int r = __ldg(sr + k);
      if (kChecks && (r < -1 || r >= p.T * p.K)) {
        set_error(p.err, ERR_DEVICE_CHECK);  // not a row of x_perm: skip it
        continue;
      }
      if (r >= 0) st_v4(dst + (size_t)r * row_bytes + (size_t)c * 16, v);
    }
  }
}

}  // namespace

int permute_blocks(int T) { return (T + PB - 1) / PB; }

cudaError_t launch_permute(const PermuteArgs& p, int num_sms, cudaStream_t st) {
  if (p.T <= 0) {
    // no tokens: empty segments
    return cudaMemsetAsync(p.offsets, 0, sizeof(int32_t) * (p.N + 1), st);
  }
  const int nb = permute_blocks(p.T);
  if (p.capacity_drop) {
    static bool smem_set[64] = {false};  // the attribute is set once per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !smem_set[dev]) {
      const cudaError_t ea = cudaFuncSetAttribute(
          drop_threshold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
          (int)(DROP_SMEM_KEYS * sizeof(unsigned long long)));
      if (ea != cudaSuccess) return ea;
      if (dev >= 0 && dev < 64) smem_set[dev] = true;
    }
    const cudaError_t e = launch_pdl(drop_threshold_kernel, dim3(p.D), dim3(DROP_THREADS),
                                     DROP_SMEM_KEYS * sizeof(unsigned long long), st, p);
    if (e != cudaSuccess) return e;
  }
  if (p.T <= SB_MAX_T) {
    const int W = (p.T + 31) / 32;
    int threads = ((p.T + 31) / 32) * 32;
    if (threads < p.N) threads = ((p.N + 31) / 32) * 32;
    const int ctas = p.N < SB_CTAS ? p.N : SB_CTAS;
    const int epb = (p.N + ctas - 1) / ctas;
    return launch_pdl(perm_small_kernel, dim3(ctas), dim3(threads),
                      (size_t)(epb * W + 2 * p.N + 1) * sizeof(uint32_t), st, p);
  }
  cudaError_t e = launch_pdl(perm_hist_kernel, dim3(nb), dim3(PB), p.N * 8 * sizeof(uint32_t), st, p);
  if (e == cudaSuccess) e = launch_pdl(perm_scan_kernel, dim3(1), dim3(256), 0, st, p, nb);
  if (e == cudaSuccess) e = launch_pdl(perm_scatter_kernel, dim3(nb), dim3(PB), 0, st, p);
  return e;
}

cudaError_t launch_dispatch(const PermuteArgs& p, int num_sms, cudaStream_t st) {
  if (p.T <= 0 || p.x == nullptr || p.x_perm == nullptr) return cudaSuccess;
  const size_t n = (size_t)p.T * ((size_t)p.H * p.elem_bytes / 16);
  size_t blocks = (n + 255) / 256;
  if (blocks > (size_t)num_sms * 16) blocks = (size_t)num_sms * 16;
  return launch_pdl(dispatch_rows_kernel, dim3((int)blocks), dim3(256), 0, st, p);
}

}  // namespace moe
