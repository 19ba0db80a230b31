// bf16 grouped GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
//   MODE_GATE: u[t, e] = x[t] . W_g[e] + gate_bias[e]  (fp32 out; router linear layer,
//              "从零构建DeepSeekMoE", section 5.2)
//   MODE_UP:   h[r, j] = silu(A[r] . W13_p[j]) * (A[r] . W13_p[I + j])   (bf16 out)
//   MODE_DOWN: y[r, o] = h[r] . W2_p[o]                                   (bf16 out)
// Problem p < n_routed is expert p's segment (rows offsets[p] .. offsets[p+1]-1, read on the
// device); p == n_routed is the shared experts over all T tokens, with S shared experts
// stacked into one of intermediate size S*I ("DeepSeek MoE：从v1到v3的演进", DeepSeek-v1
// fine-grained experts and shared-expert isolation).
//
// Persistent kernel, one 192-thread CTA per SM, static round-robin over output tiles of
// 128 rows x 256 columns (UP: 128 gate + 128 up columns of the same 128 intermediate
// features, so the SwiGLU is applied in the epilogue). Tiles run problem by problem, weight
// tile by weight tile, row tile fastest, so CTAs that run together share weight tiles in L2.
//   warp 0      TMA producer: A tile [128 x 64] and B tile [256 x 64] per stage, 128-byte
//               swizzle, 4-stage ring of 48 KB stages guarded by full/empty mbarriers.
//   warp 1      TMEM owner and MMA issuer: one thread issues 4 tcgen05.mma (M=128, N=256,
//               K=16) per stage into one of two 256-column fp32 accumulators, commits the
//               stage back to the producer and the finished accumulator to the epilogue.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes
//               32*(w%4)..+31 = tile rows), SwiGLU / bias, row-predicated 16-byte stores.
// Rows of a tile past the segment end belong to the next expert (or lie beyond the tensor,
// where TMA fills zeros); they are computed and never stored. Every mbarrier wait is bounded:
// on timeout the CTA raises an abort flag and the device error word, drains, frees TMEM and
// returns.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int MAXP = 258;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
constexpr unsigned long long TIMEOUT_NS = 2000000000ull;    // 2 s per wait
constexpr unsigned long long GRACE_NS = 100000000ull;       // drain after an abort

struct TcParams {
  CUtensorMap tmA0, tmA1, tmB0, tmB1;
  const int32_t* offsets;
  int n_routed, has_shared, T, H, I, S, N;
  void* out0;
  void* out1;
  const float* gate_bias;
  int* err;
};

struct SmemCtl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int nprob;
  int total_tiles;
  int tile_start[MAXP + 1];
  int row0[MAXP];
  int rows[MAXP];
};

constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + sizeof(SmemCtl);

template <int MODE>
__device__ __forceinline__ int n_tiles_of(const TcParams& p, bool shared) {
  if (MODE == MODE_UP) return (shared ? p.S * p.I : p.I) / 128;
  if (MODE == MODE_DOWN) return (p.H + BN - 1) / BN;
  return 1;
}
template <int MODE>
__device__ __forceinline__ int k_blocks_of(const TcParams& p, bool shared) {
  if (MODE == MODE_DOWN) return (shared ? p.S * p.I : p.I) / BK;
  return p.H / BK;
}

struct Tile {
  int prob, m0, n0, row0, rows, kb;
  bool shared;
};

template <int MODE>
__device__ __forceinline__ Tile decode_tile(const TcParams& p, const SmemCtl& c, int tile) {
  int lo = 0, hi = c.nprob - 1;  // largest q with tile_start[q] <= tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (c.tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  Tile t;
  t.prob = lo;
  t.shared = (MODE != MODE_GATE) && lo >= p.n_routed;
  t.row0 = c.row0[lo];
  t.rows = c.rows[lo];
  const int mt = (t.rows + BM - 1) / BM;
  const int local = tile - c.tile_start[lo];
  const int n = local / mt;
  const int m = local - n * mt;
  t.m0 = m * BM;
  t.n0 = (MODE == MODE_UP) ? n * 128 : n * BN;
  t.kb = k_blocks_of<MODE>(p, t.shared);
  return t;
}

__device__ __forceinline__ void grace_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > GRACE_NS) break;
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return g / (1.0f + __expf(-g)) * u;
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms want 1 KB alignment
  uint8_t* sgen = smem_raw + (sbase - raw);
  SmemCtl& c = *reinterpret_cast<SmemCtl*>(sgen + (size_t)STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  auto bar = [](const uint64_t& b) { return smem_u32(&b); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(bar(c.full[s]), 1); mbar_init(bar(c.empty[s]), 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(bar(c.tfull[a]), 1); mbar_init(bar(c.tempty[a]), 4); }
    mbar_init(bar(c.drain), 1);
    c.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(&c.tmem_base), TMEM_COLS);

  // ---- problem table and tile prefix (tile counts depend on device-resident offsets)
  const int nprob = (MODE == MODE_GATE) ? 1 : p.n_routed + p.has_shared;
  for (int q = threadIdx.x; q < nprob; q += THREADS) {
    if (MODE != MODE_GATE && q < p.n_routed) {
      const int r0 = p.offsets[q];
      c.row0[q] = r0;
      c.rows[q] = p.offsets[q + 1] - r0;
    } else {
      c.row0[q] = 0;
      c.rows[q] = p.T;
    }
  }
  __syncthreads();
  if (warp == 0) {
    int run = 0;
    for (int b = 0; b < nprob; b += 32) {
      const int q = b + lane;
      int cnt = 0;
      if (q < nprob) {
        const bool sh = (MODE != MODE_GATE) && q >= p.n_routed;
        const int rows = c.rows[q] > 0 ? c.rows[q] : 0;
        cnt = ((rows + BM - 1) / BM) * n_tiles_of<MODE>(p, sh);
      }
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(FULL_MASK, incl, o);
        if (lane >= o) incl += v;
      }
      if (q < nprob) c.tile_start[q] = run + incl - cnt;
      run += __shfl_sync(FULL_MASK, incl, 31);
    }
    if (lane == 0) { c.tile_start[nprob] = run; c.total_tiles = run; c.nprob = nprob; }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = c.tmem_base;
  const int total = c.total_tiles;
  volatile int* abort_flag = &c.abort_flag;

  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.tmA0);
      tma_prefetch_desc(&p.tmB0);
      if (MODE != MODE_GATE && p.has_shared) { tma_prefetch_desc(&p.tmA1); tma_prefetch_desc(&p.tmB1); }
    }
    uint32_t stage = 0, phase = 0;
    uint32_t issued_mask = 0, last_parity = 0;  // per stage: issued at least once / its parity
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const Tile t = decode_tile<MODE>(p, c, tile);
      for (int kb = 0; kb < t.kb; ++kb) {
        if (!warp_wait_bounded(bar(c.empty[stage]), phase ^ 1u, abort_flag, p.err, TIMEOUT_NS)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t fb = bar(c.full[stage]);
          mbar_expect_tx(fb, STAGE_BYTES);
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          const int k0 = kb * BK;
          tma_load_2d(sa, t.shared ? &p.tmA1 : &p.tmA0, fb, k0, t.row0 + t.m0);
          if (MODE == MODE_UP) {
            int yg;
            if (!t.shared) yg = t.prob * 2 * p.I + t.n0;
            else yg = (t.n0 / p.I) * 2 * p.I + (t.n0 % p.I);
            const CUtensorMap* tb = t.shared ? &p.tmB1 : &p.tmB0;
            tma_load_2d(sb, tb, fb, k0, yg);                  // gate projection rows
            tma_load_2d(sb + B_BYTES / 2, tb, fb, k0, yg + p.I);  // up projection rows
          } else if (MODE == MODE_DOWN) {
            if (!t.shared) tma_load_2d(sb, &p.tmB0, fb, k0, t.prob * p.H + t.n0);
            else tma_load_2d(sb, &p.tmB1, fb, k0 % p.I, (k0 / p.I) * p.H + t.n0);
          } else {
            tma_load_2d(sb, &p.tmB0, fb, k0, 0);
          }
        }
        __syncwarp();
        issued_mask |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (ok) {
      // tail: wait until the MMA warp has released every stage (all its commits landed)
      for (int i = 0; i < STAGES; ++i) {
        if (!warp_wait_bounded(bar(c.empty[stage]), phase ^ 1u, abort_flag, p.err, TIMEOUT_NS)) break;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (*abort_flag && lane == 0) {
      for (int s = 0; s < STAGES; ++s)
        if ((issued_mask >> s) & 1u) grace_wait(bar(c.full[s]), (last_parity >> s) & 1u);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    uint32_t stage = 0, phase = 0, acc = 0, aphase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const Tile t = decode_tile<MODE>(p, c, tile);
      if (!warp_wait_bounded(bar(c.tempty[acc]), aphase ^ 1u, abort_flag, p.err, TIMEOUT_NS)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < t.kb; ++kb) {
        if (!warp_wait_bounded(bar(c.full[stage]), phase, abort_flag, p.err, TIMEOUT_NS)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          const uint64_t ad = sdesc_k_sw128(sa);
          const uint64_t bd = sdesc_k_sw128(sa + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_f16(d_tmem, ad + 2u * kk, bd + 2u * kk, IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
          tc_commit(bar(c.empty[stage]));
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(bar(c.tfull[acc]));
      __syncwarp();
      acc ^= 1u;
      if (acc == 0) aphase ^= 1u;
    }
    if (*abort_flag && lane == 0) {
      tc_commit(bar(c.drain));  // arrives once every MMA issued above has completed
      grace_wait(bar(c.drain), 0);
    }
  } else {
    // ================================================================ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint32_t acc = 0, aphase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = decode_tile<MODE>(p, c, tile);
      if (!warp_wait_bounded(bar(c.tfull[acc]), aphase, abort_flag, p.err, TIMEOUT_NS)) break;
      tc_fence_after();
      const int r = q * 32 + lane;
      const bool row_ok = t.m0 + r < t.rows;
      const size_t grow = (size_t)(t.row0 + t.m0 + r);
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if (MODE == MODE_UP) {
        const int ld = t.shared ? p.S * p.I : p.I;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(t.shared ? p.out1 : p.out0);
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t g[32], u[32];
          tmem_ld_32cols(tb + cc * 32, g);
          tmem_ld_32cols(tb + 128 + cc * 32, u);
          tmem_wait_ld_fence(g);
          reg_fence(u);
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(out + grow * ld + t.n0 + cc * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t w4[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int j = v * 8 + 2 * i;
                w4[i] = pack_bf16x2(silu_mul(__uint_as_float(g[j]), __uint_as_float(u[j])),
                                    silu_mul(__uint_as_float(g[j + 1]), __uint_as_float(u[j + 1])));
              }
              dst[v] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
        }
      } else if (MODE == MODE_DOWN) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(t.shared ? p.out1 : p.out0);
#pragma unroll 1
        for (int cc = 0; cc < BN / 32; ++cc) {
          uint32_t v32[32];
          tmem_ld_32cols(tb + cc * 32, v32);
          tmem_wait_ld_fence(v32);
          if (row_ok && t.n0 + cc * 32 < p.H) {
            uint4* dst = reinterpret_cast<uint4*>(out + grow * p.H + t.n0 + cc * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t w4[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int j = v * 8 + 2 * i;
                w4[i] = pack_bf16x2(__uint_as_float(v32[j]), __uint_as_float(v32[j + 1]));
              }
              dst[v] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
        }
      } else {
        float* out = static_cast<float*>(p.out0);
#pragma unroll 1
        for (int cc = 0; cc < BN / 32; ++cc) {
          uint32_t v32[32];
          tmem_ld_32cols(tb + cc * 32, v32);
          tmem_wait_ld_fence(v32);
          if (row_ok) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int col = cc * 32 + i;
              if (col < p.N)
                out[grow * p.N + col] =
                    __uint_as_float(v32[i]) + (p.gate_bias ? p.gate_bias[col] : 0.0f);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(c.tempty[acc]));
      acc ^= 1u;
      if (acc == 0) aphase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// One CTA waits on an mbarrier that nothing ever arrives on; the bounded wait must give up,
// raise the error word and return.
__global__ void wait_selftest_kernel(int* err, unsigned long long timeout_ns) {
  __shared__ uint64_t b;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&b), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  warp_wait_bounded(smem_u32(&b), 0, &abort_flag, err, timeout_ns);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2D bf16 row-major tensor [outer, inner], box [box_outer, 64], 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  auto fn = encode_fn();
  if (fn == nullptr || base == nullptr || inner == 0 || outer == 0) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
cudaError_t launch_mode(const TcParams& prm, int num_sms, cudaStream_t st) {
  static int attr_set_for_device[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set_for_device[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set_for_device[dev] = 1;
  }
  tc_gemm_kernel<MODE><<<num_sms, THREADS, SMEM_BYTES, st>>>(prm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_tc(const GemmArgs& a, int num_sms, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  TcParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.offsets = a.offsets;
  prm.n_routed = a.n_routed;
  prm.has_shared = a.has_shared;
  prm.T = a.T; prm.H = a.H; prm.I = a.I; prm.S = a.S; prm.N = a.N;
  prm.out0 = a.out0; prm.out1 = a.out1;
  prm.gate_bias = a.gate_bias;
  prm.err = a.err;
  const uint64_t H = a.H, I = a.I, S = a.S, N = a.N, T = a.T, R = a.rows_cap;
  bool ok = true;
  if (a.mode == MODE_GATE) {
    ok = make_map(&prm.tmA0, a.a0, H, T, 128) && make_map(&prm.tmB0, a.b0, H, N, 256);
    if (!ok) return cudaErrorInvalidValue;
    return launch_mode<MODE_GATE>(prm, num_sms, st);
  }
  if (a.mode == MODE_UP) {
    if (a.n_routed > 0) ok = ok && make_map(&prm.tmA0, a.a0, H, R, 128) &&
                             make_map(&prm.tmB0, a.b0, H, N * 2 * I, 128);
    if (a.has_shared) ok = ok && make_map(&prm.tmA1, a.a1, H, T, 128) &&
                           make_map(&prm.tmB1, a.b1, H, S * 2 * I, 128);
    if (!ok) return cudaErrorInvalidValue;
    return launch_mode<MODE_UP>(prm, num_sms, st);
  }
  if (a.n_routed > 0) ok = ok && make_map(&prm.tmA0, a.a0, I, R, 128) &&
                           make_map(&prm.tmB0, a.b0, I, N * H, 256);
  if (a.has_shared) ok = ok && make_map(&prm.tmA1, a.a1, S * I, T, 128) &&
                         make_map(&prm.tmB1, a.b1, I, S * H, 256);
  if (!ok) return cudaErrorInvalidValue;
  return launch_mode<MODE_DOWN>(prm, num_sms, st);
}

cudaError_t launch_wait_selftest(int* err, unsigned long long timeout_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace moe
