// Gate scores, group / device limited top-K routing, and expert-load statistics.
//
// Routing ("DeepSeek MoE：从v1到v3的演进", DeepSeek-v2 device-limited routing and DeepSeek-v3
// sigmoid gate + selection bias; "DeepSeek-V3的Group-Limited Expert Routing与负载均衡优化实践",
// sections 1 and 3, group-limited routing):
//   key_e = s_e + b_e, s = softmax(u) or sigmoid(u);
//   group score = sum of the group's top-n keys; keep the best Gk groups (ties: lower group);
//   take the K best keys among their experts (ties: lower expert); w = s (/sum) * scale.
//
// One warp routes one token; lane l holds experts l, l+32, ... (coalesced loads of the
// logit row). Keys are first evaluated in fp32. The chosen set then equals the exact (fp64)
// one unless a decision margin (K-th vs (K+1)-th eligible key, Gk-th vs (Gk+1)-th group
// score) lies within the fp32 error bound of the keys; such a token is rechecked by the same
// warp: for a sigmoid gate only the groups and experts inside the error band are rescored in
// fp64 (refine_sigmoid), otherwise the whole token is redone in fp64. For a softmax gate with no selection bias and max-based (or no) group scores the
// logits themselves order the experts exactly (softmax is monotone), so no exp is needed.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int MAXJ = 8;   // experts per lane: N <= 256

template <typename KT> __device__ __forceinline__ KT neg_inf();
template <> __device__ __forceinline__ float neg_inf<float>() { return -INFINITY; }
template <> __device__ __forceinline__ double neg_inf<double>() { return -(double)INFINITY; }

// Warp-wide argmax on (value desc, index asc); result in every lane.
template <typename KT>
__device__ __forceinline__ void warp_argmax(KT& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    KT ov = __shfl_xor_sync(FULL_MASK, v, o);
    int oi = __shfl_xor_sync(FULL_MASK, i, o);
    if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
  }
}

template <typename KT>
__device__ __forceinline__ KT warp_sum(KT v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
  return v;
}
template <typename KT>
__device__ __forceinline__ KT warp_max(KT v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(FULL_MASK, v, o));
  return v;
}

struct Selection {
  int e;           // lane r < K: the r-th chosen expert
  double kth;      // key of the K-th choice
  double emargin;  // K-th key minus best remaining eligible key (+inf if none)
  double gkth;     // Gk-th group score
  double gmargin;  // Gk-th minus (Gk+1)-th group score (+inf if G == Gk)
  uint32_t gmask;  // chosen groups
  bool ok;
};

// Group scores (sum of each group's top-n keys, n = 1 or 2) of keys held lane-strided (expert
// e = j*32 + lane): lane g < G returns group g's score, the other lanes -inf.
template <typename KT>
__device__ __forceinline__ KT group_scores(const KT (&key)[MAXJ], int lane, int N, int G, int topn,
                                           int J) {
  const int gsz = N / G;
  KT my_gs = neg_inf<KT>();
  {
    if (gsz == 32 && G == J) {
      // group g is register g of every lane: reduce all groups' top-2 side by side
      KT a1[MAXJ], a2[MAXJ];
#pragma unroll
      for (int j = 0; j < MAXJ; ++j) {
        a1[j] = j < J ? key[j] : neg_inf<KT>();
        a2[j] = neg_inf<KT>();
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int j = 0; j < MAXJ; ++j) {
          const KT b1 = __shfl_xor_sync(FULL_MASK, a1[j], o);
          const KT b2 = __shfl_xor_sync(FULL_MASK, a2[j], o);
          const KT n2 = max(min(a1[j], b1), max(a2[j], b2));
          a1[j] = max(a1[j], b1);
          a2[j] = n2;
        }
      }
#pragma unroll
      for (int j = 0; j < MAXJ; ++j)
        if (lane == j) my_gs = (topn == 1) ? a1[j] : a1[j] + a2[j];
    } else {
      for (int g = 0; g < G; ++g) {
        KT a1 = neg_inf<KT>(), a2 = neg_inf<KT>();
#pragma unroll
        for (int j = 0; j < MAXJ; ++j) {
          const int e = j * 32 + lane;
          if (j < J && e < N && e / gsz == g) {
            const KT v = key[j];
            if (v > a1) { a2 = a1; a1 = v; } else if (v > a2) { a2 = v; }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const KT b1 = __shfl_xor_sync(FULL_MASK, a1, o);
          const KT b2 = __shfl_xor_sync(FULL_MASK, a2, o);
          const KT n1 = max(a1, b1);
          const KT n2 = max(min(a1, b1), max(a2, b2));
          a1 = n1; a2 = n2;
        }
        const KT gsv = (topn == 1) ? a1 : a1 + a2;
        if (lane == g) my_gs = gsv;
      }
    }
  }
  return my_gs;
}

// Group-limited top-K over keys held lane-strided (expert e = j*32 + lane).
template <typename KT>
__device__ __forceinline__ Selection select_experts(const KT (&key)[MAXJ], int lane, int N, int K,
                                                    int G, int Gk, int topn, int J) {
  Selection out;
  out.ok = true;
  const int gsz = N / G;
  uint32_t gmask = 0xffffffffu;
  out.gmargin = INFINITY;
  out.gkth = INFINITY;
  if (G > 1) {
    const KT my_gs = group_scores<KT>(key, lane, N, G, topn, J);
    gmask = 0;
    bool taken = false;
    KT last = neg_inf<KT>();
    for (int r = 0; r <= Gk && r < G; ++r) {
      KT v = (lane < G && !taken) ? my_gs : neg_inf<KT>();
      int i = (lane < G && !taken) ? lane : 0x7fffffff;
      warp_argmax(v, i);
      if (r < Gk) {
        if (i == 0x7fffffff) { out.ok = false; break; }
        gmask |= 1u << i;
        if (lane == i) taken = true;
        last = v;
      } else {
        out.gmargin = (double)last - (double)v;
      }
    }
    out.gkth = (double)last;
  }
  out.gmask = gmask;

  uint32_t elig = 0, taken = 0;
#pragma unroll
  for (int j = 0; j < MAXJ; ++j) {
    const int e = j * 32 + lane;
    if (j < J && e < N && ((gmask >> (e / gsz)) & 1u)) elig |= 1u << j;
  }
  out.e = -1;
  KT kth = neg_inf<KT>();
  for (int r = 0; r <= K; ++r) {
    KT v = neg_inf<KT>();
    int i = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) {
      if (((elig & ~taken) >> j) & 1u) {
        if (key[j] > v || i == 0x7fffffff) { v = key[j]; i = j * 32 + lane; }
      }
    }
    warp_argmax(v, i);
    if (r < K) {
      if (i == 0x7fffffff) { out.ok = false; break; }
#pragma unroll
      for (int j = 0; j < MAXJ; ++j)
        if (i == j * 32 + lane) taken |= 1u << j;
      if (lane == r) out.e = i;
      kth = v;
    } else {
      out.emargin = (i == 0x7fffffff) ? (double)INFINITY : (double)kth - (double)v;
    }
  }
  out.kth = (double)kth;
  return out;
}

__device__ __forceinline__ float key_tol(double v) {
  // Bound on |fp32 key - exact key|: a sigmoid or softmax score carries a few ulps of error
  // (expf <= 2 ulp, one IEEE division, one sum), the + bias one rounding; 2e-6 * max(1,|v|)
  // is several times that bound.
  return 2e-6f * fmaxf(1.0f, fabsf((float)v));
}

// One out-of-line copy: the recheck runs for a handful of tokens per launch, with its code
// fetched cold, so its size (not its arithmetic) sets its cost.
__device__ __noinline__ double exact_sigmoid_key(float u, float b) {
  return 1.0 / (1.0 + exp(-(double)u)) + (double)b;
}

// Order-preserving map of a (non-NaN) double onto a signed 64-bit integer: comparisons of the
// exact keys run on the integer pipes instead of the (slow) fp64 one.
__device__ __forceinline__ long long ord64(double d) {
  const long long i = __double_as_longlong(d);
  return i >= 0 ? i : i ^ 0x7fffffffffffffffll;
}
constexpr long long ORD_NONE = (long long)0x8000000000000000ull;  // below every ord64
__device__ __forceinline__ double unord64(long long o) {
  return __longlong_as_double(o >= 0 ? o : o ^ 0x7fffffffffffffffll);
}

// Warp-wide argmax on (ordered key desc, index asc); result in every lane.
__device__ __forceinline__ void warp_argmax_ord(long long& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const long long ov = __shfl_xor_sync(FULL_MASK, v, o);
    const int oi = __shfl_xor_sync(FULL_MASK, i, o);
    if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
  }
}

// Exact selection for a sigmoid gate whose fp32 decision lies within its error bound. Every
// fp32 key is within tol of its exact (fp64) value and every fp32 group score within gtol, so a
// group whose fp32 score exceeds the Gk-th by more than 2 gtol is among the exact best Gk, one
// below it by more than 2 gtol is not, and only the groups inside that band are rescored in
// fp64 (all their experts) when the band holds more groups than places left; likewise for the
// experts around the K-th eligible key with 2 tol. The band's members are ranked by their exact
// values (ties: lower index). The keys are recomputed here from the logits exactly as the fp32
// pass computes them. Lane r < K receives the r-th chosen expert in ascending order; false if a
// rank is missing (the caller then redoes the token entirely in fp64). fp_gmask and fp_kth are
// the fp32 pass's chosen groups and K-th key: when the groups stand, its K-th key is reused.
__device__ __noinline__ bool refine_sigmoid(const float* ut, const float* bias, int lane, int N,
                                            int K, int G, int Gk, int topn, uint32_t fp_gmask,
                                            float fp_kth, int& sel_e) {
  constexpr int NONE = 0x7fffffff;
  const int J = (N + 31) >> 5;
  const int gsz = N / G;
  float u[MAXJ], b[MAXJ], key[MAXJ];
  float kmax = 0.0f;
#pragma unroll 1
  for (int j = 0; j < MAXJ; ++j) {
    const int e = j * 32 + lane;
    const bool v = j < J && e < N;
    u[j] = v ? ut[e] : -INFINITY;
    b[j] = (v && bias != nullptr) ? bias[e] : 0.0f;
    const float s = 1.0f / (1.0f + expf(-u[j]));
    key[j] = v ? s + b[j] : -INFINITY;
    if (v) kmax = fmaxf(kmax, fabsf(key[j]));
  }
  kmax = warp_max(kmax);

  uint32_t gmask = 0xffffffffu;
  if (G > Gk) {
    const float gs = group_scores<float>(key, lane, N, G, topn, J);
    int rnk = 0;  // rank of this lane's group (ties: lower group)
    for (int g = 0; g < G; ++g) {
      const float v = __shfl_sync(FULL_MASK, gs, g);
      if (lane < G && (v > gs || (v == gs && g < lane))) ++rnk;
    }
    const uint32_t at = __ballot_sync(FULL_MASK, lane < G && rnk == Gk - 1);
    const double vg = (double)__shfl_sync(FULL_MASK, gs, __ffs(at) - 1);
    const double gtol = topn * (double)key_tol(kmax) + 6e-8 * fabs(vg);
    const bool in = lane < G && (double)gs > vg + 2.0 * gtol;
    const uint32_t cin = __ballot_sync(FULL_MASK, in);
    const uint32_t band = __ballot_sync(FULL_MASK, lane < G && !in && (double)gs >= vg - 2.0 * gtol);
    const int need = Gk - __popc(cin);
    uint32_t picked = 0;
    if (__popc(band) == need) {
      picked = band;  // every band group is in: no exact score needed
    } else {
      long long gx = ORD_NONE;  // lane g: exact score of band group g (ordered)
      for (uint32_t m = band; m; m &= m - 1) {
        const int g = __ffs(m) - 1;
        long long a1 = ORD_NONE, a2 = ORD_NONE;
        if (gsz == 32 && G == J) {  // group g is register g of every lane
          a1 = ord64(exact_sigmoid_key(u[g], b[g]));
        } else {
#pragma unroll 1
          for (int j = 0; j < MAXJ; ++j) {
            const int e = j * 32 + lane;
            const bool mine = j < J && e < N && e / gsz == g;
            if (__any_sync(FULL_MASK, mine) && mine) {
              const long long o = ord64(exact_sigmoid_key(u[j], b[j]));
              if (o > a1) { a2 = a1; a1 = o; } else if (o > a2) { a2 = o; }
            }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {  // top-2 of the group, compared as integers
          const long long b1 = __shfl_xor_sync(FULL_MASK, a1, o);
          const long long b2 = __shfl_xor_sync(FULL_MASK, a2, o);
          if (b1 > a1) { a2 = max(a1, b2); a1 = b1; }
          else { a2 = max(a2, b1); }
        }
        if (lane == g) gx = ord64(topn == 1 ? unord64(a1) : unord64(a1) + unord64(a2));
      }
      for (int r = 0; r < need; ++r) {
        const bool cand = ((band & ~picked) >> lane) & 1u;
        long long v = cand ? gx : ORD_NONE;
        int i = cand ? lane : NONE;
        warp_argmax_ord(v, i);
        if (i == NONE) return false;
        picked |= 1u << i;
      }
    }
    gmask = cin | picked;
  }

  uint32_t elig = 0;
#pragma unroll 1
  for (int j = 0; j < MAXJ; ++j) {
    const int e = j * 32 + lane;
    if (j < J && e < N && ((gmask >> (e / gsz)) & 1u)) elig |= 1u << j;
  }
  float vk = fp_kth;  // K-th best fp32 eligible key
  uint32_t taken = 0;
  for (int r = 0; r < K && gmask != fp_gmask; ++r) {
    float v = -INFINITY;
    int i = NONE;
#pragma unroll 1
    for (int j = 0; j < MAXJ; ++j)
      if (((elig & ~taken) >> j) & 1u)
        if (key[j] > v || i == NONE) { v = key[j]; i = j * 32 + lane; }
    warp_argmax(v, i);
    if (i == NONE) return false;
#pragma unroll 1
    for (int j = 0; j < MAXJ; ++j)
      if (i == j * 32 + lane) taken |= 1u << j;
    vk = v;
  }
  const double tol = 2.0 * (double)key_tol(vk);
  uint32_t cin = 0, band = 0;
#pragma unroll 1
  for (int j = 0; j < MAXJ; ++j) {
    if ((elig >> j) & 1u) {
      const double d = (double)key[j] - (double)vk;
      if (d > tol) cin |= 1u << j;
      else if (d >= -tol) band |= 1u << j;
    }
  }
  const int need = K - warp_sum(__popc(cin));
  uint32_t picked = 0;
  if (warp_sum(__popc(band)) == need) {
    picked = band;  // every band expert is in
  } else {
    long long kd[MAXJ];
#pragma unroll 1
    for (int j = 0; j < MAXJ; ++j) {
      kd[j] = ORD_NONE;
      const bool mine = (band >> j) & 1u;
      if (__any_sync(FULL_MASK, mine) && mine) kd[j] = ord64(exact_sigmoid_key(u[j], b[j]));
    }
    for (int r = 0; r < need; ++r) {
      long long v = ORD_NONE;
      int i = NONE;
#pragma unroll 1
      for (int j = 0; j < MAXJ; ++j)
        if (((band & ~picked) >> j) & 1u)
          if (kd[j] > v || i == NONE) { v = kd[j]; i = j * 32 + lane; }
      warp_argmax_ord(v, i);
      if (i == NONE) return false;
#pragma unroll 1
      for (int j = 0; j < MAXJ; ++j)
        if (i == j * 32 + lane) picked |= 1u << j;
    }
  }
  // lane r < K takes the r-th chosen expert (any order: the caller sorts them)
  __shared__ int slot[256 / 32][32];
  const uint32_t chosen = cin | picked;
  const int cnt = __popc(chosen);
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += v;
  }
  const int total = __shfl_sync(FULL_MASK, incl, 31);
  if (total != K) return false;
  int* sw = slot[threadIdx.x >> 5];
  int pos = incl - cnt;
#pragma unroll 1
  for (int j = 0; j < MAXJ; ++j)
    if ((chosen >> j) & 1u) sw[pos++] = j * 32 + lane;
  __syncwarp();
  sel_e = lane < K ? sw[lane] : -1;
  __syncwarp();
  return true;
}

__global__ void __launch_bounds__(256) route_kernel(RouteArgs a) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int J = (a.N + 31) >> 5;
  const bool sigmoid = a.score_fn == 1;
  // Softmax with no selection bias and max-based (or no) group limit: order by the logits.
  const bool exact_logit_keys = !sigmoid && a.bias == nullptr && (a.G == 1 || a.topn == 1);

  float b[MAXJ];
#pragma unroll
  for (int j = 0; j < MAXJ; ++j) {
    const int e = j * 32 + lane;
    b[j] = (a.bias != nullptr && j < J && e < a.N) ? a.bias[e] : 0.0f;
  }

  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < a.T; t += warps) {
    const float* ut = a.u + (size_t)t * a.N;
    float u[MAXJ];
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) {
      const int e = j * 32 + lane;
      u[j] = (j < J && e < a.N) ? ut[e] : -INFINITY;
    }
    // ---- fp32 scores and keys
    float s[MAXJ], key[MAXJ];
    float umax = u[0];
#pragma unroll
    for (int j = 1; j < MAXJ; ++j) umax = fmaxf(umax, u[j]);
    umax = warp_max(umax);
    if (sigmoid) {
#pragma unroll
      for (int j = 0; j < MAXJ; ++j) s[j] = 1.0f / (1.0f + expf(-u[j]));
    } else {
      float z = 0.0f;
#pragma unroll
      for (int j = 0; j < MAXJ; ++j) { s[j] = expf(u[j] - umax); z += s[j]; }
      z = warp_sum(z);
#pragma unroll
      for (int j = 0; j < MAXJ; ++j) s[j] = s[j] / z;
    }
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) key[j] = exact_logit_keys ? u[j] : s[j] + b[j];

    Selection sel = select_experts<float>(key, lane, a.N, a.K, a.G, a.Gk, a.topn, J);
    bool redo;
    if (exact_logit_keys) {
      // Logit order equals exact-probability order except where exp underflows in fp64 or two
      // distinct logits are so close that their fp64 probabilities may coincide.
      const double tiny = 1e-9 * fmax(1.0, fabs(sel.kth));
      redo = !sel.ok || (sel.kth - umax < -600.0) || (a.G > a.Gk && sel.gkth - umax < -600.0) ||
             (sel.emargin > 0.0 && sel.emargin < tiny) ||
             (a.G > a.Gk && sel.gmargin > 0.0 && sel.gmargin < 1e-9 * fmax(1.0, fabs(sel.gkth)));
    } else {
      // A group score is the fp32 sum of its top-n keys: it is off by at most n key errors
      // (the n-th largest of perturbed values moves by at most the largest perturbation) plus
      // the rounding of the sum.
      float kmax = 0.0f;
#pragma unroll
      for (int j = 0; j < MAXJ; ++j)
        if (j < J && j * 32 + lane < a.N) kmax = fmaxf(kmax, fabsf(key[j]));
      kmax = warp_max(kmax);
      const double gtol = a.topn * (double)key_tol(kmax) + 6e-8 * fabs(sel.gkth);
      redo = !sel.ok || sel.emargin <= 2.0 * key_tol(sel.kth) ||
             (a.G > a.Gk && sel.gmargin <= 2.0 * gtol);
    }
    redo = __any_sync(FULL_MASK, redo);
    int sel_e = sel.e;
    if (redo && sigmoid && sel.ok && !a.precise_w) {
      // rescore only the groups and experts within the error bound of a decision
      int e_ref = -1;
      if (refine_sigmoid(ut, a.bias, lane, a.N, a.K, a.G, a.Gk, a.topn, sel.gmask, (float)sel.kth,
                         e_ref)) {
        sel_e = e_ref;
        redo = false;
      }
    }

    // ---- weights: scores of the chosen experts (fp32 unless an fp64 pass is needed)
    double sd_z = 0.0;  // fp64 softmax normaliser (fp64 passes only)
    double sel_s = 0.0;
    const bool need_f64 = redo || a.precise_w;
    if (need_f64) {
      double sd[MAXJ];
      if (sigmoid) {
#pragma unroll
        for (int j = 0; j < MAXJ; ++j) sd[j] = 1.0 / (1.0 + exp(-(double)u[j]));
      } else {
        double z = 0.0;
#pragma unroll
        for (int j = 0; j < MAXJ; ++j) { sd[j] = exp((double)u[j] - (double)umax); z += sd[j]; }
        sd_z = warp_sum(z);
#pragma unroll
        for (int j = 0; j < MAXJ; ++j) sd[j] = sd[j] / sd_z;
      }
      if (redo) {
        double kd[MAXJ];
#pragma unroll
        for (int j = 0; j < MAXJ; ++j)
          kd[j] = (j < J && j * 32 + lane < a.N) ? sd[j] + (double)b[j] : neg_inf<double>();
        Selection sd_sel = select_experts<double>(kd, lane, a.N, a.K, a.G, a.Gk, a.topn, J);
        if (!sd_sel.ok) set_error(a.err, ERR_DEVICE_CHECK);
        sel_e = sd_sel.e;
      }
      // fetch s of each chosen expert from its owner lane
      for (int r = 0; r < a.K; ++r) {
        const int e = __shfl_sync(FULL_MASK, sel_e, r);
        double mine = 0.0;
#pragma unroll
        for (int j = 0; j < MAXJ; ++j)
          if (e == j * 32 + lane) mine = sd[j];
        const double v = __shfl_sync(FULL_MASK, mine, e & 31);
        if (lane == r) sel_s = v;
      }
      double denom = warp_sum(lane < a.K ? sel_s : 0.0);
      double wv = sel_s;
      if (a.norm_topk) wv = wv / denom;
      wv = wv * (double)a.scale;
      sel_s = wv;
    } else {
      float mine_s = 0.0f, ss = 0.0f;
      for (int r = 0; r < a.K; ++r) {
        const int e = __shfl_sync(FULL_MASK, sel_e, r);
        mine_s = 0.0f;
#pragma unroll
        for (int j = 0; j < MAXJ; ++j)
          if (e == j * 32 + lane) mine_s = s[j];
        const float v = __shfl_sync(FULL_MASK, mine_s, e & 31);
        if (lane == r) ss = v;
      }
      float denom = warp_sum(lane < a.K ? ss : 0.0f);
      float wv = ss;
      if (a.norm_topk) wv = wv / denom;
      sel_s = (double)(wv * a.scale);
    }
    if (!sel.ok && !redo) set_error(a.err, ERR_DEVICE_CHECK);

    // ---- write in ascending expert order
    int rank = 0;
    for (int r = 0; r < a.K; ++r) {
      const int e = __shfl_sync(FULL_MASK, sel_e, r);
      if (lane < a.K && e < sel_e) ++rank;
    }
    if (lane < a.K) {
      const int e = (sel_e >= 0 && sel_e < a.N) ? sel_e : 0;
      a.idx[(size_t)t * a.K + rank] = e;
      a.w[(size_t)t * a.K + rank] = (float)sel_s;
    }
  }
}

// ---------------------------------------------------------------- load statistics
// Per-block partial sums of the scores of every expert and of lse, lse^2 over its tokens.
__global__ void __launch_bounds__(256) stats_partial_kernel(StatsArgs a) {
  __shared__ float red[8][256];
  __shared__ double redl[8][2];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int J = (a.N + 31) >> 5;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  float acc[MAXJ];
#pragma unroll
  for (int j = 0; j < MAXJ; ++j) acc[j] = 0.0f;
  double l1 = 0.0, l2 = 0.0;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < a.T; t += warps) {
    const float* ut = a.u + (size_t)t * a.N;
    float u[MAXJ];
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) {
      const int e = j * 32 + lane;
      u[j] = (j < J && e < a.N) ? ut[e] : -INFINITY;
    }
    float m = u[0];
#pragma unroll
    for (int j = 1; j < MAXJ; ++j) m = fmaxf(m, u[j]);
    m = warp_max(m);
    float ex[MAXJ], z = 0.0f;
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) { ex[j] = expf(u[j] - m); z += ex[j]; }
    z = warp_sum(z);
    if (a.score_fn == 1) {
#pragma unroll
      for (int j = 0; j < MAXJ; ++j)
        if (j < J && j * 32 + lane < a.N) acc[j] += 1.0f / (1.0f + expf(-u[j]));
    } else {
#pragma unroll
      for (int j = 0; j < MAXJ; ++j) acc[j] += ex[j] / z;
    }
    const double lse = (double)m + log((double)z);
    l1 += lse;
    l2 += lse * lse;
  }
#pragma unroll
  for (int j = 0; j < MAXJ; ++j) {
    const int e = j * 32 + lane;
    if (e < 256) red[wid][e] = (j < J && e < a.N) ? acc[j] : 0.0f;
  }
  if (lane == 0) { redl[wid][0] = l1; redl[wid][1] = l2; }
  __syncthreads();
  for (int e = threadIdx.x; e < a.N; e += blockDim.x) {
    float s = 0.0f;
    for (int w = 0; w < 8; ++w) s += red[w][e];
    a.part_s[(size_t)blockIdx.x * a.N + e] = s;
  }
  if (threadIdx.x == 0) {
    double s1 = 0.0, s2 = 0.0;
    for (int w = 0; w < 8; ++w) { s1 += redl[w][0]; s2 += redl[w][1]; }
    a.part_lse[blockIdx.x * 2 + 0] = s1;
    a.part_lse[blockIdx.x * 2 + 1] = s2;
  }
}

__global__ void stats_count_kernel(const int32_t* idx, long long n, int N, int32_t* counts,
                                   int* err) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int e = idx[i];
    if (e >= 0 && e < N) atomicAdd(&counts[e], 1);
    else set_error(err, ERR_DEVICE_CHECK);
  }
}

// Fixed-order fp64 reduction of the partials: f, P, L_B, L_Z, mean lse.
__global__ void __launch_bounds__(256) stats_final_kernel(StatsArgs a) {
  __shared__ double colsum[256];
  __shared__ double term[256];
  const int e = threadIdx.x;
  double cs = 0.0;
  if (e < a.N)
    for (int b = 0; b < a.nblk; ++b) cs += (double)a.part_s[(size_t)b * a.N + e];
  colsum[e] = cs;
  __syncthreads();
  if (e == 0) {
    double tot = 0.0;
    for (int i = 0; i < a.N; ++i) tot += colsum[i];
    term[0] = tot;
  }
  __syncthreads();
  const double total = term[0];
  __syncthreads();
  double fe = 0.0, pe = 0.0;
  if (e < a.N) {
    fe = (double)a.counts[e] / ((double)a.T * a.K);
    pe = colsum[e] / total;
    if (a.f) a.f[e] = (float)fe;
    if (a.P) a.P[e] = (float)pe;
  }
  term[e] = (e < a.N) ? fe * pe : 0.0;
  __syncthreads();
  if (e == 0 && a.lb_z) {
    double lb = 0.0;
    for (int i = 0; i < a.N; ++i) lb += term[i];
    double s1 = 0.0, s2 = 0.0;
    for (int b = 0; b < a.nblk; ++b) { s1 += a.part_lse[2 * b]; s2 += a.part_lse[2 * b + 1]; }
    a.lb_z[0] = (float)(lb * a.N);
    a.lb_z[1] = (float)(s2 / a.T);
    a.lb_z[2] = (float)(s1 / a.T);
  }
}

// Per token: expert counts, and one received token for each distinct device it uses.
__global__ void group_count_kernel(GroupLossArgs a) {
  const int per = a.st.N / a.G;
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < a.st.T; t += gridDim.x * blockDim.x) {
    uint32_t devs = 0;
    for (int k = 0; k < a.st.K; ++k) {
      const int e = a.st.idx[(size_t)t * a.st.K + k];
      if (e < 0 || e >= a.st.N) { set_error(a.st.err, ERR_DEVICE_CHECK); continue; }
      atomicAdd(&a.st.counts[e], 1);
      devs |= 1u << (e / per);
    }
    while (devs) {
      const int d = __ffs(devs) - 1;
      devs &= devs - 1;
      atomicAdd(&a.recv[d], 1);
    }
  }
}

// Fixed-order fp64 reduction: per-expert score sums and counts -> per-device shares -> losses.
__global__ void __launch_bounds__(256) group_final_kernel(GroupLossArgs a) {
  __shared__ double colsum[256];
  __shared__ double tot[1];
  const int e = threadIdx.x, N = a.st.N;
  double cs = 0.0;
  if (e < N)
    for (int b = 0; b < a.st.nblk; ++b) cs += (double)a.st.part_s[(size_t)b * N + e];
  colsum[e] = cs;
  __syncthreads();
  if (e == 0) {
    double t = 0.0;
    for (int i = 0; i < N; ++i) t += colsum[i];
    tot[0] = t;
  }
  __syncthreads();
  if (e == 0) {
    const int per = N / a.G;
    double recv_tot = 0.0;
    for (int d = 0; d < a.G; ++d) recv_tot += (double)a.recv[d];
    double l_dev = 0.0, l_comm = 0.0;
    for (int d = 0; d < a.G; ++d) {
      double f = 0.0, P = 0.0;
      for (int i = d * per; i < (d + 1) * per; ++i) {
        f += (double)a.st.counts[i] / ((double)a.st.T * a.st.K);
        P += colsum[i] / tot[0];
      }
      l_dev += f * P;
      l_comm += (double)a.recv[d] / recv_tot * P;
    }
    a.out[0] = (float)(a.G * l_dev);
    a.out[1] = (float)(a.G * l_comm);
  }
}

}  // namespace

cudaError_t launch_group_losses(const GroupLossArgs& a, cudaStream_t st) {
  if (a.st.T <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(a.st.counts, 0, sizeof(int32_t) * a.st.N, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(a.recv, 0, sizeof(int32_t) * a.G, st);
  if (e != cudaSuccess) return e;
  int cb = (a.st.T + 255) / 256;
  if (cb > 1184) cb = 1184;
  group_count_kernel<<<cb, 256, 0, st>>>(a);
  stats_partial_kernel<<<a.st.nblk, 256, 0, st>>>(a.st);
  group_final_kernel<<<1, 256, 0, st>>>(a);
  note_launches(3);
  return cudaGetLastError();
}

cudaError_t launch_route(const RouteArgs& a, int num_sms, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  const int warps_needed = a.T;
  int blocks = (warps_needed + 7) / 8;
  const int cap = num_sms * 8;
  if (blocks > cap) blocks = cap;
  route_kernel<<<blocks, 256, 0, st>>>(a);
  note_launches(1);
  return cudaGetLastError();
}

int stats_blocks(int T) {
  int b = (T + 63) / 64;  // 8 warps x 8 tokens
  if (b < 1) b = 1;
  if (b > 1184) b = 1184;
  return b;
}

cudaError_t launch_stats(const StatsArgs& a, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(a.counts, 0, sizeof(int32_t) * a.N, st);
  if (e != cudaSuccess) return e;
  const long long n = (long long)a.T * a.K;
  int cb = (int)((n + 255) / 256);
  if (cb > 1184) cb = 1184;
  stats_count_kernel<<<cb, 256, 0, st>>>(a.idx, n, a.N, a.counts, a.err);
  stats_partial_kernel<<<a.nblk, 256, 0, st>>>(a);
  stats_final_kernel<<<1, 256, 0, st>>>(a);
  note_launches(3);
  return cudaGetLastError();
}

}  // namespace moe
