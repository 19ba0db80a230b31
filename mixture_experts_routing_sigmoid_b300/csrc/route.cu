// Gate scores, group / device limited top-K routing, and expert-load statistics.
//
// Routing ("DeepSeek MoE：从v1到v3的演进", DeepSeek-v2 device-limited routing and DeepSeek-v3
// sigmoid gate + selection bias; "DeepSeek-V3的Group-Limited Expert Routing与负载均衡优化实践",
// sections 1 and 3, group-limited routing):
//   key_e = s_e + b_e, s = softmax(u) or sigmoid(u);
//   group score = sum of the group's top-n keys; keep the best Gk groups (ties: lower group);
//   take the K best keys among their experts (ties: lower expert); w = s (/sum) * scale.
// The order is that of the real numbers key_e (and of the real sums of them). Two values closer
// than 2^-80 of their size count as equal, and the lower index wins, as for exact ties.
//
// One warp routes one token; lane l holds experts l, l+32, ... (coalesced loads of the logit
// row). Keys are first evaluated in fp32 and the choice is made with warp reductions
// (redux.sync max / min over order-preserving integer images of the keys: one reduction per
// group score half, per kept group and per chosen expert). That choice is the real one unless a
// decision margin (K-th vs (K+1)-th eligible key, Gk-th vs (Gk+1)-th group score) lies within the
// fp32 error bound of the keys. Such a token is rechecked by the same warp:
//   - sigmoid gate: only the groups and experts inside the error band are rescored, in
//     double-double arithmetic (~100 bits, refine_sigmoid), which settles their real order;
//   - softmax gate with no selection bias and max-based (or no) group scores: the logits
//     themselves give the real order (softmax is monotone), so nothing is ever rechecked;
//   - other softmax combinations (a selection bias, or group scores that sum two keys; no page
//     describes them): the token is redone with fp64 keys, whose order matches the real one
//     except for keys within a few fp64 units of each other.
// Weights are fp32 (within a few ulps), or, when the v2 drop will rank them, computed in fp64
// and rounded once.
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

// Order-preserving map of a non-NaN float onto uint32 (0 stays free: "no key").
__device__ __forceinline__ uint32_t ord32(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float unord32(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// Bound on |fp32 key - real key| for keys of magnitude at most |v| (or 1).
//   sigmoid: expf is within 2 ulp (2.4e-7 relative), 1 + e and the IEEE division add 6e-8
//   each, so s is within 3.6e-7 (absolute, s < 1); + b adds half an ulp of the key: 4.2e-7 in
//   all for |key| <= 1, bounded here by 5e-7 * max(1, |v|).
//   softmax: besides the exp, the normaliser is a sum of up to 256 terms (8 per lane, then a
//   5-level warp tree), within 1e-6 relative; 2e-6 * max(1, |v|) bounds the score's error.
__device__ __forceinline__ float key_tol(float v, bool sigmoid) {
  return (sigmoid ? 5e-7f : 2e-6f) * fmaxf(1.0f, fabsf(v));
}

// ---------------------------------------------------------------- fp32 choice (redux)
struct FastSel {
  int e;          // lane r < K: the r-th chosen expert (in choice order)
  float se;       // lane r < K: its score s
  float ssum;     // sum of the K chosen scores (every lane)
  float kth;      // K-th chosen key
  float next;     // best remaining eligible key (-inf if none)
  float gkth;     // Gk-th group score (+inf if G == Gk)
  float gnext;    // (Gk+1)-th group score (-inf if none)
  uint32_t gmask; // kept groups
  bool ok;
};

// gj[j]: group of this lane's expert j*32 + lane; ok[j]: its ordered key (0: no expert).
// JM: experts per lane the caller holds (a compile-time bound on ceil(N / 32)).
template <int JM>
__device__ __forceinline__ FastSel fast_select(const uint32_t (&ok)[JM], const float (&s)[JM],
                                               const int (&gj)[JM], int lane, int K, int G,
                                               int Gk, int topn) {
  FastSel out;
  out.ok = true;
  out.gmask = 0xffffffffu;
  out.gkth = INFINITY;
  out.gnext = -INFINITY;
  if (G > Gk) {
    // group scores: the group's best key, plus (topn == 2) the best of the rest
    float gs = -INFINITY;  // lane g < G: group g's score
    for (int g = 0; g < G; ++g) {
      uint32_t l1 = 0, l2 = 0;
#pragma unroll
      for (int j = 0; j < JM; ++j) {
        if (gj[j] == g) {
          const uint32_t v = ok[j];
          if (v > l1) { l2 = l1; l1 = v; } else if (v > l2) { l2 = v; }
        }
      }
      const uint32_t m1 = __reduce_max_sync(FULL_MASK, l1);
      float v = unord32(m1);
      if (topn == 2) {
        const int holder = __ffs(__ballot_sync(FULL_MASK, l1 == m1)) - 1;
        v += unord32(__reduce_max_sync(FULL_MASK, lane == holder ? l2 : l1));
      }
      if (lane == g) gs = v;
    }
    const uint32_t go = lane < G ? ord32(gs) : 0u;
    bool taken = false;
    uint32_t last = 0;
    out.gmask = 0;
    for (int r = 0; r <= Gk && r < G; ++r) {
      const uint32_t v = taken ? 0u : go;
      const uint32_t m = __reduce_max_sync(FULL_MASK, v);
      const uint32_t bal = __ballot_sync(FULL_MASK, m != 0u && v == m);
      if (bal == 0u) { out.ok = false; break; }
      const int gi = __ffs(bal) - 1;  // the lowest group among equal scores
      if (r < Gk) {
        out.gmask |= 1u << gi;
        if (lane == gi) taken = true;
        last = m;
      } else {
        out.gnext = unord32(m);
      }
    }
    out.gkth = last ? unord32(last) : -INFINITY;
  }
  uint32_t avail = 0;  // bit j: expert j*32 + lane is eligible and not chosen yet
#pragma unroll
  for (int j = 0; j < JM; ++j)
    if (ok[j] != 0u && gj[j] >= 0 && ((out.gmask >> gj[j]) & 1u)) avail |= 1u << j;
  out.e = -1;
  out.se = 0.0f;
  out.ssum = 0.0f;
  out.next = -INFINITY;
  uint32_t kth = 0;
  for (int r = 0; r <= K; ++r) {
    uint32_t best = 0;
    int bj = 0;
    float bs = 0.0f;
#pragma unroll
    for (int j = 0; j < JM; ++j)
      if (((avail >> j) & 1u) && ok[j] > best) { best = ok[j]; bj = j; bs = s[j]; }
    const uint32_t m = __reduce_max_sync(FULL_MASK, best);
    if (r == K) {
      if (m != 0u) out.next = unord32(m);
      break;
    }
    if (m == 0u) { out.ok = false; break; }
    // the lowest expert among the lanes holding the maximum (each lane offers its lowest)
    const uint32_t e = __reduce_min_sync(FULL_MASK, best == m ? (uint32_t)(bj * 32 + lane) : ~0u);
    const float se = __shfl_sync(FULL_MASK, bs, e & 31);
    if (lane == (int)(e & 31)) avail &= ~(1u << (e >> 5));
    if (lane == r) { out.e = (int)e; out.se = se; }
    out.ssum += se;
    kth = m;
  }
  out.kth = kth ? unord32(kth) : -INFINITY;
  return out;
}

// ---------------------------------------------------------------- fp64 choice (cold path)
struct Selection {
  int e;           // lane r < K: the r-th chosen expert
  bool ok;
};

// Group scores (sum of each group's top-n keys, n = 1 or 2) of keys held lane-strided (expert
// e = j*32 + lane): lane g < G returns group g's score, the other lanes -inf.
template <typename KT>
__device__ __forceinline__ KT group_scores(const KT (&key)[MAXJ], int lane, int N, int G, int topn,
                                           int J) {
  const int gsz = N / G;
  KT my_gs = neg_inf<KT>();
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
  if (G > 1) {
    const KT my_gs = group_scores<KT>(key, lane, N, G, topn, J);
    gmask = 0;
    bool taken = false;
    for (int r = 0; r < Gk && r < G; ++r) {
      KT v = (lane < G && !taken) ? my_gs : neg_inf<KT>();
      int i = (lane < G && !taken) ? lane : 0x7fffffff;
      warp_argmax(v, i);
      if (i == 0x7fffffff) { out.ok = false; break; }
      gmask |= 1u << i;
      if (lane == i) taken = true;
    }
  }
  uint32_t elig = 0, taken = 0;
#pragma unroll
  for (int j = 0; j < MAXJ; ++j) {
    const int e = j * 32 + lane;
    if (j < J && e < N && ((gmask >> (e / gsz)) & 1u)) elig |= 1u << j;
  }
  out.e = -1;
  for (int r = 0; r < K; ++r) {
    KT v = neg_inf<KT>();
    int i = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) {
      if (((elig & ~taken) >> j) & 1u) {
        if (key[j] > v || i == 0x7fffffff) { v = key[j]; i = j * 32 + lane; }
      }
    }
    warp_argmax(v, i);
    if (i == 0x7fffffff) { out.ok = false; break; }
#pragma unroll
    for (int j = 0; j < MAXJ; ++j)
      if (i == j * 32 + lane) taken |= 1u << j;
    if (lane == r) out.e = i;
  }
  return out;
}

// ---------------------------------------------------------------- double-double arithmetic
// Values as unevaluated sums hi + lo of two doubles (~106 bits), from the error-free
// transformations of Knuth (two-sum) and Dekker (two-product, here with an FMA). The exp follows
// the scheme of Hida, Li and Bailey's double-double library: reduce by k ln 2, scale by 2^-9, a
// Taylor series for expm1, nine doublings expm1(2y) = 2 expm1(y) + expm1(y)^2, then 2^k.
struct DD {
  double hi, lo;
};
__device__ __forceinline__ DD dd_two_sum(double a, double b) {
  const double s = a + b;
  const double bb = s - a;
  return {s, (a - (s - bb)) + (b - bb)};
}
__device__ __forceinline__ DD dd_fast_two_sum(double a, double b) {  // |a| >= |b|
  const double s = a + b;
  return {s, b - (s - a)};
}
__device__ __forceinline__ DD dd_add(DD a, DD b) {
  DD s = dd_two_sum(a.hi, b.hi);
  const DD t = dd_two_sum(a.lo, b.lo);
  s.lo += t.hi;
  s = dd_fast_two_sum(s.hi, s.lo);
  s.lo += t.lo;
  return dd_fast_two_sum(s.hi, s.lo);
}
__device__ __forceinline__ DD dd_neg(DD a) { return {-a.hi, -a.lo}; }
__device__ __forceinline__ DD dd_mul(DD a, DD b) {
  const double p = a.hi * b.hi;
  double e = fma(a.hi, b.hi, -p);
  e = fma(a.hi, b.lo, e);
  e = fma(a.lo, b.hi, e);
  return dd_fast_two_sum(p, e);
}
__device__ __forceinline__ DD dd_mul_d(DD a, double b) {
  const double p = a.hi * b;
  double e = fma(a.hi, b, -p);
  e = fma(a.lo, b, e);
  return dd_fast_two_sum(p, e);
}
__device__ __forceinline__ DD dd_div(DD a, DD b) {
  const double q1 = a.hi / b.hi;
  DD r = dd_add(a, dd_neg(dd_mul_d(b, q1)));
  const double q2 = r.hi / b.hi;
  r = dd_add(r, dd_neg(dd_mul_d(b, q2)));
  const double q3 = r.hi / b.hi;
  return dd_add(dd_fast_two_sum(q1, q2), DD{q3, 0.0});
}
__device__ __noinline__ DD dd_exp(double x) {
  if (x > 709.0) return {INFINITY, 0.0};
  if (x < -745.0) return {0.0, 0.0};
  const DD ln2 = {0x1.62e42fefa39efp-1, 0x1.abc9e3b39803fp-56};
  const double k = rint(x / ln2.hi);
  DD r = dd_add(DD{x, 0.0}, dd_neg(dd_mul_d(ln2, k)));
  r.hi *= 0x1p-9;
  r.lo *= 0x1p-9;
  // 1/n for n = 2..10 as double-double pairs (rounded to nearest, the rest in the low part)
  const double inv_hi[9] = {0x1p-1, 0x1.5555555555555p-2, 0x1p-2, 0x1.999999999999ap-3,
                            0x1.5555555555555p-3, 0x1.2492492492492p-3, 0x1p-3,
                            0x1.c71c71c71c71cp-4, 0x1.999999999999ap-4};
  const double inv_lo[9] = {0.0, 0x1.5555555555555p-56, 0.0, -0x1.999999999999ap-57,
                            0x1.5555555555555p-57, 0x1.2492492492492p-57, 0.0,
                            0x1.c71c71c71c71cp-58, -0x1.999999999999ap-58};
  DD p = r, s = r;
#pragma unroll 1
  for (int n = 2; n <= 10; ++n) {
    p = dd_mul(dd_mul(p, r), DD{inv_hi[n - 2], inv_lo[n - 2]});
    s = dd_add(s, p);
  }
#pragma unroll 1
  for (int i = 0; i < 9; ++i) s = dd_add(dd_mul_d(s, 2.0), dd_mul(s, s));
  s = dd_add(s, DD{1.0, 0.0});
  const int ki = (int)k;
  return {ldexp(s.hi, ki), ldexp(s.lo, ki)};
}
// sigmoid(u) + b in double-double.
__device__ __noinline__ DD dd_sigmoid_key(float u, float b) {
  const DD e = dd_exp(-(double)u);
  DD s = {0.0, 0.0};
  if (e.hi != INFINITY) s = dd_div(DD{1.0, 0.0}, dd_add(DD{1.0, 0.0}, e));
  return dd_add(s, DD{(double)b, 0.0});
}
// Real order with ties: -1 if a is larger, +1 if b is, 0 if they are within 2^-80 of their size.
__device__ __forceinline__ int dd_cmp(DD a, DD b) {
  const DD d = dd_add(a, dd_neg(b));
  const double tie = 0x1p-80 * fmax(fabs(a.hi), fabs(b.hi));
  return d.hi > tie ? -1 : (d.hi < -tie ? 1 : 0);
}
// Warp-wide argmax of (dd value desc under dd_cmp, index asc) over lanes with `valid`; i = -1 if
// no lane is valid. Result in every lane.
__device__ __forceinline__ void warp_argmax_dd(DD& v, int& i, bool valid) {
  if (!valid) i = -1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    DD ov;
    ov.hi = __shfl_xor_sync(FULL_MASK, v.hi, o);
    ov.lo = __shfl_xor_sync(FULL_MASK, v.lo, o);
    const int oi = __shfl_xor_sync(FULL_MASK, i, o);
    bool take;
    if (oi < 0) take = false;
    else if (i < 0) take = true;
    else {
      const int c = dd_cmp(ov, v);
      take = c < 0 || (c == 0 && oi < i);
    }
    if (take) { v = ov; i = oi; }
  }
}

// fp64 key sigmoid(u) + b: within a few units in the last place of the real key (one out-of-line
// copy: the recheck runs for a handful of tokens per launch, with its code fetched cold).
__device__ __noinline__ double sigmoid_key64(float u, float b) {
  return 1.0 / (1.0 + exp(-(double)u)) + (double)b;
}
// fp64 keys (and sums of two) carry a few units in the last place of error, far below this
// distance; two fp64 values closer than it are ordered in double-double instead.
__device__ __forceinline__ bool near64(double a, double b) {
  return fabs(a - b) <= 1e-14 * fmax(1.0, fmax(fabs(a), fabs(b)));
}
// Order-preserving map of a (non-NaN) double onto a signed 64-bit integer: comparisons of the
// fp64 keys run on the integer pipes instead of the (slow) fp64 one.
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

// Exact selection for a sigmoid gate whose fp32 decision lies within its error bound. Every fp32
// key is within tol of its real value and every fp32 group score within gtol, so a group whose
// fp32 score exceeds the Gk-th by more than 2 gtol is among the real best Gk, one below it by more
// than 2 gtol is not, and only the groups inside that band are rescored (all their experts) when
// the band holds more groups than places left; likewise for the experts around the K-th eligible
// key with 2 tol. The band is ranked by fp64 keys first; only when the fp64 values on both sides
// of the cut are within near64() of each other is the band ranked again by double-double values
// (dd_cmp; ties: lower index). The fp32 keys are recomputed here from the logits exactly as the
// fp32 pass computes them. Lane r < K receives the r-th chosen expert; false if a rank is missing.
// fp_gmask and fp_kth are the fp32 pass's chosen groups and K-th key: when the groups stand, its
// K-th key is reused.
__device__ __noinline__ bool refine_sigmoid(const float* ut, const float* bias, int lane, int N,
                                            int K, int G, int Gk, int topn, uint32_t fp_gmask,
                                            float fp_kth, int& sel_e) {
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
    const double gtol = topn * (double)key_tol(kmax, true) + 6e-8 * fabs(vg);
    const bool in = lane < G && (double)gs > vg + 2.0 * gtol;
    const uint32_t cin = __ballot_sync(FULL_MASK, in);
    const uint32_t band = __ballot_sync(FULL_MASK, lane < G && !in && (double)gs >= vg - 2.0 * gtol);
    const int need = Gk - __popc(cin);
    uint32_t picked = 0;
    if (__popc(band) == need) {
      picked = band;  // every band group is in: no exact score needed
    } else {
      // fp64 scores of the band groups (lane g: group g's, ordered)
      long long gx = ORD_NONE;
      for (uint32_t m = band; m; m &= m - 1) {
        const int g = __ffs(m) - 1;
        long long a1 = ORD_NONE, a2 = ORD_NONE;
#pragma unroll 1
        for (int j = 0; j < MAXJ; ++j) {
          const int e = j * 32 + lane;
          const bool mine = j < J && e < N && e / gsz == g;
          if (__any_sync(FULL_MASK, mine) && mine) {
            const long long o = ord64(sigmoid_key64(u[j], b[j]));
            if (o > a1) { a2 = a1; a1 = o; } else if (o > a2) { a2 = o; }
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
      long long v_cut = ORD_NONE, v_next = ORD_NONE;
      for (int r = 0; r <= need; ++r) {
        const bool cand = ((band & ~picked) >> lane) & 1u;
        long long v = cand ? gx : ORD_NONE;
        int i = cand ? lane : 0x7fffffff;
        warp_argmax_ord(v, i);
        if (r == need) { v_next = v; break; }
        if (i == 0x7fffffff) return false;
        picked |= 1u << i;
        v_cut = v;
      }
      if (v_next != ORD_NONE && v_cut != ORD_NONE && near64(unord64(v_cut), unord64(v_next))) {
        // fp64 cannot settle the cut: real scores of the band groups in double-double
        DD gd = {0.0, 0.0};
        for (uint32_t m = band; m; m &= m - 1) {
          const int g = __ffs(m) - 1;
          DD a1 = {0.0, 0.0}, a2 = {0.0, 0.0};
          bool h1 = false, h2 = false;
#pragma unroll 1
          for (int j = 0; j < MAXJ; ++j) {
            const int e = j * 32 + lane;
            const bool mine = j < J && e < N && e / gsz == g;
            if (__any_sync(FULL_MASK, mine) && mine) {
              const DD k = dd_sigmoid_key(u[j], b[j]);
              if (!h1 || dd_cmp(k, a1) < 0) { a2 = a1; h2 = h1; a1 = k; h1 = true; }
              else if (!h2 || dd_cmp(k, a2) < 0) { a2 = k; h2 = true; }
            }
          }
#pragma unroll 1
          for (int o = 16; o > 0; o >>= 1) {
            DD b1, b2;
            b1.hi = __shfl_xor_sync(FULL_MASK, a1.hi, o);
            b1.lo = __shfl_xor_sync(FULL_MASK, a1.lo, o);
            b2.hi = __shfl_xor_sync(FULL_MASK, a2.hi, o);
            b2.lo = __shfl_xor_sync(FULL_MASK, a2.lo, o);
            const bool g1 = __shfl_xor_sync(FULL_MASK, h1, o);
            const bool g2 = __shfl_xor_sync(FULL_MASK, h2, o);
            // merge the two sorted pairs (a1 >= a2, b1 >= b2) into the top two
            if (g1 && (!h1 || dd_cmp(b1, a1) < 0)) {
              const bool second_b2 = g2 && (!h1 || dd_cmp(b2, a1) < 0);
              a2 = second_b2 ? b2 : a1;
              h2 = second_b2 ? true : h1;
              a1 = b1;
              h1 = true;
            } else if (g1 && (!h2 || dd_cmp(b1, a2) < 0)) {
              a2 = b1;
              h2 = true;
            }
          }
          const DD score = (topn == 1 || !h2) ? a1 : dd_add(a1, a2);
          if (lane == g) gd = score;
        }
        picked = 0;
        for (int r = 0; r < need; ++r) {
          const bool cand = ((band & ~picked) >> lane) & 1u;
          DD v = gd;
          int i = lane;
          warp_argmax_dd(v, i, cand);
          if (i < 0) return false;
          picked |= 1u << i;
        }
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
    int i = 0x7fffffff;
#pragma unroll 1
    for (int j = 0; j < MAXJ; ++j)
      if (((elig & ~taken) >> j) & 1u)
        if (key[j] > v || i == 0x7fffffff) { v = key[j]; i = j * 32 + lane; }
    warp_argmax(v, i);
    if (i == 0x7fffffff) return false;
#pragma unroll 1
    for (int j = 0; j < MAXJ; ++j)
      if (i == j * 32 + lane) taken |= 1u << j;
    vk = v;
  }
  const double tol = 2.0 * (double)key_tol(kmax, true);
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
    long long kx[MAXJ];
#pragma unroll 1
    for (int j = 0; j < MAXJ; ++j) {
      kx[j] = ORD_NONE;
      const bool mine = (band >> j) & 1u;
      if (__any_sync(FULL_MASK, mine) && mine) kx[j] = ord64(sigmoid_key64(u[j], b[j]));
    }
    long long v_cut = ORD_NONE, v_next = ORD_NONE;
    for (int r = 0; r <= need; ++r) {
      long long v = ORD_NONE;
      int i = 0x7fffffff;
#pragma unroll 1
      for (int j = 0; j < MAXJ; ++j)
        if (((band & ~picked) >> j) & 1u)
          if (kx[j] > v || i == 0x7fffffff) { v = kx[j]; i = j * 32 + lane; }
      warp_argmax_ord(v, i);
      if (r == need) { v_next = v; break; }
      if (i == 0x7fffffff) return false;
#pragma unroll 1
      for (int j = 0; j < MAXJ; ++j)
        if (i == j * 32 + lane) picked |= 1u << j;
      v_cut = v;
    }
    if (v_next != ORD_NONE && v_cut != ORD_NONE && near64(unord64(v_cut), unord64(v_next))) {
      // fp64 cannot settle the cut: real keys of the band experts in double-double
      DD kd[MAXJ];
#pragma unroll 1
      for (int j = 0; j < MAXJ; ++j) {
        kd[j] = DD{0.0, 0.0};
        const bool mine = (band >> j) & 1u;
        if (__any_sync(FULL_MASK, mine) && mine) kd[j] = dd_sigmoid_key(u[j], b[j]);
      }
      picked = 0;
      for (int r = 0; r < need; ++r) {
        // this lane's best remaining band expert (lowest index among real ties), then the warp's
        DD v = {0.0, 0.0};
        int i = -1;
#pragma unroll 1
        for (int j = 0; j < MAXJ; ++j)
          if (((band & ~picked) >> j) & 1u)
            if (i < 0 || dd_cmp(kd[j], v) < 0) { v = kd[j]; i = j * 32 + lane; }
        warp_argmax_dd(v, i, i >= 0);
        if (i < 0) return false;
#pragma unroll 1
        for (int j = 0; j < MAXJ; ++j)
          if (i == j * 32 + lane) picked |= 1u << j;
      }
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

// fp64 redo of one token (cold): scores and keys in fp64 from the logits ut and the bias, the
// choice by select_experts<double>. Lane r < K gets the r-th chosen expert in sel_e; false on an
// internal inconsistency. Reloads its inputs, so the caller's registers stay out of memory.
__device__ __noinline__ bool redo_fp64(const float* ut, const float* bias, bool sigmoid, int lane,
                                       int N, int K, int G, int Gk, int topn, int& sel_e) {
  const int J = (N + 31) >> 5;
  double u[MAXJ], kd[MAXJ];
  double umax = -INFINITY;
#pragma unroll
  for (int j = 0; j < MAXJ; ++j) {
    const int e = j * 32 + lane;
    u[j] = (j < J && e < N) ? (double)ut[e] : -INFINITY;
    umax = fmax(umax, u[j]);
  }
  umax = warp_max(umax);
  double z = 0.0;
  if (!sigmoid) {
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) z += (j < J && j * 32 + lane < N) ? exp(u[j] - umax) : 0.0;
    z = warp_sum(z);
  }
#pragma unroll
  for (int j = 0; j < MAXJ; ++j) {
    const int e = j * 32 + lane;
    const bool v = j < J && e < N;
    const double s = sigmoid ? 1.0 / (1.0 + exp(-u[j])) : exp(u[j] - umax) / z;
    kd[j] = v ? s + (bias != nullptr ? (double)bias[e] : 0.0) : neg_inf<double>();
  }
  const Selection sel = select_experts<double>(kd, lane, N, K, G, Gk, topn, J);
  sel_e = sel.e;
  return sel.ok;
}

// MINB: CTAs per SM the registers must allow. The calls to the exact recheck (rare: no token of
// the V3 prefill batch takes it) make the compiler size the kernel for the recheck's registers
// (123), two CTAs per SM; large batches, which need the warps to hide the loads, cap it at four
// CTAs (64 registers; the recheck spills, measured 61.6 -> 54.6 us at 16384 tokens), while small
// batches, where one warp's latency is the kernel's, keep the registers (8.0 vs 9.9 us at 512).
// JM: experts per lane, a compile-time bound on ceil(N / 32) (the launcher picks 2, 4, 5 or 8).
template <int MINB, int JM>
__global__ void __launch_bounds__(256, MINB) route_kernel(RouteArgs a) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int J = (a.N + 31) >> 5;
  const int gsz = a.N / a.G;
  const bool sigmoid = a.score_fn == 1;
  // Softmax with no selection bias and max-based (or no) group limit: the logits give the order.
  const bool logit_keys = !sigmoid && a.bias == nullptr && (a.G == 1 || a.topn == 1);

  pdl_wait();
  pdl_trigger();
  float b[JM];
  int gj[JM];
#pragma unroll
  for (int j = 0; j < JM; ++j) {
    const int e = j * 32 + lane;
    const bool v = j < J && e < a.N;
    b[j] = (a.bias != nullptr && v) ? a.bias[e] : 0.0f;
    gj[j] = v ? e / gsz : -1;
  }

  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < a.T; t += warps) {
    const float* ut = a.u + (size_t)t * a.N;
    float u[JM];
#pragma unroll
    for (int j = 0; j < JM; ++j) u[j] = gj[j] >= 0 ? ut[j * 32 + lane] : -INFINITY;
    // ---- fp32 scores and keys
    float s[JM];
    float umax = u[0];
#pragma unroll
    for (int j = 1; j < JM; ++j) umax = fmaxf(umax, u[j]);
    umax = warp_max(umax);
    if (sigmoid) {
#pragma unroll
      for (int j = 0; j < JM; ++j) s[j] = 1.0f / (1.0f + expf(-u[j]));
    } else {
      float z = 0.0f;
#pragma unroll
      for (int j = 0; j < JM; ++j) { s[j] = expf(u[j] - umax); z += s[j]; }
      z = warp_sum(z);
#pragma unroll
      for (int j = 0; j < JM; ++j) s[j] = s[j] / z;
    }
    uint32_t ok[JM];
    float kmax = 0.0f;
#pragma unroll
    for (int j = 0; j < JM; ++j) {
      const float key = logit_keys ? u[j] : s[j] + b[j];
      ok[j] = gj[j] >= 0 ? ord32(key) : 0u;
      if (gj[j] >= 0) kmax = fmaxf(kmax, fabsf(key));
    }

    const FastSel sel = fast_select(ok, s, gj, lane, a.K, a.G, a.Gk, a.topn);
    bool redo = !sel.ok;
    if (!logit_keys && !redo) {
      // A group score is the fp32 sum of its top-n keys: it is off by at most n key errors
      // (the n-th largest of perturbed values moves by at most the largest perturbation) plus
      // the rounding of the sum.
      kmax = warp_max(kmax);
      const float tol = key_tol(kmax, sigmoid);  // every key's error, whatever its size
      const float gtol = a.topn * tol + 6e-8f * fabsf(sel.gkth);
      redo = (double)sel.kth - (double)sel.next <= 2.0 * tol ||
             (a.G > a.Gk && (double)sel.gkth - (double)sel.gnext <= 2.0 * gtol);
    }
    int sel_e = sel.e;
    float sel_s = sel.se, ssum = sel.ssum;
    if (redo) {
      bool settled = false;
      if (sigmoid && sel.ok)  // rescore only the groups and experts within the error bound
        settled = refine_sigmoid(ut, a.bias, lane, a.N, a.K, a.G, a.Gk, a.topn, sel.gmask,
                                 sel.kth, sel_e);
      if (!settled && !redo_fp64(ut, a.bias, sigmoid, lane, a.N, a.K, a.G, a.Gk, a.topn, sel_e))
        set_error(a.err, ERR_DEVICE_CHECK);
      // scores of the chosen experts, from their owner lanes
      ssum = 0.0f;
      for (int r = 0; r < a.K; ++r) {
        const int e = __shfl_sync(FULL_MASK, sel_e, r);
        float mine = 0.0f;
#pragma unroll
        for (int j = 0; j < JM; ++j)
          if (e == j * 32 + lane) mine = s[j];
        const float v = __shfl_sync(FULL_MASK, mine, e & 31);
        if (lane == r) sel_s = v;
        ssum += v;
      }
    }

    // ---- weights
    float wv;
    if (a.precise_w) {
      // fp64 scores of the chosen experts, rounded once (the v2 drop ranks these values)
      double z = 0.0;
      if (!sigmoid) {
#pragma unroll
        for (int j = 0; j < JM; ++j)
          z += gj[j] >= 0 ? exp((double)u[j] - (double)umax) : 0.0;
        z = warp_sum(z);
      }
      // the logit of each chosen expert, from its owner lane
      float ul = 0.0f;
      for (int r = 0; r < a.K; ++r) {
        const int er = __shfl_sync(FULL_MASK, sel_e, r);
        float mine = 0.0f;
#pragma unroll
        for (int j = 0; j < JM; ++j)
          if (er == j * 32 + lane) mine = u[j];
        const float v = __shfl_sync(FULL_MASK, mine, er & 31);
        if (lane == r) ul = v;
      }
      const double sd = lane < a.K ? (sigmoid ? 1.0 / (1.0 + exp(-(double)ul))
                                              : exp((double)ul - (double)umax) / z)
                                   : 0.0;
      double wd = sd;
      if (a.norm_topk) wd = wd / warp_sum(sd);
      wv = (float)(wd * (double)a.scale);
    } else {
      float w32 = sel_s;
      if (a.norm_topk) w32 = w32 / ssum;
      wv = w32 * a.scale;
    }

    // ---- write in ascending expert order
    int rank = 0;
    for (int r = 0; r < a.K; ++r) {
      const int e = __shfl_sync(FULL_MASK, sel_e, r);
      if (lane < a.K && e < sel_e) ++rank;
    }
    if (lane < a.K) {
      const int e = (sel_e >= 0 && sel_e < a.N) ? sel_e : 0;
      a.idx[(size_t)t * a.K + rank] = e;
      a.w[(size_t)t * a.K + rank] = wv;
    }
  }
}

// ---------------------------------------------------------------- load statistics
// All in fp32: this part's fp64 throughput is a small fraction of its fp32 rate, and a reduction
// on one SM in fp64 cost more than the rest of the statistics together. Long sums are
// compensated (Kahan) and every sum has a fixed order, so the results are deterministic and far
// inside the 1e-5 relative accuracy the statistics are held to.
struct Kahan {
  float s = 0.0f, c = 0.0f;
  __device__ __forceinline__ void add(float v) {
    const float y = v - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
  }
};

// Per-block partial sums over the block's tokens (one warp per token, STATS_TOK_PER_WARP tokens
// each): the scores of every expert, lse and lse^2, and (with part_c) the assignment counts.
constexpr int STATS_TOK_PER_WARP = 2;
constexpr int STATS_THREADS = 256;
template <int JM>  // experts per lane (a compile-time bound on ceil(N / 32))
__global__ void __launch_bounds__(STATS_THREADS) stats_partial_kernel(StatsArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[8][256];
  __shared__ float redl[8][2];
  __shared__ int cnt[256];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int J = (a.N + 31) >> 5;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  if (a.part_c != nullptr)
    for (int e = threadIdx.x; e < 256; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  float acc[JM];
#pragma unroll
  for (int j = 0; j < JM; ++j) acc[j] = 0.0f;
  float l1 = 0.0f, l2 = 0.0f;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < a.T; t += warps) {
    const float* ut = a.u + (size_t)t * a.N;
    float u[JM];
#pragma unroll
    for (int j = 0; j < JM; ++j) {
      const int e = j * 32 + lane;
      u[j] = (j < J && e < a.N) ? ut[e] : -INFINITY;
    }
    if (a.part_c != nullptr && lane < a.K) {
      const int e = a.idx[(size_t)t * a.K + lane];
      if (e >= 0 && e < a.N) atomicAdd(&cnt[e], 1);
      else set_error(a.err, ERR_DEVICE_CHECK);
    }
    float m = u[0];
#pragma unroll
    for (int j = 1; j < JM; ++j) m = fmaxf(m, u[j]);
    m = warp_max(m);
    float ex[JM], z = 0.0f;
#pragma unroll
    for (int j = 0; j < JM; ++j) { ex[j] = expf(u[j] - m); z += ex[j]; }
    z = warp_sum(z);
    if (a.score_fn == 1) {
#pragma unroll
      for (int j = 0; j < JM; ++j)
        if (j < J && j * 32 + lane < a.N) acc[j] += 1.0f / (1.0f + expf(-u[j]));
    } else {
#pragma unroll
      for (int j = 0; j < JM; ++j) acc[j] += ex[j] / z;
    }
    const float lse = m + logf(z);
    l1 += lse;
    l2 += lse * lse;
  }
#pragma unroll
  for (int j = 0; j < JM; ++j) {
    const int e = j * 32 + lane;
    if (e < 256) red[wid][e] = (j < J && e < a.N) ? acc[j] : 0.0f;
  }
  if (lane == 0) { redl[wid][0] = l1; redl[wid][1] = l2; }
  __syncthreads();
  for (int e = threadIdx.x; e < a.N; e += blockDim.x) {
    float s = 0.0f;
    for (int w = 0; w < 8; ++w) s += red[w][e];
    a.part_s[(size_t)blockIdx.x * a.N + e] = s;
    if (a.part_c != nullptr) a.part_c[(size_t)blockIdx.x * a.N + e] = cnt[e];
  }
  if (threadIdx.x == 0) {
    float s1 = 0.0f, s2 = 0.0f;
    for (int w = 0; w < 8; ++w) { s1 += redl[w][0]; s2 += redl[w][1]; }
    a.part_lse[blockIdx.x * 2 + 0] = s1;
    a.part_lse[blockIdx.x * 2 + 1] = s2;
  }
}

// Sums of NV values over the 1024 threads of a block, each in a fixed order (a shuffle tree in
// every warp, then one over the 32 warp sums); every thread gets the results. sh: [32][NV].
template <int NV>
__device__ __forceinline__ void block_sums_1024(float (&v)[NV], float (*sh)[NV]) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[i] += __shfl_down_sync(FULL_MASK, v[i], o);
  }
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < NV; ++i) sh[wid][i] = v[i];
  }
  __syncthreads();
  if (wid == 0) {
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      float x = sh[lane][i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x += __shfl_down_sync(FULL_MASK, x, o);
      v[i] = x;
    }
    __syncwarp();
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < NV; ++i) sh[0][i] = v[i];
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < NV; ++i) v[i] = sh[0][i];
  __syncthreads();
}

// Fixed-order reduction of the partials: counts, f, P, L_B, L_Z, mean lse. Q = 1024 / N' threads
// share each expert's column of partials (N' = N rounded up to a power of two): thread (q, e)
// sums blocks q, q + Q, ... (compensated, eight loads in flight), then the Q sums of a column are
// added in the order q = 0 .. Q-1.
constexpr int STATS_FINAL_THREADS = 1024;
__global__ void __launch_bounds__(STATS_FINAL_THREADS) stats_final_kernel(StatsArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ float tree[STATS_FINAL_THREADS];
  __shared__ int ctree[STATS_FINAL_THREADS];
  int np2 = 1;
  while (np2 < a.N) np2 <<= 1;
  const int Q = STATS_FINAL_THREADS / np2;
  const int e = threadIdx.x % np2, q = threadIdx.x / np2;
  Kahan cs;
  int cc = 0;
  if (e < a.N) {
    for (int b0 = q; b0 < a.nblk; b0 += 8 * Q) {
      float v[8];
      int c[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int b = b0 + Q * j;
        v[j] = b < a.nblk ? a.part_s[(size_t)b * a.N + e] : 0.0f;
        c[j] = (b < a.nblk && a.part_c != nullptr) ? a.part_c[(size_t)b * a.N + e] : 0;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cs.add(v[j]);
        cc += c[j];
      }
    }
  }
  // lse sums: blocks strided over the threads (compensated), then a tree
  Kahan s1, s2;
  for (int b = threadIdx.x; b < a.nblk; b += STATS_FINAL_THREADS) {
    s1.add(a.part_lse[2 * b]);
    s2.add(a.part_lse[2 * b + 1]);
  }
  tree[threadIdx.x] = cs.s;
  ctree[threadIdx.x] = cc;
  __syncthreads();
  float colsum = 0.0f;
  int count = 0;
  if (q == 0 && e < a.N) {
    Kahan col;
    for (int i = 0; i < Q; ++i) {
      col.add(tree[i * np2 + e]);
      count += ctree[i * np2 + e];
    }
    colsum = col.s;
    if (a.part_c == nullptr) count = a.counts[e];
  }
  __syncthreads();
  // the column total and the two lse sums in one pass, then L_B's sum
  __shared__ float sums[32][3];
  float r3[3] = {q == 0 ? colsum : 0.0f, s1.s, s2.s};
  block_sums_1024<3>(r3, sums);
  const float total = r3[0], l1 = r3[1], l2 = r3[2];
  float fe = 0.0f, pe = 0.0f;
  if (q == 0 && e < a.N) {
    if (a.part_c != nullptr) a.counts[e] = count;
    fe = (float)count / ((float)a.T * (float)a.K);
    pe = colsum / total;
    if (a.f) a.f[e] = fe;
    if (a.P) a.P[e] = pe;
  }
  float r1[1] = {fe * pe};
  block_sums_1024<1>(r1, reinterpret_cast<float (*)[1]>(&sums[0][0]));
  const float lb = r1[0];
  if (threadIdx.x == 0 && a.lb_z) {
    a.lb_z[0] = lb * a.N;
    a.lb_z[1] = l2 / a.T;
    a.lb_z[2] = l1 / a.T;
  }
}

// Per token: expert counts, and one received token for each distinct device it uses.
__global__ void group_count_kernel(GroupLossArgs a) {
  pdl_wait();
  pdl_trigger();
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
  pdl_wait();
  pdl_trigger();
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

// The instantiation whose experts-per-lane bound JM covers ceil(N / 32) with the least waste.
template <int MINB>
cudaError_t launch_route_jm(const RouteArgs& a, dim3 grid, cudaStream_t st) {
  const int J = (a.N + 31) >> 5;
  if (J <= 2) return launch_pdl(route_kernel<MINB, 2>, grid, dim3(256), 0, st, a);
  if (J <= 4) return launch_pdl(route_kernel<MINB, 4>, grid, dim3(256), 0, st, a);
  if (J <= 5) return launch_pdl(route_kernel<MINB, 5>, grid, dim3(256), 0, st, a);
  return launch_pdl(route_kernel<MINB, 8>, grid, dim3(256), 0, st, a);
}
cudaError_t launch_stats_partial(const StatsArgs& a, dim3 grid, cudaStream_t st) {
  const int J = (a.N + 31) >> 5;
  if (J <= 2) return launch_pdl(stats_partial_kernel<2>, grid, dim3(STATS_THREADS), 0, st, a);
  if (J <= 4) return launch_pdl(stats_partial_kernel<4>, grid, dim3(STATS_THREADS), 0, st, a);
  if (J <= 5) return launch_pdl(stats_partial_kernel<5>, grid, dim3(STATS_THREADS), 0, st, a);
  return launch_pdl(stats_partial_kernel<8>, grid, dim3(STATS_THREADS), 0, st, a);
}

cudaError_t launch_group_losses(const GroupLossArgs& a, cudaStream_t st) {
  if (a.st.T <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(a.st.counts, 0, sizeof(int32_t) * a.st.N, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(a.recv, 0, sizeof(int32_t) * a.G, st);
  if (e != cudaSuccess) return e;
  int cb = (a.st.T + 255) / 256;
  if (cb > 1184) cb = 1184;
  e = launch_pdl(group_count_kernel, dim3(cb), dim3(256), 0, st, a);
  if (e == cudaSuccess) e = launch_stats_partial(a.st, dim3(a.st.nblk), st);
  if (e == cudaSuccess) e = launch_pdl(group_final_kernel, dim3(1), dim3(256), 0, st, a);
  return e;
}

constexpr int kRouteWideMinTokens = 1024;  // batches above this use route_kernel<4, *>

cudaError_t launch_route(const RouteArgs& a, int num_sms, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  const int warps_needed = a.T;
  int blocks = (warps_needed + 7) / 8;
  const int cap = num_sms * 8;
  if (blocks > cap) blocks = cap;
  return a.T > kRouteWideMinTokens ? launch_route_jm<4>(a, dim3(blocks), st)
                                   : launch_route_jm<1>(a, dim3(blocks), st);
}

int stats_blocks(int T) {
  int b = (T + 8 * STATS_TOK_PER_WARP - 1) / (8 * STATS_TOK_PER_WARP);  // 8 warps per block
  if (b < 1) b = 1;
  if (b > 1184) b = 1184;
  return b;
}

cudaError_t launch_stats(const StatsArgs& a, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  cudaError_t e = launch_stats_partial(a, dim3(a.nblk), st);
  if (e == cudaSuccess)
    e = launch_pdl(stats_final_kernel, dim3(1), dim3(STATS_FINAL_THREADS), 0, st, a);
  return e;
}

}  // namespace moe
