// Oracle: a plain, slow fp64 CPU statement of the DeepSeekMoE layer forward.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the library path may call this file; only the tests,
// the package's smoke check and the benchmark's CPU-baseline leg do. It shares no code,
// header, table or constant with the CUDA kernels: it is written from the pages' definitions.
//
// Sources (page title, section):
//   [P3] "DeepSeek MoE：从v1到v3的演进" (wln20.github.io)
//        - ST-MoE: auxiliary load-balance loss (f_i, P_i, L_B) and the router Z-loss L_Z
//        - DeepSeek-v1: fine-grained expert segmentation, shared-expert isolation
//        - DeepSeek-v2: device-limited routing (M devices), device-level token drop
//        - DeepSeek-v3: sigmoid gate, selection-only bias b_i (auxiliary-loss-free balancing)
//   [P4] "DeepSeek-V3的Group-Limited Expert Routing与负载均衡优化实践" (mhpn.cn)
//        - sections 1 and 3: 8 groups of 32 experts, keep the best 4 groups, pick 8 experts
//          among their 128; scores viewed per group, top groups chosen, the rest masked.
//   [P2] "从零构建DeepSeekMoE" (opc.csdn.net), section 2.2: layer output = shared experts'
//        sum + routed experts' weighted sum.
//
// Readings where the pages are silent or garbled are listed at each function.
// Everything is fp64 with plain loops; OpenMP only splits independent tokens / rows.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include <quadmath.h>

extern "C" {

// Layer shape and routing rule. (Own definition: the oracle includes no library header.)
typedef struct {
  int T, H, N;          // tokens, hidden size, routed experts
  int G, Gk;            // groups (or virtual devices) and how many a token may use
  int K;                // routed experts per token
  int topn;             // group score = sum of the group's top-`topn` selection scores
  int score_fn;         // 0 = softmax over all N, 1 = sigmoid per expert
  int norm_topk;        // 1 = divide the K weights by their sum
  double routed_scale;  // routed weights are multiplied by this
  int S, I;             // shared experts, intermediate size of one expert
  int capacity_drop;    // 1 = v2 device-level token drop
} oracle_cfg;

int oracle_abi_version(void) { return 2; }

// Router linear: u[t,e] = sum_h x[t,h] * Wg[e,h] + gb[e]   ([P2] section 5.2 router = nn.Linear)
void oracle_gate_logits(int T, int H, int N, const double* x, const double* wg, const double* gb,
                        double* u) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < N; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h) acc += x[(size_t)t * H + h] * wg[(size_t)e * H + h];
      u[(size_t)t * N + e] = acc + (gb ? gb[e] : 0.0);
    }
}

// Gate scores. [P3] DeepSeek-v3 "Softmax->Sigmoid": v1/v2 normalise with a softmax over all
// experts; v3 scores every expert independently with a sigmoid.
void oracle_scores(int T, int N, int score_fn, const double* u, double* s) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const double* ut = u + (size_t)t * N;
    double* st = s + (size_t)t * N;
    if (score_fn == 1) {
      for (int e = 0; e < N; ++e) st[e] = 1.0 / (1.0 + std::exp(-ut[e]));
    } else {
      double m = ut[0];
      for (int e = 1; e < N; ++e) m = std::max(m, ut[e]);
      double z = 0.0;
      for (int e = 0; e < N; ++e) z += std::exp(ut[e] - m);
      for (int e = 0; e < N; ++e) st[e] = std::exp(ut[e] - m) / z;
    }
  }
}

// Routing of one token from its scores s[N] and the selection bias b[N] (may be NULL).
//
// [P3] DeepSeek-v3: the top-K choice uses s_i + b_i; the gate weight stays s_i.
// [P4] sections 1 and 3: experts form G groups of N/G (group g = experts g*N/G .. (g+1)*N/G-1);
//      every group gets a score, the best Gk groups are kept and the others are masked out;
//      the final K experts are taken from the kept groups.
// [P3] DeepSeek-v2: the M devices holding the highest-scoring experts are chosen, then the
//      top-K over all experts on them. This is the same procedure with the group score equal
//      to the group's best expert score (topn = 1).
//
// Readings (the pages leave these open):
//   * group score = sum of the group's `topn` highest keys s_i + b_i, summed from largest down;
//   * experts outside the kept groups are excluded outright (not given score zero), so a
//     negative biased key can never pull in an expert from a dropped group;
//   * ties: higher key first, then the lower group / expert index;
//   * weights: w = s_e; if norm_topk, divided by the sum over the K chosen; times routed_scale;
//   * the K chosen experts are written in ascending expert index (the set is what is defined).
// margin_out (nullable) gets min(k-th key - (k+1)-th eligible key, Gk-th group score -
// (Gk+1)-th group score); +inf where no competitor exists.
// Keys of one token: fp64 values, and on demand their values in quad precision (__float128)
// from the logits, used to decide comparisons that fp64 cannot.
//
// What the method defines is the order of the real numbers key_e = s_e + b_e (and of group scores,
// sums of real keys). fp64 evaluation carries a few units in the last place of error (exp, the
// divisions and sums), so two keys closer than that may compare either way in fp64 depending on
// the exp implementation. Here two values are compared in fp64 when their fp64 values differ by
// more than kNear * max(1, |a|, |b|) (far above the fp64 error, so the fp64 order is the real
// order); otherwise in quad precision (relative error ~1e-33), where values within
// kTieRel * max(|a|, |b|) of each other count as equal (equal real numbers, e.g.
// sigmoid(u) + sigmoid(-u) = 1, do not come out exactly equal in any finite precision) and the
// lower index wins, like exact ties. Without logits the fp64 values decide alone.
constexpr double kNear = 1e-14;
constexpr double kTieRel = 0x1p-80;

struct TokenKeys {
  const oracle_cfg* c;
  const double* u;     // logits of the token (nullable)
  const double* b;     // selection bias (nullable)
  std::vector<double> key;
  std::vector<__float128> qkey;
  std::vector<char> has_q;

  TokenKeys(const oracle_cfg* cfg, const double* st, const double* ut, const double* bias)
      : c(cfg), u(ut), b(bias), key(cfg->N), qkey(cfg->N), has_q(cfg->N, 0) {
    for (int e = 0; e < c->N; ++e) key[e] = st[e] + (b ? b[e] : 0.0);
  }
  // key_e in quad precision: sigmoid(u) or softmax(u) (max-subtracted), plus the bias
  __float128 q(int e) {
    if (!has_q[e]) {
      __float128 s;
      if (c->score_fn == 1) {
        s = 1 / (1 + expq(-(__float128)u[e]));
      } else {
        double m = u[0];
        for (int j = 1; j < c->N; ++j) m = std::max(m, u[j]);
        __float128 z = 0;
        for (int j = 0; j < c->N; ++j) z += expq((__float128)u[j] - (__float128)m);
        s = expq((__float128)u[e] - (__float128)m) / z;
      }
      qkey[e] = s + (__float128)(b ? b[e] : 0.0);
      has_q[e] = 1;
    }
    return qkey[e];
  }
};

// -1 if a comes first (larger), +1 if b does, 0 if equal (then the caller breaks the tie by
// index). fa / fb: fp64 values; qa / qb: their quad values, computed only when needed.
}  // extern "C"
template <typename QA, typename QB>
static int compare_values(double fa, double fb, bool refine, QA qa, QB qb) {
  if (!refine || std::fabs(fa - fb) > kNear * std::max({1.0, std::fabs(fa), std::fabs(fb)}))
    return fa > fb ? -1 : (fa < fb ? 1 : 0);
  const __float128 a = qa(), b = qb();
  const __float128 tie = (__float128)kTieRel * fmaxq(fabsq(a), fabsq(b));
  if (a - b > tie) return -1;
  if (b - a > tie) return 1;
  return 0;
}

extern "C" {
static void route_one(const oracle_cfg* c, const double* st, const double* ut, const double* b,
                      int32_t* idx, double* w, double* margin_out) {
  const int N = c->N, G = c->G, Gk = c->Gk, K = c->K, gs = c->N / c->G;
  TokenKeys tk(c, st, ut, b);
  const std::vector<double>& key = tk.key;
  const bool refine = ut != nullptr;
  auto key_before = [&](int a, int bb) {
    const int r = compare_values(key[a], key[bb], refine, [&] { return tk.q(a); },
                                 [&] { return tk.q(bb); });
    return r != 0 ? r < 0 : a < bb;
  };

  // group scores: the sum of the group's topn largest keys (largest first)
  std::vector<double> gscore(G);
  std::vector<std::vector<int>> gtop(G);
  for (int g = 0; g < G; ++g) {
    std::vector<int> v(gs);
    for (int j = 0; j < gs; ++j) v[j] = g * gs + j;
    std::sort(v.begin(), v.end(), key_before);
    double acc = 0.0;
    for (int j = 0; j < c->topn && j < gs; ++j) {
      acc += key[v[j]];
      gtop[g].push_back(v[j]);
    }
    gscore[g] = acc;
  }
  auto gscore_q = [&](int g) {
    __float128 acc = 0;
    for (int e : gtop[g]) acc += tk.q(e);
    return acc;
  };
  std::vector<int> gorder(G);
  for (int g = 0; g < G; ++g) gorder[g] = g;
  std::sort(gorder.begin(), gorder.end(), [&](int a, int bb) {
    const int r = compare_values(gscore[a], gscore[bb], refine, [&] { return gscore_q(a); },
                                 [&] { return gscore_q(bb); });
    return r != 0 ? r < 0 : a < bb;
  });
  std::vector<char> gkeep(G, 0);
  for (int j = 0; j < Gk; ++j) gkeep[gorder[j]] = 1;

  // final top-K among experts of kept groups
  std::vector<int> cand;
  for (int e = 0; e < N; ++e)
    if (gkeep[e / gs]) cand.push_back(e);
  std::sort(cand.begin(), cand.end(), key_before);
  std::vector<int> chosen(cand.begin(), cand.begin() + K);
  std::sort(chosen.begin(), chosen.end());

  double denom = 0.0;
  for (int j = 0; j < K; ++j) denom += st[chosen[j]];
  for (int j = 0; j < K; ++j) {
    idx[j] = chosen[j];
    double wj = st[chosen[j]];
    if (c->norm_topk) wj = wj / denom;
    w[j] = wj * c->routed_scale;
  }
  if (margin_out) {
    double m = INFINITY;
    if ((int)cand.size() > K) m = std::min(m, key[cand[K - 1]] - key[cand[K]]);
    if (G > Gk) m = std::min(m, gscore[gorder[Gk - 1]] - gscore[gorder[Gk]]);
    *margin_out = m;
  }
}

// u (nullable): the logits the scores came from; with them, near ties are decided by the real
// order of the keys (see TokenKeys), without them by the fp64 scores alone.
void oracle_route(const oracle_cfg* c, const double* s, const double* u, const double* sel_bias,
                  int32_t* idx, double* w, double* margin) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < c->T; ++t)
    route_one(c, s + (size_t)t * c->N, u ? u + (size_t)t * c->N : nullptr, sel_bias,
              idx + (size_t)t * c->K, w + (size_t)t * c->K, margin ? margin + t : nullptr);
}

// [P3] ST-MoE auxiliary load-balance loss and router Z-loss over a batch of T tokens.
//   counts[e] = number of (token, slot) assignments to expert e
//   f[e]      = counts[e] / (T K)   fraction of the batch's assignments that went to e
//   P[e]      = sum_t s[t,e] / sum_t sum_j s[t,j]  share of all router score given to e
//   L_B       = N * sum_e f[e] P[e]
//   lse_t     = log sum_j exp(u[t,j]);  L_Z = (1/T) sum_t lse_t^2;  also (1/T) sum_t lse_t
// Readings: the page's f_i is a per-token count (sums to K) while its stated minimum 1/N and
// L_B = 1 under uniform routing need f to sum to 1, so f is the fraction of assignments.
// P_i follows the page's wording (score share of the total), which equals the (1/T) sum of
// probabilities for a softmax gate. The Z-loss formula lost its square in extraction; the
// squared log-sum-exp is used and the plain mean is reported beside it.
void oracle_load_stats(const oracle_cfg* c, const double* u, const double* s, const int32_t* idx,
                       int64_t* counts, double* f, double* P, double* out3) {
  const int T = c->T, N = c->N, K = c->K;
  for (int e = 0; e < N; ++e) counts[e] = 0;
  for (size_t a = 0; a < (size_t)T * K; ++a) counts[idx[a]] += 1;
  std::vector<double> col(N, 0.0);
  double total = 0.0;
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < N; ++e) {
      col[e] += s[(size_t)t * N + e];
      total += s[(size_t)t * N + e];
    }
  double lb = 0.0;
  for (int e = 0; e < N; ++e) {
    f[e] = (double)counts[e] / ((double)T * K);
    P[e] = col[e] / total;
    lb += f[e] * P[e];
  }
  lb *= N;
  double z2 = 0.0, z1 = 0.0;
  for (int t = 0; t < T; ++t) {
    const double* ut = u + (size_t)t * N;
    double m = ut[0];
    for (int e = 1; e < N; ++e) m = std::max(m, ut[e]);
    double acc = 0.0;
    for (int e = 0; e < N; ++e) acc += std::exp(ut[e] - m);
    double lse = m + std::log(acc);
    z2 += lse * lse;
    z1 += lse;
  }
  out3[0] = lb;
  out3[1] = z2 / T;
  out3[2] = z1 / T;
}

// [P3] DeepSeek-v2 device-level token drop: C = the average number of assignments a device
// receives; a device receiving T_d > C keeps its C highest-scored and drops the rest.
// Readings: D = G virtual devices, device(e) = e / (N/G); one unit is one (token, slot)
// assignment; C = ceil(T K / D); the score ranked is the routing weight w, compared as its
// correctly rounded fp32 value (the precision the kernels keep weights in, so both sides
// take this integer decision in the same precision); ties keep the lower token index, then
// the lower slot. kept[a] = 1 / 0.
void oracle_capacity_drop(const oracle_cfg* c, const int32_t* idx, const double* w,
                          uint8_t* kept) {
  const int T = c->T, K = c->K, D = c->G, per = c->N / c->G;
  const long long A = (long long)T * K;
  const long long C = (A + D - 1) / D;
  for (long long a = 0; a < A; ++a) kept[a] = 1;
  for (int d = 0; d < D; ++d) {
    std::vector<long long> mine;
    for (long long a = 0; a < A; ++a)
      if (idx[a] / per == d) mine.push_back(a);
    if ((long long)mine.size() <= C) continue;
    std::sort(mine.begin(), mine.end(), [&](long long a, long long bb) {
      const float wa = (float)w[a], wb = (float)w[bb];  // round to nearest even
      if (wa != wb) return wa > wb;
      return a < bb;  // a = t*K + k: lower token first, then lower slot
    });
    for (size_t j = (size_t)C; j < mine.size(); ++j) kept[mine[j]] = 0;
  }
}

// Token permutation by expert (the dispatch that expert parallelism implies, [P3] GShard EP,
// [P4] section 5 all-to-all). Kept assignments are grouped into one contiguous segment per
// expert, experts in ascending order, rows inside a segment in ascending token order.
//   offsets[N+1]  exclusive scan of kept counts
//   row_token[R]  token of each row
//   slot_row[T*K] row of assignment (t,k), or -1 when dropped
void oracle_permute(const oracle_cfg* c, const int32_t* idx, const uint8_t* kept,
                    int32_t* offsets, int32_t* row_token, int32_t* slot_row) {
  const int T = c->T, K = c->K, N = c->N;
  std::vector<long long> cnt(N, 0);
  for (long long a = 0; a < (long long)T * K; ++a)
    if (!kept || kept[a]) cnt[idx[a]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < N; ++e) offsets[e + 1] = offsets[e] + (int32_t)cnt[e];
  for (long long a = 0; a < (long long)T * K; ++a) slot_row[a] = -1;
  for (int e = 0; e < N; ++e) {
    int32_t r = offsets[e];
    for (int t = 0; t < T; ++t)
      for (int k = 0; k < K; ++k) {
        long long a = (long long)t * K + k;
        if (idx[a] == e && (!kept || kept[a])) {
          row_token[r] = t;
          slot_row[a] = r;
          ++r;
        }
      }
  }
}

// One expert FFN over n rows. SwiGLU reading (the pages show only fc1/fc2): with W13 holding
// the gate projection in rows 0..I-1 and the up projection in rows I..2I-1,
//   a = x W13[0:I]^T,  g = x W13[I:2I]^T,  h = a * sigmoid(a) * g,  y = h W2^T.
// Fine-grained segmentation ([P3] DeepSeek-v1, [P2] section 2.1) only changes I and K.
// Weights are read through widen(): double as is, bf16 bit patterns exactly to double.
// OpenMP splits the independent output features.
}  // extern "C"
static inline double widen(double v) { return v; }
static inline double widen(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, sizeof(f));
  return (double)f;
}
template <typename E>
static void swiglu_rows_impl(int n, int H, int I, const double* x, const E* w13, const E* w2,
                             double* y) {
  std::vector<double> hbuf((size_t)n * I);
  for (int r = 0; r < n; ++r) {
    const double* xr = x + (size_t)r * H;
#pragma omp parallel for schedule(static)
    for (int j = 0; j < I; ++j) {
      double a = 0.0, g = 0.0;
      for (int h = 0; h < H; ++h) {
        a += xr[h] * widen(w13[(size_t)j * H + h]);
        g += xr[h] * widen(w13[(size_t)(I + j) * H + h]);
      }
      hbuf[(size_t)r * I + j] = a / (1.0 + std::exp(-a)) * g;
    }
#pragma omp parallel for schedule(static)
    for (int o = 0; o < H; ++o) {
      double acc = 0.0;
      for (int j = 0; j < I; ++j) acc += hbuf[(size_t)r * I + j] * widen(w2[(size_t)o * I + j]);
      y[(size_t)r * H + o] = acc;
    }
  }
}
extern "C" {

void oracle_swiglu_rows(int n, int H, int I, const double* x, const double* w13,
                        const double* w2, double* y) {
  swiglu_rows_impl(n, H, I, x, w13, w2, y);
}

// Same, with the weights given as bf16 bit patterns.
void oracle_swiglu_rows_bf16w(int n, int H, int I, const double* x, const uint16_t* w13,
                              const uint16_t* w2, double* y) {
  swiglu_rows_impl(n, H, I, x, w13, w2, y);
}

// Layer output ([P2] section 2.2 forward: shared experts' sum plus routed experts' output;
// [P3] DeepSeek-v1 shared-expert isolation):
//   out[t] = sum_k kept(t,k) w[t,k] y[slot_row(t,k)] + y_shared[t]
// y_rows holds one row per kept assignment (indexed through slot_row); y_shared may be NULL.
void oracle_combine(int T, int H, int K, const double* y_rows, const int32_t* slot_row,
                    const double* w, const double* y_shared, double* out) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k) {
        int32_t r = slot_row[(size_t)t * K + k];
        if (r >= 0) acc += w[(size_t)t * K + k] * y_rows[(size_t)r * H + h];
      }
      if (y_shared) acc += y_shared[(size_t)t * H + h];
      out[(size_t)t * H + h] = acc;
    }
}

// [P3] DeepSeek-v3 auxiliary-loss-free balancing: e_i = mean(c) - c_i; b_i += u * sign(e_i).
void oracle_bias_update(int N, const int64_t* counts, double rate, double* b) {
  double mean = 0.0;
  for (int e = 0; e < N; ++e) mean += (double)counts[e];
  mean /= N;
  for (int e = 0; e < N; ++e) {
    double err = mean - (double)counts[e];
    double sg = err > 0 ? 1.0 : (err < 0 ? -1.0 : 0.0);
    b[e] += rate * sg;
  }
}

}  // extern "C"
