// C ABI of the library (declared in include/moe.h): argument checks, workspace carving and
// the order of launches. No device memory is allocated here; every launch goes on the
// caller's stream.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <new>

#include "../../include/moe.h"
#include "common.cuh"
#include "internal.h"

using namespace moe;

namespace {

thread_local char g_detail[256] = "";

moe_status fail(moe_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
  va_end(ap);
  return s;
}

// Per-device error word (one int per device that has used the library).
__device__ int g_error_word[1];

std::mutex g_symbol_mutex;

int* error_word() {
  static moe::SymbolCache cache;
  std::lock_guard<std::mutex> lock(g_symbol_mutex);
  return static_cast<int*>(cache.get(g_error_word));
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) n = 148;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_cfg(const moe_config* c, int32_t T) {
  if (c == nullptr) return fail(MOE_ERR_INVALID_ARG, "cfg is NULL");
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T=%d < 0", T);
  if (c->hidden <= 0 || c->inter <= 0 || c->n_routed <= 0 || c->top_k <= 0 || c->n_shared < 0)
    return fail(MOE_ERR_INVALID_ARG, "non-positive size in config");
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16)
    return fail(MOE_ERR_INVALID_ARG, "dtype %d", c->dtype);
  if (c->score_fn != MOE_SOFTMAX && c->score_fn != MOE_SIGMOID)
    return fail(MOE_ERR_INVALID_ARG, "score_fn %d", c->score_fn);
  if (c->n_groups <= 0 || c->n_routed % c->n_groups != 0)
    return fail(MOE_ERR_INVALID_ARG, "n_groups=%d must divide n_routed=%d", c->n_groups,
                c->n_routed);
  if (c->topk_groups <= 0 || c->topk_groups > c->n_groups)
    return fail(MOE_ERR_INVALID_ARG, "topk_groups=%d not in [1, n_groups=%d]", c->topk_groups,
                c->n_groups);
  const int gsz = c->n_routed / c->n_groups;
  if (c->top_k > c->topk_groups * gsz)
    return fail(MOE_ERR_INVALID_ARG, "top_k=%d exceeds the experts of %d groups (%d)", c->top_k,
                c->topk_groups, c->topk_groups * gsz);
  if (c->group_score_topn < 1 || c->group_score_topn > gsz)
    return fail(MOE_ERR_INVALID_ARG, "group_score_topn=%d not in [1, %d]", c->group_score_topn,
                gsz);
  if (!(c->routed_scale > 0.0f) || !std::isfinite(c->routed_scale))
    return fail(MOE_ERR_INVALID_ARG, "routed_scale must be finite and > 0");
  if (c->n_routed > 256) return fail(MOE_ERR_UNSUPPORTED, "n_routed=%d > 256", c->n_routed);
  if (c->top_k > 16) return fail(MOE_ERR_UNSUPPORTED, "top_k=%d > 16", c->top_k);
  if (c->n_groups > 32) return fail(MOE_ERR_UNSUPPORTED, "n_groups=%d > 32", c->n_groups);
  if (c->group_score_topn > 2)
    return fail(MOE_ERR_UNSUPPORTED, "group_score_topn=%d > 2", c->group_score_topn);
  if ((long long)T * c->top_k > 0x7fffffffLL)
    return fail(MOE_ERR_UNSUPPORTED, "T*top_k overflows int32");
  if (c->dtype == MOE_BF16) {
    if (c->hidden % 64 != 0)
      return fail(MOE_ERR_UNSUPPORTED, "bf16 path needs hidden %% 64 == 0 (hidden=%d)", c->hidden);
    if (c->inter % 128 != 0)
      return fail(MOE_ERR_UNSUPPORTED, "bf16 path needs inter %% 128 == 0 (inter=%d)", c->inter);
  } else {
    if (c->hidden % 4 != 0)
      return fail(MOE_ERR_UNSUPPORTED, "f32 path needs hidden %% 4 == 0 (hidden=%d)", c->hidden);
  }
  return MOE_OK;
}

size_t align_up(size_t v) { return (v + 255) & ~(size_t)255; }

// Largest batch whose routed rows the layer's up projection gathers from x (see layer_steps).
constexpr int32_t kGatherMaxTokens = 32;

// Workspace carve for one config and token count. Every region is 256-byte aligned.
struct Layout {
  size_t u, idx, w, offsets, slot_row, row_token, masks, cnt, base, thr, part_s, part_c, part_lse,
      counts, recv, seq_s, seq_c, seq_lb, gate_part, sched, split_part, xy_perm, h, h_sh, y_sh,
      total;
};

Layout layout(const moe_config* c, int32_t T) {
  Layout L;
  const size_t N = c->n_routed, K = c->top_k, H = c->hidden, I = c->inter, S = c->n_shared;
  const size_t eb = c->dtype == MOE_BF16 ? 2 : 4;
  const size_t Tt = T > 0 ? (size_t)T : 1;
  const size_t A = Tt * K;
  const size_t nb = (size_t)permute_blocks((int)Tt);
  const size_t nbs = (size_t)stats_blocks((int)Tt);
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes); return at; };
  L.u = take(Tt * N * 4);
  L.idx = take(A * 4);
  L.w = take(A * 4);
  L.offsets = take((N + 1) * 4);
  L.slot_row = take(A * 4);
  L.row_token = take(A * 4);
  L.masks = take(nb * N * 8 * 4);
  L.cnt = take(nb * N * 4);
  L.base = take(nb * N * 4);
  L.thr = take((size_t)c->n_groups * 8);
  L.part_s = take(nbs * N * 4);
  L.part_c = take(nbs * N * 4);
  L.part_lse = take(nbs * 2 * 8);
  L.counts = take(N * 4);
  L.recv = take(32 * 4);
  // sequence-wise loss: B * chunks <= T / 64 + B <= T + T / 64 partial rows for any seq_len
  const size_t seq_rows = Tt + Tt / 64 + 1;
  L.seq_s = take(seq_rows * N * 4);
  L.seq_c = take(seq_rows * N * 4);
  L.seq_lb = take(Tt * 8);
  L.gate_part = take((size_t)GATE_PART_ROWS * N * 4);
  L.sched = take(kSchedInts * 4);  // tile and split counters of the up and down GEMMs
  L.split_part = take(c->dtype == MOE_BF16 ? kSplitMaxPieces * kSplitPieceFloats * 4 : 0);
  L.xy_perm = take(A * H * eb);   // x_perm, then reused for y_perm
  L.h = take(A * I * eb);
  L.h_sh = take(Tt * (S > 0 ? S : 1) * I * eb);
  L.y_sh = take(Tt * H * eb);
  L.total = o;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

moe_status check_ws(const moe_config* c, int32_t T, const void* ws, size_t ws_bytes) {
  const size_t need = layout(c, T).total;
  if (ws == nullptr) return fail(MOE_ERR_WORKSPACE, "ws is NULL (need %zu bytes)", need);
  if (ws_bytes < need) return fail(MOE_ERR_WORKSPACE, "ws_bytes=%zu < %zu", ws_bytes, need);
  if (!aligned16(ws)) return fail(MOE_ERR_INVALID_ARG, "ws not 16-byte aligned");
  return MOE_OK;
}

moe_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return MOE_OK;
  return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CHECK_PTR(p)                                                              \
  do {                                                                            \
    if ((p) == nullptr) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", #p);       \
    if (!aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "%s not 16-byte aligned", #p); \
  } while (0)
#define CHECK_ALIGN(p)                                                            \
  do {                                                                            \
    if ((p) != nullptr && !aligned16(p))                                          \
      return fail(MOE_ERR_INVALID_ARG, "%s not 16-byte aligned", #p);             \
  } while (0)

cudaStream_t S_(moe_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

#define TRY_S(expr)                       \
  do {                                    \
    moe_status _s = (expr);               \
    if (_s != MOE_OK) return _s;          \
  } while (0)

// ---------------------------------------------------------------- optional stage timing
// While active (moe_stage_timing_start .. _stop, one host thread), every moe_layer_forward
// records a CUDA event on its stream at each stage boundary, so that the time of each stage
// can be read back per call without synchronising inside the call.
enum { STAGE_GATE = 0, STAGE_ROUTE, STAGE_STATS, STAGE_PERMUTE, STAGE_DISPATCH, STAGE_UP,
       STAGE_DOWN, STAGE_COMBINE, N_STAGES };
static_assert(N_STAGES == MOE_N_STAGES, "stage list of the header");

struct StageTiming {
  bool on = false;
  int max_calls = 0;
  int calls = 0;        // forwards recorded so far
  int cur = -1;         // call being recorded, -1 = none
  cudaEvent_t* ev = nullptr;   // [max_calls][N_STAGES + 1]
};
StageTiming g_timing;

// Boundary b (the start of stage b; b == N_STAGES is the end of the call) of the current call.
// Under stream capture the record becomes an event-record node of the graph (it then records
// each time the graph runs).
void stage_mark(int b, cudaStream_t st) {
  if (!g_timing.on || g_timing.cur < 0) return;
  cudaEvent_t ev = g_timing.ev[(size_t)g_timing.cur * (N_STAGES + 1) + b];
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) == cudaSuccess && cap == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, st);
}

// ---------------------------------------------------------------- step implementations
moe_status do_gate(const moe_config* c, int32_t T, const void* x, const moe_weights* w, float* u,
                   void* ws, cudaStream_t st) {
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.mode = MODE_GATE;
  g.T = T; g.H = c->hidden; g.I = c->inter; g.S = c->n_shared; g.N = c->n_routed;
  g.a0 = x; g.b0 = w->w_gate; g.out0 = u; g.gate_bias = w->gate_logit_bias;
  if (ws != nullptr) {  // split-K scratch for few-token batches
    g.gate_part = at<float>(ws, layout(c, T).gate_part);
    g.gate_part_floats = (size_t)GATE_PART_ROWS * c->n_routed;
  }
  g.err = error_word();
  cudaError_t e = c->dtype == MOE_BF16 ? launch_gemm_tc(g, num_sms(), st) : launch_gemm_simt(g, st);
  return cuda_status(e, "gate GEMM");
}

moe_status do_route(const moe_config* c, int32_t T, const float* u, const moe_weights* w,
                    int32_t* idx, float* wt, cudaStream_t st) {
  RouteArgs r;
  r.T = T; r.N = c->n_routed; r.K = c->top_k; r.G = c->n_groups; r.Gk = c->topk_groups;
  r.topn = c->group_score_topn; r.score_fn = c->score_fn; r.norm_topk = c->norm_topk ? 1 : 0;
  r.precise_w = c->capacity_drop ? 1 : 0;
  r.scale = c->routed_scale;
  r.u = u; r.bias = w ? w->select_bias : nullptr;
  r.idx = idx; r.w = wt; r.err = error_word();
  return cuda_status(launch_route(r, num_sms(), st), "route");
}

moe_status do_stats(const moe_config* c, int32_t T, const float* u, const int32_t* idx,
                    int32_t* counts, float* f, float* P, float* lb_z, void* ws, cudaStream_t st) {
  const Layout L = layout(c, T);
  StatsArgs s;
  s.T = T; s.N = c->n_routed; s.K = c->top_k; s.score_fn = c->score_fn;
  s.u = u; s.idx = idx;
  s.counts = counts ? counts : at<int32_t>(ws, L.counts);
  s.f = f; s.P = P; s.lb_z = lb_z;
  s.part_s = at<float>(ws, L.part_s);
  s.part_c = at<int32_t>(ws, L.part_c);
  s.part_lse = at<float>(ws, L.part_lse);
  s.nblk = stats_blocks(T);
  s.err = error_word();
  return cuda_status(launch_stats(s, st), "load stats");
}

// x_perm == nullptr: the permutation only (no row copies; the up GEMM then gathers its rows).
moe_status do_permute(const moe_config* c, int32_t T, const int32_t* idx, const float* wt,
                      const void* x, int32_t* offsets, int32_t* row_token, float* row_w,
                      int32_t* slot_row,
                      void* x_perm, void* ws, cudaStream_t st, int32_t* sched_zero = nullptr) {
  const Layout L = layout(c, T);
  PermuteArgs p;
  p.T = T; p.N = c->n_routed; p.K = c->top_k; p.D = c->n_groups;
  p.capacity_drop = c->capacity_drop ? 1 : 0;
  p.idx = idx; p.w = wt; p.x = x; p.H = c->hidden; p.elem_bytes = c->dtype == MOE_BF16 ? 2 : 4;
  p.offsets = offsets; p.row_token = row_token; p.row_w = row_w; p.slot_row = slot_row;
  p.x_perm = x_perm;
  p.masks = at<uint32_t>(ws, L.masks);
  p.cnt = at<int32_t>(ws, L.cnt);
  p.base = at<int32_t>(ws, L.base);
  p.thr = at<unsigned long long>(ws, L.thr);
  p.sched_zero = sched_zero;
  p.err = error_word();
  TRY_S(cuda_status(launch_permute(p, num_sms(), st), "permute"));
  stage_mark(STAGE_DISPATCH, st);
  return cuda_status(launch_dispatch(p, num_sms(), st), "row dispatch");
}

// Zero the up and down GEMMs' tile and split counters in the workspace (one memset node per
// FFN).
moe_status reset_sched(const moe_config* c, int32_t T, void* ws, cudaStream_t st) {
  if (c->dtype != MOE_BF16) return MOE_OK;
  return cuda_status(cudaMemsetAsync(at<int32_t>(ws, layout(c, T).sched), 0,
                                     kSchedInts * sizeof(int32_t), st),
                     "tile counter reset");
}

// sched: the workspace's scheduling ints (tile counters of up and down, then their split
// counters), zeroed by reset_sched or the permutation, or nullptr (static schedule, no tail
// split). split_part: the workspace's split partial accumulators (used with sched).
// row_token != nullptr (bf16 only): the routed rows are gathered from x (x_perm unused).
// offsets_early: the offsets were written at least two kernels back in the stream (or before a
// memset node), so the GEMM builds its tile schedule before waiting for the kernel just ahead.
moe_status do_up(const moe_config* c, int32_t T, const void* x_perm, const int32_t* offsets,
                 const void* x, const moe_weights* w, void* h, void* h_sh, int32_t* sched,
                 float* split_part, cudaStream_t st, const int32_t* row_token = nullptr,
                 bool offsets_early = false) {
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.mode = MODE_UP;
  g.T = T; g.H = c->hidden; g.I = c->inter; g.S = c->n_shared; g.N = c->n_routed;
  g.n_routed = c->n_routed; g.has_shared = c->n_shared > 0 ? 1 : 0;
  g.offsets = offsets; g.rows_cap = T * c->top_k;
  g.a0 = row_token != nullptr ? x : x_perm; g.a1 = x; g.b0 = w->w13; g.b1 = w->w13_shared;
  g.out0 = h; g.out1 = h_sh; g.err = error_word();
  g.sched = sched;
  g.split_cnt = sched ? sched + 2 : nullptr;
  g.split_part = sched ? split_part : nullptr;
  g.row_token = row_token;
  g.offsets_early = offsets_early ? 1 : 0;
  cudaError_t e = c->dtype == MOE_BF16 ? launch_gemm_tc(g, num_sms(), st) : launch_gemm_simt(g, st);
  return cuda_status(e, "expert up GEMM");
}

moe_status do_down(const moe_config* c, int32_t T, const void* h, const int32_t* offsets,
                   const void* h_sh, const moe_weights* w, void* y, void* y_sh, int32_t* sched,
                   float* split_part, cudaStream_t st, bool offsets_early = false) {
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.mode = MODE_DOWN;
  g.T = T; g.H = c->hidden; g.I = c->inter; g.S = c->n_shared; g.N = c->n_routed;
  g.n_routed = c->n_routed; g.has_shared = c->n_shared > 0 ? 1 : 0;
  g.offsets = offsets; g.rows_cap = T * c->top_k;
  g.a0 = h; g.a1 = h_sh; g.b0 = w->w2; g.b1 = w->w2_shared;
  g.out0 = y; g.out1 = y_sh; g.err = error_word();
  g.sched = sched ? sched + 1 : nullptr;
  g.split_cnt = sched ? sched + 2 + kSplitCounters : nullptr;
  g.split_part = sched ? split_part : nullptr;
  g.offsets_early = offsets_early ? 1 : 0;
  cudaError_t e = c->dtype == MOE_BF16 ? launch_gemm_tc(g, num_sms(), st) : launch_gemm_simt(g, st);
  return cuda_status(e, "expert down GEMM");
}

moe_status do_combine(const moe_config* c, int32_t T, const void* y, const int32_t* slot_row,
                      const float* wt, const void* y_sh, void* out, cudaStream_t st) {
  CombineArgs a;
  a.T = T; a.H = c->hidden; a.K = c->top_k; a.dtype = c->dtype;
  a.y = y; a.slot_row = slot_row; a.w = wt; a.ys = y_sh; a.out = out;
  a.rows = T * c->top_k;
  a.err = error_word();
  return cuda_status(launch_combine(a, num_sms(), st), "combine");
}

moe_status check_weights(const moe_config* c, const moe_weights* w, bool need_gate,
                         bool need_experts) {
  if (w == nullptr) return fail(MOE_ERR_INVALID_ARG, "weights is NULL");
  if (need_gate) CHECK_PTR(w->w_gate);
  CHECK_ALIGN(w->gate_logit_bias);
  CHECK_ALIGN(w->select_bias);
  if (need_experts) {
    CHECK_PTR(w->w13);
    CHECK_PTR(w->w2);
    if (c->n_shared > 0) {
      CHECK_PTR(w->w13_shared);
      CHECK_PTR(w->w2_shared);
    }
  }
  return MOE_OK;
}

#define TRY(expr)                         \
  do {                                    \
    moe_status _s = (expr);               \
    if (_s != MOE_OK) return _s;          \
  } while (0)

// The whole layer on `st`, intermediates carved from `ws` (arguments already checked).
moe_status layer_steps(const moe_config* cfg, int32_t T, const void* x, const moe_weights* w,
                       void* out, int32_t* counts, float* lb_z, void* ws, cudaStream_t st) {
  const Layout L = layout(cfg, T);
  float* u = at<float>(ws, L.u);
  int32_t* idx = at<int32_t>(ws, L.idx);
  float* wt = at<float>(ws, L.w);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* slot_row = at<int32_t>(ws, L.slot_row);
  int32_t* row_token = at<int32_t>(ws, L.row_token);
  void* xy = at<char>(ws, L.xy_perm);
  void* h = at<char>(ws, L.h);
  void* h_sh = cfg->n_shared > 0 ? at<char>(ws, L.h_sh) : nullptr;
  void* y_sh = cfg->n_shared > 0 ? at<char>(ws, L.y_sh) : nullptr;

  stage_mark(STAGE_GATE, st);
  TRY(do_gate(cfg, T, x, w, u, ws, st));
  stage_mark(STAGE_ROUTE, st);
  TRY(do_route(cfg, T, u, w, idx, wt, st));
  stage_mark(STAGE_STATS, st);
  if (counts != nullptr || lb_z != nullptr)
    TRY(do_stats(cfg, T, u, idx, counts, nullptr, nullptr, lb_z, ws, st));
  // Batches of at most 32 tokens (bf16): every expert segment has at most 32 rows, and the up
  // GEMM gathers them straight from x through row_token (tile::gather4 loads) at the speed of
  // contiguous loads, so the x_perm copy is skipped (the dispatch stage stays empty). Larger
  // segments load contiguous x_perm rows: a row gather issues one load per four rows, and with
  // hundreds of token rows per tile those loads, not the memory, bound the GEMM.
  const bool gather = cfg->dtype == MOE_BF16 && T <= kGatherMaxTokens;
  // the permutation also zeroes the expert GEMMs' tile counters (no memset between the kernels,
  // so each kernel can start while the one ahead of it finishes)
  int32_t* sched = at<int32_t>(ws, L.sched);
  stage_mark(STAGE_PERMUTE, st);
  TRY(do_permute(cfg, T, idx, wt, x, offsets, row_token, nullptr, slot_row,
                 gather ? nullptr : xy, ws, st, sched));
  stage_mark(STAGE_UP, st);
  float* split_part = at<float>(ws, L.split_part);
  // the up GEMM follows the permutation directly when it gathers, else the dispatch; the down
  // GEMM follows the up GEMM
  TRY(do_up(cfg, T, xy, offsets, x, w, h, h_sh, sched, split_part, st,
            gather ? row_token : nullptr, /*offsets_early=*/!gather));
  stage_mark(STAGE_DOWN, st);
  TRY(do_down(cfg, T, h, offsets, h_sh, w, xy, y_sh, sched, split_part, st,
              /*offsets_early=*/true));  // y_perm overwrites x_perm
  stage_mark(STAGE_COMBINE, st);
  return do_combine(cfg, T, xy, slot_row, wt, y_sh, out, st);
}

}  // namespace

// Accessors for other entry-point files of this library (same checks, same error reporting).
namespace moe {

uintptr_t current_context() {
  using Fn = CUresult (*)(CUcontext*);
  static const Fn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<Fn>(p);
    return static_cast<Fn>(nullptr);
  }();
  CUcontext ctx = nullptr;
  if (fn == nullptr || fn(&ctx) != CUDA_SUCCESS) return 0;
  return reinterpret_cast<uintptr_t>(ctx);
}

namespace {
std::atomic<unsigned long long> g_launches{0};
}
void note_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }
moe_status abi_check_config(const moe_config* c, int32_t T) {
  g_detail[0] = 0;
  return check_cfg(c, T);
}
moe_status abi_fail(moe_status s, const char* msg) { return fail(s, "%s", msg); }
moe_status abi_cuda_status(cudaError_t e, const char* what) { return cuda_status(e, what); }
int* abi_error_word() { return error_word(); }
int abi_num_sms() { return num_sms(); }
}  // namespace moe

// ==================================================================== exported entry points
extern "C" {

size_t moe_workspace_size(const moe_config* cfg, int32_t T) {
  if (check_cfg(cfg, T) != MOE_OK) return 0;
  return layout(cfg, T).total;
}

moe_status moe_route(const moe_config* cfg, int32_t T, const void* x, const moe_weights* w,
                     const float* logits_in, float* logits_out, int32_t* topk_idx, float* topk_w,
                     void* ws, size_t ws_bytes, moe_stream_t stream) {
  g_detail[0] = 0;
  TRY(check_cfg(cfg, T));
  if (T == 0) return MOE_OK;
  CHECK_PTR(topk_idx);
  CHECK_PTR(topk_w);
  CHECK_ALIGN(logits_out);
  if (w != nullptr) CHECK_ALIGN(w->select_bias);
  const float* u = logits_in;
  if (u == nullptr) {
    CHECK_PTR(x);
    TRY(check_weights(cfg, w, true, false));
    float* dst = logits_out;
    if (dst == nullptr) {
      TRY(check_ws(cfg, T, ws, ws_bytes));
      dst = at<float>(ws, layout(cfg, T).u);
    }
    // the workspace, when one is given, also holds the split-K scratch of small batches
    const bool ws_ok = ws != nullptr && ws_bytes >= layout(cfg, T).total && aligned16(ws);
    TRY(do_gate(cfg, T, x, w, dst, ws_ok ? ws : nullptr, S_(stream)));
    u = dst;
  } else {
    CHECK_PTR(logits_in);
  }
  return do_route(cfg, T, u, w, topk_idx, topk_w, S_(stream));
}

moe_status moe_load_stats(const moe_config* cfg, int32_t T, const float* logits,
                          const int32_t* topk_idx, int32_t* counts, float* f, float* P,
                          float* lb_z, void* ws, size_t ws_bytes, moe_stream_t stream) {
  g_detail[0] = 0;
  TRY(check_cfg(cfg, T));
  if (T == 0) return fail(MOE_ERR_INVALID_ARG, "load statistics need T > 0");
  CHECK_PTR(logits);
  CHECK_PTR(topk_idx);
  CHECK_ALIGN(counts);
  CHECK_ALIGN(f);
  CHECK_ALIGN(P);
  CHECK_ALIGN(lb_z);
  TRY(check_ws(cfg, T, ws, ws_bytes));
  return do_stats(cfg, T, logits, topk_idx, counts, f, P, lb_z, ws, S_(stream));
}

moe_status moe_permute(const moe_config* cfg, int32_t T, const int32_t* topk_idx,
                       const float* topk_w, const void* x, int32_t* offsets, int32_t* row_token,
                       float* row_w,
                       int32_t* slot_row, void* x_perm, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
  g_detail[0] = 0;
  TRY(check_cfg(cfg, T));
  CHECK_PTR(offsets);
  if (T > 0) {
    CHECK_PTR(topk_idx);
    CHECK_PTR(topk_w);
    CHECK_PTR(row_token);
    CHECK_PTR(slot_row);
    CHECK_ALIGN(x);
    CHECK_ALIGN(row_w);
    if (x != nullptr) CHECK_PTR(x_perm);
  }
  TRY(check_ws(cfg, T, ws, ws_bytes));
  return do_permute(cfg, T, topk_idx, topk_w, x, offsets, row_token, row_w, slot_row, x_perm, ws,
                    S_(stream));
}

moe_status moe_expert_up(const moe_config* cfg, int32_t T, const void* x_perm,
                         const int32_t* offsets, const void* x, const moe_weights* w, void* h,
                         void* h_shared, moe_stream_t stream) {
  g_detail[0] = 0;
  TRY(check_cfg(cfg, T));
  if (T == 0) return MOE_OK;
  TRY(check_weights(cfg, w, false, true));
  CHECK_PTR(x_perm);
  CHECK_PTR(offsets);
  CHECK_PTR(h);
  if (cfg->n_shared > 0) {
    CHECK_PTR(x);
    CHECK_PTR(h_shared);
  }
  return do_up(cfg, T, x_perm, offsets, x, w, h, h_shared, nullptr, nullptr, S_(stream));
}

moe_status moe_expert_up_gather(const moe_config* cfg, int32_t T, const void* x,
                                const int32_t* row_token, const int32_t* offsets,
                                const moe_weights* w, void* h, void* h_shared,
                                moe_stream_t stream) {
  g_detail[0] = 0;
  TRY(check_cfg(cfg, T));
  if (T == 0) return MOE_OK;
  if (cfg->dtype != MOE_BF16)
    return fail(MOE_ERR_UNSUPPORTED, "the row gather runs on the bf16 tensor-core path only");
  TRY(check_weights(cfg, w, false, true));
  CHECK_PTR(x);
  CHECK_PTR(row_token);
  CHECK_PTR(offsets);
  CHECK_PTR(h);
  if (cfg->n_shared > 0) CHECK_PTR(h_shared);
  return do_up(cfg, T, nullptr, offsets, x, w, h, h_shared, nullptr, nullptr, S_(stream),
               row_token);
}

moe_status moe_expert_down(const moe_config* cfg, int32_t T, const void* h,
                           const int32_t* offsets, const void* h_shared, const moe_weights* w,
                           void* y_perm, void* y_shared, moe_stream_t stream) {
  g_detail[0] = 0;
  TRY(check_cfg(cfg, T));
  if (T == 0) return MOE_OK;
  TRY(check_weights(cfg, w, false, true));
  CHECK_PTR(h);
  CHECK_PTR(offsets);
  CHECK_PTR(y_perm);
  if (cfg->n_shared > 0) {
    CHECK_PTR(h_shared);
    CHECK_PTR(y_shared);
  }
  return do_down(cfg, T, h, offsets, h_shared, w, y_perm, y_shared, nullptr, nullptr, S_(stream));
}

moe_status moe_expert_ffn(const moe_config* cfg, int32_t T, const void* x_perm,
                          const int32_t* offsets, const void* x, const moe_weights* w,
                          void* y_perm, void* y_shared, void* ws, size_t ws_bytes,
                          moe_stream_t stream) {
  g_detail[0] = 0;
  TRY(check_cfg(cfg, T));
  if (T == 0) return MOE_OK;
  TRY(check_ws(cfg, T, ws, ws_bytes));
  TRY(check_weights(cfg, w, false, true));
  CHECK_PTR(x_perm);
  CHECK_PTR(offsets);
  CHECK_PTR(y_perm);
  if (cfg->n_shared > 0) {
    CHECK_PTR(x);
    CHECK_PTR(y_shared);
  }
  const Layout L = layout(cfg, T);
  void* h = at<char>(ws, L.h);
  void* h_sh = cfg->n_shared > 0 ? at<char>(ws, L.h_sh) : nullptr;
  int32_t* sched = at<int32_t>(ws, L.sched);
  TRY(reset_sched(cfg, T, ws, S_(stream)));
  float* split_part = at<float>(ws, L.split_part);
  // after the memset node: the caller's offsets are complete before either GEMM starts
  TRY(do_up(cfg, T, x_perm, offsets, x, w, h, h_sh, sched, split_part, S_(stream), nullptr,
            /*offsets_early=*/true));
  return do_down(cfg, T, h, offsets, h_sh, w, y_perm, y_shared, sched, split_part, S_(stream),
                 /*offsets_early=*/true);
}

moe_status moe_combine(const moe_config* cfg, int32_t T, const void* y_perm,
                       const int32_t* slot_row, const float* topk_w, const void* y_shared,
                       void* out, moe_stream_t stream) {
  g_detail[0] = 0;
  TRY(check_cfg(cfg, T));
  if (T == 0) return MOE_OK;
  CHECK_PTR(y_perm);
  CHECK_PTR(slot_row);
  CHECK_PTR(topk_w);
  CHECK_ALIGN(y_shared);
  CHECK_PTR(out);
  return do_combine(cfg, T, y_perm, slot_row, topk_w, y_shared, out, S_(stream));
}

moe_status moe_layer_forward(const moe_config* cfg, int32_t T, const void* x,
                             const moe_weights* w, void* out, int32_t* counts, float* lb_z,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
  g_detail[0] = 0;
  TRY(check_cfg(cfg, T));
  if (T == 0) return MOE_OK;
  CHECK_PTR(x);
  CHECK_PTR(out);
  CHECK_ALIGN(counts);
  CHECK_ALIGN(lb_z);
  TRY(check_weights(cfg, w, true, true));
  TRY(check_ws(cfg, T, ws, ws_bytes));
  const bool timed = g_timing.on && g_timing.calls < g_timing.max_calls;
  if (timed) g_timing.cur = g_timing.calls++;
  const moe_status s = layer_steps(cfg, T, x, w, out, counts, lb_z, ws, S_(stream));
  if (timed) {
    stage_mark(N_STAGES, S_(stream));
    g_timing.cur = -1;
  }
  return s;
}

moe_status moe_bias_update(const moe_config* cfg, const int32_t* counts, float rate,
                           float* select_bias, moe_stream_t stream) {
  g_detail[0] = 0;
  TRY(check_cfg(cfg, 0));
  CHECK_PTR(counts);
  CHECK_PTR(select_bias);
  if (!std::isfinite(rate) || rate < 0.0f)
    return fail(MOE_ERR_INVALID_ARG, "rate must be finite and >= 0");
  BiasUpdateArgs a;
  a.N = cfg->n_routed;
  a.counts = counts;
  a.rate = rate;
  a.bias = select_bias;
  return cuda_status(launch_bias_update(a, S_(stream)), "bias update");
}

moe_status moe_group_balance_losses(const moe_config* cfg, int32_t T, const float* logits,
                                    const int32_t* topk_idx, float* losses, void* ws,
                                    size_t ws_bytes, moe_stream_t stream) {
  g_detail[0] = 0;
  TRY(check_cfg(cfg, T));
  if (T == 0) return fail(MOE_ERR_INVALID_ARG, "the group losses need T > 0");
  CHECK_PTR(logits);
  CHECK_PTR(topk_idx);
  CHECK_PTR(losses);
  TRY(check_ws(cfg, T, ws, ws_bytes));
  const Layout L = layout(cfg, T);
  GroupLossArgs a;
  a.st.T = T; a.st.N = cfg->n_routed; a.st.K = cfg->top_k; a.st.score_fn = cfg->score_fn;
  a.st.u = logits; a.st.idx = topk_idx;
  a.st.counts = at<int32_t>(ws, L.counts);
  a.st.f = nullptr; a.st.P = nullptr; a.st.lb_z = nullptr;
  a.st.part_s = at<float>(ws, L.part_s);
  a.st.part_c = nullptr;  // the device-loss kernels count on their own
  a.st.part_lse = at<float>(ws, L.part_lse);
  a.st.nblk = stats_blocks(T);
  a.st.err = error_word();
  a.G = cfg->n_groups;
  a.recv = at<int32_t>(ws, L.recv);
  a.out = losses;
  return cuda_status(launch_group_losses(a, S_(stream)), "group balance losses");
}

moe_status moe_seq_balance_loss(const moe_config* cfg, int32_t T, int32_t seq_len,
                                const float* logits, const int32_t* topk_idx, float* per_seq,
                                float* loss, void* ws, size_t ws_bytes, moe_stream_t stream) {
  g_detail[0] = 0;
  TRY(check_cfg(cfg, T));
  if (T == 0) return fail(MOE_ERR_INVALID_ARG, "the sequence loss needs T > 0");
  if (seq_len < 1 || T % seq_len != 0)
    return fail(MOE_ERR_INVALID_ARG, "seq_len=%d must divide T=%d", seq_len, T);
  CHECK_PTR(logits);
  CHECK_PTR(topk_idx);
  CHECK_ALIGN(per_seq);
  CHECK_PTR(loss);
  TRY(check_ws(cfg, T, ws, ws_bytes));
  const Layout L = layout(cfg, T);
  SeqLossArgs a;
  a.T = T; a.N = cfg->n_routed; a.K = cfg->top_k; a.L = seq_len; a.B = T / seq_len;
  a.cps = seq_loss_chunks(seq_len);
  a.score_fn = cfg->score_fn;
  a.u = logits; a.idx = topk_idx;
  a.part_s = at<float>(ws, L.seq_s);
  a.part_c = at<int32_t>(ws, L.seq_c);
  a.seq_lb = at<double>(ws, L.seq_lb);
  a.per_seq = per_seq; a.mean = loss;
  a.err = error_word();
  return cuda_status(launch_seq_loss(a, S_(stream)), "sequence balance loss");
}

moe_status moe_stage_timing_start(int32_t max_calls) {
  g_detail[0] = 0;
  if (max_calls < 1 || max_calls > 100000)
    return fail(MOE_ERR_INVALID_ARG, "max_calls=%d not in [1, 100000]", max_calls);
  if (g_timing.on) return fail(MOE_ERR_INVALID_ARG, "stage timing already active");
  const size_t n = (size_t)max_calls * (N_STAGES + 1);
  cudaEvent_t* ev = new (std::nothrow) cudaEvent_t[n];
  if (ev == nullptr) return fail(MOE_ERR_INVALID_ARG, "host memory for %zu events", n);
  for (size_t i = 0; i < n; ++i) {
    const cudaError_t e = cudaEventCreate(&ev[i]);
    if (e != cudaSuccess) {
      for (size_t j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
      delete[] ev;
      return cuda_status(e, "cudaEventCreate");
    }
  }
  g_timing.ev = ev;
  g_timing.max_calls = max_calls;
  g_timing.calls = 0;
  g_timing.cur = -1;
  g_timing.on = true;
  return MOE_OK;
}

moe_status moe_stage_timing_stop(float* stage_ms, int32_t n_stages, int32_t* calls) {
  g_detail[0] = 0;
  if (!g_timing.on) return fail(MOE_ERR_INVALID_ARG, "stage timing not active");
  moe_status st = MOE_OK;
  if (stage_ms != nullptr && (n_stages < 0 || n_stages > N_STAGES))
    st = fail(MOE_ERR_INVALID_ARG, "n_stages=%d not in [0, %d]", n_stages, N_STAGES);
  const int nc = g_timing.calls;
  if (st == MOE_OK && stage_ms != nullptr) {
    for (int b = 0; b < n_stages; ++b) stage_ms[b] = 0.0f;
    for (int c = 0; c < nc && st == MOE_OK; ++c) {
      cudaEvent_t* e = g_timing.ev + (size_t)c * (N_STAGES + 1);
      cudaError_t ce = cudaEventSynchronize(e[N_STAGES]);
      if (ce != cudaSuccess) { st = cuda_status(ce, "cudaEventSynchronize"); break; }
      for (int b = 0; b < n_stages; ++b) {
        float ms = 0.0f;
        ce = cudaEventElapsedTime(&ms, e[b], e[b + 1]);
        if (ce != cudaSuccess) { st = cuda_status(ce, "cudaEventElapsedTime"); break; }
        stage_ms[b] += ms;
      }
    }
  }
  if (calls != nullptr) *calls = nc;
  const size_t n = (size_t)g_timing.max_calls * (N_STAGES + 1);
  for (size_t i = 0; i < n; ++i) cudaEventDestroy(g_timing.ev[i]);
  delete[] g_timing.ev;
  g_timing = StageTiming();
  return st;
}

moe_status moe_get_error(moe_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(S_(stream));
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "stream sync: %s", cudaGetErrorString(e));
  int* p = error_word();
  if (p == nullptr) return fail(MOE_ERR_CUDA, "error word unavailable");
  int v = 0;
  e = cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "read error word: %s", cudaGetErrorString(e));
  if (v != 0) {
    const int zero = 0;
    cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice);
  }
  return static_cast<moe_status>(v);
}

moe_status moe_selftest_wait_timeout(int32_t timeout_us, moe_stream_t stream) {
  g_detail[0] = 0;
  if (timeout_us < 1 || timeout_us > 10000000)
    return fail(MOE_ERR_INVALID_ARG, "timeout_us=%d not in [1, 1e7]", timeout_us);
  int* err = error_word();
  if (err == nullptr) return fail(MOE_ERR_CUDA, "error word unavailable");
  return cuda_status(launch_wait_selftest(err, 1000ull * timeout_us, S_(stream)), "selftest");
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "device consistency check failed";
  }
  return "unknown status";
}

const char* moe_last_error_detail(void) { return g_detail; }

unsigned long long moe_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
