// Launchers shared between the C-ABI layer (abi.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Count of kernels this library has launched (abi.cu); every launcher adds its launches.
void note_launches(int n);

// Launch with programmatic stream serialization: the kernel's CTAs may start (and run their
// prologue) while the kernel ahead of it in the stream is finishing; each kernel of this library
// waits for its predecessor (pdl_wait) before its first access to global memory. Counts the launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  note_launches(1);
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- routing (route.cu)
struct RouteArgs {
  int T, N, K, G, Gk, topn, score_fn, norm_topk, precise_w;
  float scale;
  const float* u;       // [T, N] logits
  const float* bias;    // [N] selection bias or nullptr
  int32_t* idx;         // [T, K]
  float* w;             // [T, K]
  int* err;
};
cudaError_t launch_route(const RouteArgs& a, int num_sms, cudaStream_t st);

struct StatsArgs {
  int T, N, K, score_fn;
  const float* u;       // [T, N]
  const int32_t* idx;   // [T, K]
  int32_t* counts;      // [N] (scratch or caller's)
  float* f;             // [N] or nullptr
  float* P;             // [N] or nullptr
  float* lb_z;          // [3] or nullptr
  float* part_s;        // scratch [nblk, N]
  int32_t* part_c;      // scratch [nblk, N] assignment counts, or nullptr (counts are given)
  float* part_lse;      // scratch [nblk, 2]
  int nblk;
  int* err;
};
int stats_blocks(int T);
cudaError_t launch_stats(const StatsArgs& a, cudaStream_t st);

// Device-level and communication balance losses over the n_groups devices (route.cu).
struct GroupLossArgs {
  StatsArgs st;         // logits, idx, counts scratch, score partials (lb_z, f, P unused)
  int G;
  int32_t* recv;        // scratch [G]: tokens each device receives
  float* out;           // [2]: L_dev, L_comm
};
cudaError_t launch_group_losses(const GroupLossArgs& a, cudaStream_t st);

// ---------------------------------------------------------------- balancing (balance.cu)
struct BiasUpdateArgs {
  int N;
  const int32_t* counts;  // [N]
  float rate;
  float* bias;            // [N] in/out
};
cudaError_t launch_bias_update(const BiasUpdateArgs& a, cudaStream_t st);

struct SeqLossArgs {
  int T, N, K, L, B, cps, score_fn;  // B = T / L sequences, cps chunks per sequence
  const float* u;         // [T, N] logits
  const int32_t* idx;     // [T, K]
  float* part_s;          // scratch [B * cps, N]
  int32_t* part_c;        // scratch [B * cps, N]
  double* seq_lb;         // scratch [B]
  float* per_seq;         // [B] or nullptr
  float* mean;            // [1]
  int* err;
};
int seq_loss_chunks(int L);
cudaError_t launch_seq_loss(const SeqLossArgs& a, cudaStream_t st);

// ---------------------------------------------------------------- permutation (permute.cu)
struct PermuteArgs {
  int T, N, K, D, capacity_drop;
  const int32_t* idx;   // [T, K]
  const float* w;       // [T, K]
  const void* x;        // [T, H] or nullptr
  int H, elem_bytes;
  int32_t* offsets;     // [N+1]
  int32_t* row_token;   // [T*K]
  float* row_w;         // [T*K] or nullptr: routing weight of the assignment at each row
  int32_t* slot_row;    // [T*K]
  void* x_perm;         // [T*K, H]
  // scratch
  uint32_t* masks;      // [nb, N, 8]
  int32_t* cnt;         // [nb, N]
  int32_t* base;        // [nb, N]
  unsigned long long* thr;  // [D]
  int32_t* sched_zero;  // nullptr, or kSchedInts scheduling ints the permutation zeroes (the expert
                        // GEMMs that follow claim tiles from them)
  int* err;
};
int permute_blocks(int T);
// drop thresholds, histogram, scan, scatter: offsets, row_token, slot_row
cudaError_t launch_permute(const PermuteArgs& a, int num_sms, cudaStream_t st);
// x_perm[slot_row(t,k)] = x[t] (no-op when x or x_perm is null)
cudaError_t launch_dispatch(const PermuteArgs& a, int num_sms, cudaStream_t st);

// ---------------------------------------------------------------- combine (combine.cu)
struct CombineArgs {
  int T, H, K, dtype;
  int rows;             // rows of y (slot_row values are below it)
  int* err;
  const void* y;        // [rows, H]
  const int32_t* slot_row;
  const float* w;
  const void* ys;       // [T, H] or nullptr
  void* out;            // [T, H]
};
cudaError_t launch_combine(const CombineArgs& a, int num_sms, cudaStream_t st);

// ---------------------------------------------------------------- GEMMs
enum GemmMode { MODE_GATE = 0, MODE_UP = 1, MODE_DOWN = 2 };

// Problem set of one grouped GEMM launch: n_routed expert segments (rows from `offsets`,
// device) plus, when has_shared, one shared-expert problem over all T rows.
struct GemmArgs {
  int mode;
  int T, H, I, S, N;    // N = routed experts (MODE_GATE: router outputs)
  int n_routed, has_shared;
  const int32_t* offsets;   // [n_routed+1] device, or nullptr for MODE_GATE
  int rows_cap;             // rows of the routed A / out tensors (T*K)
  const void* a0;           // routed A: x_perm [rows_cap,H] | h [rows_cap,I] | x [T,H] (gate)
  const void* a1;           // shared A: x [T,H] | h_shared [T,S*I]
  const void* b0;           // routed W: w13 [N,2I,H] | w2 [N,H,I] | w_gate [N,H]
  const void* b1;           // shared W: w13s [S,2I,H] | w2s [S,H,I]
  void* out0;               // routed out: h [rows_cap,I] | y [rows_cap,H] | u [T,N] fp32
  void* out1;               // shared out: h_shared [T,S*I] | y_shared [T,H]
  const float* gate_bias;   // MODE_GATE: [N] or nullptr
  float* gate_part;         // MODE_GATE split-K partial sums, or nullptr (no split)
  size_t gate_part_floats;  // capacity of gate_part
  int* sched;               // UP / DOWN (tcgen05): tile counter, zero at launch, for the dynamic
                            // tile schedule; nullptr: static round-robin schedule
  const int32_t* row_token; // UP (tcgen05) row gather: routed row r is x[row_token[r]], with
                            // a0 = x [T,H]; nullptr: a0 = x_perm
  float* split_part;        // UP / DOWN (tcgen05): fp32 partial accumulators of the tail tiles
                            // split along K (kSplitMaxPieces pieces), or nullptr (no split)
  int* split_cnt;           // UP / DOWN: kSplitCounters arrival counters of those pieces, zero
                            // at launch (the last arrival sets its counter back to zero)
  int offsets_early;        // UP / DOWN: 1 when `offsets` were written by a kernel at least two
                            // launches back in the stream (or before a non-kernel node), so the
                            // GEMM may read them before waiting for the kernel just ahead
  int* err;
};
// Tail split of the expert GEMMs: tiles of the last, partly filled wave are cut along K into
// pieces that idle CTA pairs take; the last piece of a tile to finish adds the pieces' fp32
// partial accumulators in piece order and runs the epilogue.
constexpr int kSplitMaxTiles = 40;                    // split tiles per launch at most
constexpr int kSplitWarps = 16;                       // epilogue warps of a CTA pair
constexpr int kSplitCounters = kSplitMaxTiles * kSplitWarps;
constexpr int kSplitMaxPieces = 80;                   // pieces per launch at most
constexpr size_t kSplitPieceFloats = 2 * 128 * 256;   // a pair's 256 x 256 fp32 accumulator
// Ints of the workspace's scheduling region: the up and down GEMMs' tile counters, then the
// up and down GEMMs' split counters. The permutation (or a memset) zeroes all of it.
constexpr int kSchedInts = 2 + 2 * kSplitCounters;
// Rows (of N floats) of the gate GEMM's split-K scratch the workspace provides.
constexpr int GATE_PART_ROWS = 16384;
// bf16 on tcgen05 / TMEM / TMA (gemm_tc.cu)
cudaError_t launch_gemm_tc(const GemmArgs& a, int num_sms, cudaStream_t st);
// fp32 on CUDA cores (gemm_simt.cu)
cudaError_t launch_gemm_simt(const GemmArgs& a, cudaStream_t st);

// Handle of the CUDA context current on the calling thread (0 if none or unknown). A device
// address looked up with cudaGetSymbolAddress belongs to that context: after a device reset
// (a new primary context) the old address is dead, so caches of such addresses key on it.
uintptr_t current_context();

// Device address of a __device__ variable on the current device, looked up once per device and
// context and cached (nullptr if the lookup failed). Not thread-safe: callers serialise.
struct SymbolCache {
  void* ptr[64] = {nullptr};
  uintptr_t ctx[64] = {0};
  template <typename Sym>
  void* get(const Sym& symbol) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    const uintptr_t now = current_context();
    if (ptr[dev] != nullptr && now != 0 && now == ctx[dev]) return ptr[dev];
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess) {
      ptr[dev] = nullptr;
      return nullptr;
    }
    ptr[dev] = p;
    ctx[dev] = current_context();  // the lookup made the device's primary context current
    return p;
  }
};

// Shared argument checking and error reporting of the C ABI (abi.cu).
}  // namespace moe
#include "../../include/moe.h"
namespace moe {
moe_status abi_check_config(const moe_config* c, int32_t T);
moe_status abi_fail(moe_status s, const char* msg);
moe_status abi_cuda_status(cudaError_t e, const char* what);
int* abi_error_word();
int abi_num_sms();

// Self-test of the bounded wait: one CTA waits on an mbarrier nothing arrives on.
cudaError_t launch_wait_selftest(int* err, unsigned long long timeout_ns, cudaStream_t st);

}  // namespace moe
