// moe_permute_static_scratch: the token permutation for callers that cannot allocate device
// memory.
//
// Some callers have no way to hand this library a workspace: code running where device
// allocation is forbidden or unavailable (an allocator-free runtime, a host framework that owns
// every device allocation and exposes none to plugins, a process that must not grow its device
// footprint after start-up). moe_permute needs a few MB of scratch (per-block expert bitmasks,
// counts, segment bases, drop thresholds) from the caller's workspace; this variant keeps that
// scratch in one file-scope device array instead. The array is part of the loaded module: every
// GPU that loads the library holds it (kScratchBytes, 2.5 MiB) until the process exits.
//
// Limits: T <= kMaxTokens (65536) tokens, n_routed <= 256, n_groups <= 32 (the last two are the
// library's general limits). Larger T is refused with MOE_ERR_UNSUPPORTED.
//
// Every call uses the same array: two calls that overlap on the GPU (different streams, or
// different host threads without ordering) race on it and give wrong results. Nothing in the
// array has to start at zero: each call writes every scratch word before it reads it.
//
// The device address of the array is looked up (cudaGetSymbolAddress, with the device current)
// on the first call made on each device, and again on the first call after that device's
// context has changed (a device reset); make those calls before any stream capture.
#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "internal.h"

namespace {

constexpr int kMaxTokens = 65536;
constexpr int kMaxExperts = 256;
constexpr int kMaxGroups = 32;
constexpr int kTokensPerBlock = 256;  // the permutation kernels' block of tokens
constexpr int kMaxBlocks = kMaxTokens / kTokensPerBlock;
constexpr size_t kMaskBytes = (size_t)kMaxBlocks * kMaxExperts * 8 * sizeof(uint32_t);
constexpr size_t kCountBytes = (size_t)kMaxBlocks * kMaxExperts * sizeof(int32_t);
constexpr size_t kThrBytes = (size_t)kMaxGroups * sizeof(unsigned long long);
constexpr size_t kScratchBytes = kMaskBytes + 2 * kCountBytes + kThrBytes;
static_assert(kMaskBytes % 256 == 0 && kCountBytes % 256 == 0, "regions stay 256-B aligned");

// Scratch of moe_permute_static_scratch. In host code this name is only a stand-in for the
// symbol, not a device address: kernels get the address looked up by scratch_on_device().
static __device__ __align__(256) unsigned char g_permute_scratch[kScratchBytes];

std::mutex g_setup_mutex;

// Device address of g_permute_scratch on the current device, looked up on the first call on
// each device (cudaGetSymbolAddress with that device current) and again whenever the device's
// context has changed since (after a device reset the old address is dead).
moe_status scratch_on_device(void** out) {
  static moe::SymbolCache cache;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  void* p = cache.get(g_permute_scratch);
  if (p == nullptr)
    return moe::abi_fail(MOE_ERR_CUDA, "cudaGetSymbolAddress(permute scratch) failed");
  *out = p;
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status moe_permute_static_scratch(const moe_config* cfg, int32_t T,
                                                 const int32_t* topk_idx, const float* topk_w,
                                                 const void* x, int32_t* offsets,
                                                 int32_t* row_token, int32_t* slot_row,
                                                 void* x_perm, moe_stream_t stream) {
  moe_status st = moe::abi_check_config(cfg, T);
  if (st != MOE_OK) return st;
  if (T > kMaxTokens)
    return moe::abi_fail(MOE_ERR_UNSUPPORTED,
                         "moe_permute_static_scratch handles at most 65536 tokens; use "
                         "moe_permute with a workspace for more");
  if (cfg->n_routed > kMaxExperts || cfg->n_groups > kMaxGroups)
    return moe::abi_fail(MOE_ERR_UNSUPPORTED, "n_routed > 256 or n_groups > 32");
  if (offsets == nullptr || !aligned16(offsets))
    return moe::abi_fail(MOE_ERR_INVALID_ARG, "offsets is NULL or not 16-byte aligned");
  if (T > 0) {
    const void* need[] = {topk_idx, topk_w, row_token, slot_row};
    for (const void* p : need)
      if (p == nullptr || !aligned16(p))
        return moe::abi_fail(MOE_ERR_INVALID_ARG,
                             "topk_idx, topk_w, row_token, slot_row must be non-NULL and "
                             "16-byte aligned");
    if (x != nullptr && (!aligned16(x) || x_perm == nullptr || !aligned16(x_perm)))
      return moe::abi_fail(MOE_ERR_INVALID_ARG, "x / x_perm NULL or not 16-byte aligned");
  }
  void* scratch = nullptr;
  st = scratch_on_device(&scratch);
  if (st != MOE_OK) return st;

  char* base = static_cast<char*>(scratch);
  moe::PermuteArgs p;
  p.T = T; p.N = cfg->n_routed; p.K = cfg->top_k; p.D = cfg->n_groups;
  p.capacity_drop = cfg->capacity_drop ? 1 : 0;
  p.idx = topk_idx; p.w = topk_w; p.x = x; p.H = cfg->hidden;
  p.elem_bytes = cfg->dtype == MOE_BF16 ? 2 : 4;
  p.offsets = offsets; p.row_token = row_token; p.row_w = nullptr; p.slot_row = slot_row;
  p.x_perm = x_perm;
  p.masks = reinterpret_cast<uint32_t*>(base);
  p.cnt = reinterpret_cast<int32_t*>(base + kMaskBytes);
  p.base = reinterpret_cast<int32_t*>(base + kMaskBytes + kCountBytes);
  p.thr = reinterpret_cast<unsigned long long*>(base + kMaskBytes + 2 * kCountBytes);
  p.sched_zero = nullptr;
  p.err = moe::abi_error_word();
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  st = moe::abi_cuda_status(moe::launch_permute(p, moe::abi_num_sms(), cs),
                            "permute (static scratch)");
  if (st != MOE_OK) return st;
  return moe::abi_cuda_status(moe::launch_dispatch(p, moe::abi_num_sms(), cs),
                              "row dispatch (static scratch)");
}
