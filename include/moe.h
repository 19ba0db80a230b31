/*
 * moe.h - C ABI of the B300 (sm_103a) DeepSeekMoE layer forward.
 *
 * One layer forward on one GPU:
 *   gate logits -> scores -> group / device limited top-K routing -> load statistics ->
 *   permutation by expert (+ v2 device-level drop) -> routed SwiGLU experts + shared experts ->
 *   weighted combine back to token order.
 *
 * Sources for what each call computes (page title, section):
 *   [P3] "DeepSeek MoE：从v1到v3的演进" (wln20.github.io): ST-MoE balance loss and Z-loss,
 *        DeepSeek-v1 fine-grained / shared experts, DeepSeek-v2 device-limited routing and
 *        device-level token drop, DeepSeek-v3 sigmoid gate and selection-only bias.
 *   [P4] "DeepSeek-V3的Group-Limited Expert Routing与负载均衡优化实践" (mhpn.cn), sections 1
 *        and 3: group-limited routing (score groups, keep the best, mask the rest, top-K).
 *   [P2] "从零构建DeepSeekMoE" (opc.csdn.net), sections 2.1, 2.2 and 5.2: fine-grained expert
 *        FFN, shared + routed forward, router linear layer.
 *
 * Conventions (every entry point):
 *   - Every tensor pointer is a DEVICE pointer on the current CUDA device unless stated, owned
 *     by the caller. The library allocates no device memory: scratch comes from `ws`, whose
 *     size moe_workspace_size() gives (one size fits every call for a given config and T).
 *     A workspace serves one call at a time: two calls in flight on different streams need
 *     two workspaces (it holds intermediates and the expert GEMMs' tile counters).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *     Nothing synchronises except moe_get_error().
 *   - Argument errors are returned synchronously before anything is launched; the text of the
 *     last one is available from moe_last_error_detail(). Launch failures return
 *     MOE_ERR_CUDA. Errors found on the device (a bounded wait that ran out) are recorded in a
 *     per-device error word read by moe_get_error().
 *   - Pointers must be 16-byte aligned. Row-major layouts; "[A, B]" means B contiguous.
 *   - dtype MOE_BF16: activations and weights bf16 (tensor cores, fp32 accumulation).
 *     dtype MOE_F32: everything fp32 with fp32 CUDA-core arithmetic (small layers).
 *     Logits, scores and routing weights are always fp32.
 *   - No C++ exception crosses this boundary.
 */
#ifndef MOE_B300_H_
#define MOE_B300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,  /* bad pointer, size or config value */
  MOE_ERR_UNSUPPORTED = -2,  /* valid, but outside what the kernels handle (see moe_config) */
  MOE_ERR_WORKSPACE = -3,    /* ws_bytes smaller than moe_workspace_size() */
  MOE_ERR_CUDA = -4,         /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = -5,      /* a kernel's bounded wait ran out (reported by moe_get_error) */
  MOE_ERR_DEVICE_CHECK = -6  /* a kernel's own consistency check failed (moe_get_error) */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;
typedef enum { MOE_SOFTMAX = 0, MOE_SIGMOID = 1 } moe_score_fn;

typedef void* moe_stream_t; /* cudaStream_t */

/*
 * Layer shape and routing rule.
 *   hidden H, n_routed N (1..256), n_shared S (>= 0), inter I (intermediate size of one
 *   fine-grained expert, [P3] DeepSeek-v1 / [P2] section 2.1), top_k K (1..16).
 *   n_groups G (1..32, divides N): expert e belongs to group e / (N/G). Groups are the v3
 *     expert groups [P4] or the v2 virtual devices [P3]; G = 1 means no group limit.
 *   topk_groups: groups (v3) or devices (v2, M) a token may use; K <= topk_groups * N/G.
 *   group_score_topn (1 or 2): a group's score is the sum of its top-n selection scores
 *     (1 = its best expert, which is the v2 device-limited rule; 2 = the v3 rule).
 *   score_fn: softmax over all N (v1/v2) or independent sigmoid (v3).
 *   norm_topk: 1 = divide the K chosen scores by their sum; routed_scale (> 0) multiplies the
 *     routed weights.
 *   capacity_drop: 1 = v2 device-level drop. Each of the G devices keeps at most
 *     C = ceil(T*K/G) assignments: the highest routing weight first, ties to the lower token
 *     then the lower slot; the weight compared is the correctly rounded fp32 weight.
 *   dtype: MOE_BF16 needs H % 64 == 0 and I % 128 == 0; MOE_F32 needs H % 4 == 0.
 */
typedef struct {
  int32_t hidden;
  int32_t n_routed;
  int32_t n_shared;
  int32_t inter;
  int32_t top_k;
  int32_t n_groups;
  int32_t topk_groups;
  int32_t group_score_topn;
  int32_t score_fn;      /* moe_score_fn */
  int32_t norm_topk;
  float routed_scale;
  int32_t capacity_drop;
  int32_t dtype;         /* moe_dtype */
} moe_config;

/* Layer parameters (device pointers, config dtype unless stated). */
typedef struct {
  const void* w_gate;             /* [N, H] router weight ([P2] section 5.2 router linear) */
  const float* gate_logit_bias;   /* [N] fp32 router bias added to the logits, or NULL */
  const float* select_bias;       /* [N] fp32 v3 selection-only bias b_i ([P3] v3), or NULL */
  const void* w13;                /* [N, 2I, H]: rows 0..I-1 gate proj., rows I..2I-1 up proj. */
  const void* w2;                 /* [N, H, I]  down projection */
  const void* w13_shared;         /* [S, 2I, H] (NULL iff S == 0) */
  const void* w2_shared;          /* [S, H, I]  (NULL iff S == 0) */
} moe_weights;

/* Bytes of scratch every entry point below accepts for this config and token count
 * (0 if the config is invalid). Host-only; launches nothing. */
size_t moe_workspace_size(const moe_config* cfg, int32_t T);

/*
 * Routing ([P3] v3 sigmoid + selection bias, [P3] v2 device-limited, [P4] sections 1 and 3).
 *   u = x W_g^T + gate_logit_bias (or u = logits_in when given; x and w_gate then unused);
 *   s = softmax(u) or sigmoid(u);  key = s + select_bias;
 *   group score = sum of the group's top-n keys; keep the best topk_groups groups (ties to the
 *   lower group); among their experts take the K highest keys (ties to the lower expert);
 *   w = s of the chosen experts (/ their sum if norm_topk) * routed_scale.
 * The chosen set is exactly the one exact (fp64) keys give: keys are evaluated in fp32, and a
 * token whose group or expert margin falls within the fp32 error bound is rechecked in fp64
 * (for a sigmoid gate only the groups and experts inside the bound are rescored).
 * ws (optional when logits_in is given) also holds the gate GEMM's split-K scratch for small
 * batches; without it the gate runs unsplit.
 *   x          [T, H] dtype (unused if logits_in)
 *   logits_in  [T, N] fp32 or NULL;  logits_out [T, N] fp32 or NULL (written when computed)
 *   topk_idx   [T, K] int32 out: chosen experts in ascending expert index
 *   topk_w     [T, K] fp32 out: their weights (correctly rounded when capacity_drop is set)
 */
moe_status moe_route(const moe_config* cfg, int32_t T, const void* x, const moe_weights* w,
                     const float* logits_in, float* logits_out, int32_t* topk_idx,
                     float* topk_w, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Expert-load statistics of one batch ([P3] ST-MoE section).
 *   counts[e] = assignments routed to e (before any drop); f[e] = counts[e] / (T K);
 *   P[e] = sum_t s[t,e] / sum_t sum_j s[t,j];  L_B = N sum_e f[e] P[e];
 *   lse_t = log sum_j exp(u[t,j]);  L_Z = mean_t lse_t^2.
 *   logits [T, N] fp32, topk_idx [T, K] int32 (from moe_route);
 *   counts [N] int32, f [N] fp32, P [N] fp32 (each may be NULL), lb_z [3] fp32 or NULL:
 *   {L_B, L_Z, mean_t lse_t}.
 */
moe_status moe_load_stats(const moe_config* cfg, int32_t T, const float* logits,
                          const int32_t* topk_idx, int32_t* counts, float* f, float* P,
                          float* lb_z, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Permutation by expert (+ v2 device-level drop when cfg->capacity_drop).
 * Kept assignments form one contiguous segment per expert, experts ascending, rows inside a
 * segment in ascending token order.
 *   topk_idx, topk_w [T, K] from moe_route;  x [T, H] dtype or NULL (then x_perm is not written)
 *   offsets [N+1] int32 out (offsets[N] = rows kept R);  row_token [T*K] int32 out (first R used)
 *   row_w [T*K] fp32 out or NULL: row_w[r] = topk_w of the assignment placed at row r (r < R)
 *   slot_row [T*K] int32 out: row of assignment (t,k), -1 if dropped;
 *   x_perm [T*K, H] dtype out: x_perm[r] = x[row_token[r]] for r < R.
 */
moe_status moe_permute(const moe_config* cfg, int32_t T, const int32_t* topk_idx,
                       const float* topk_w, const void* x, int32_t* offsets, int32_t* row_token,
                       float* row_w, int32_t* slot_row, void* x_perm, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/*
 * moe_permute without a workspace, for callers that cannot allocate device memory (a runtime
 * without a device allocator, a host framework that owns all device allocations and gives none
 * to plugins, a process that must not grow its device footprint). The pages have no
 * counterpart: this is a deployment variant of moe_permute, same arguments minus ws, same
 * outputs bit for bit.
 *   Its scratch (per-block expert bitmasks, counts, segment bases, drop thresholds) is one
 *   file-scope device array of 2.5 MiB that every GPU loading the library holds until exit.
 *   Limits: T <= 65536 (larger T returns MOE_ERR_UNSUPPORTED), n_routed <= 256, n_groups <= 32.
 *   All calls share that array: calls that overlap on the GPU race and give wrong results.
 *   Nothing in it needs clearing between calls (each call writes what it reads).
 *   The first call on a device looks up the array's device address (with that device
 *   current), and so does the first call after the device's context changed (a device reset);
 *   make those calls before any stream capture. No allocation happens, ever.
 */
moe_status moe_permute_static_scratch(const moe_config* cfg, int32_t T, const int32_t* topk_idx,
                                      const float* topk_w, const void* x, int32_t* offsets,
                                      int32_t* row_token, int32_t* slot_row, void* x_perm,
                                      moe_stream_t stream);

/*
 * Routed + shared SwiGLU experts ([P3] DeepSeek-v1, [P2] sections 2.1-2.2):
 *   for every row r of expert e's segment: h = silu(x_perm[r] W13_e[0:I]^T) * (x_perm[r] W13_e[I:2I]^T),
 *   y_perm[r] = h W2_e^T;  y_shared[t] = sum over shared experts s of the same on x[t].
 *   x_perm [T*K, H], offsets [N+1] (device; rows per expert are read on the device),
 *   x [T, H] (shared experts; may be NULL iff S == 0), y_perm [T*K, H] out, y_shared [T, H] out
 *   (NULL iff S == 0). h is rounded to dtype between the two GEMMs.
 *   ws holds h and the tile counters that let CTA pairs claim GEMM tiles as they free up (the
 *   outputs do not depend on which pair computes a tile).
 */
moe_status moe_expert_ffn(const moe_config* cfg, int32_t T, const void* x_perm,
                          const int32_t* offsets, const void* x, const moe_weights* w,
                          void* y_perm, void* y_shared, void* ws, size_t ws_bytes,
                          moe_stream_t stream);

/* The two halves of moe_expert_ffn, exposed so each GEMM can be timed on its own. With no
 * workspace they hand out tiles round robin; outputs are bitwise equal to moe_expert_ffn's.
 *   h [T*K, I] dtype out/in;  h_shared [T, S*I] dtype out/in (NULL iff S == 0). */
moe_status moe_expert_up(const moe_config* cfg, int32_t T, const void* x_perm,
                         const int32_t* offsets, const void* x, const moe_weights* w, void* h,
                         void* h_shared, moe_stream_t stream);
moe_status moe_expert_down(const moe_config* cfg, int32_t T, const void* h,
                           const int32_t* offsets, const void* h_shared, const moe_weights* w,
                           void* y_perm, void* y_shared, moe_stream_t stream);

/*
 * The up half with its routed rows read straight from x in token order ([P4] section 5's
 * dispatch done as a row gather inside the GEMM instead of a copy): row r of expert e's
 * segment is x[row_token[r]]. This is what moe_layer_forward runs on the bf16 path, so that
 * the permuted copy x_perm is never written or read. Outputs are bitwise equal to
 * moe_expert_up's on x_perm = x[row_token]. bf16 only (MOE_ERR_UNSUPPORTED for fp32).
 *   x [T, H] bf16;  row_token [T*K] int32 and offsets [N+1] int32 from moe_permute (values are
 *   clamped to [0, T-1] on the device);  h, h_shared as for moe_expert_up.
 */
moe_status moe_expert_up_gather(const moe_config* cfg, int32_t T, const void* x,
                                const int32_t* row_token, const int32_t* offsets,
                                const moe_weights* w, void* h, void* h_shared,
                                moe_stream_t stream);

/*
 * Weighted combine back to token order ([P2] section 2.2 forward):
 *   out[t] = sum_k [slot_row(t,k) >= 0] topk_w[t,k] y_perm[slot_row(t,k)] + y_shared[t]
 *   (fp32 accumulation; y_shared may be NULL). out [T, H] dtype.
 */
moe_status moe_combine(const moe_config* cfg, int32_t T, const void* y_perm,
                       const int32_t* slot_row, const float* topk_w, const void* y_shared,
                       void* out, moe_stream_t stream);

/*
 * The whole layer: moe_route -> [moe_load_stats] -> moe_permute -> moe_expert_ffn ->
 * moe_combine, all on `stream`, intermediates in `ws`.
 *   x [T, H] dtype, out [T, H] dtype; counts [N] int32 or NULL, lb_z [3] fp32 or NULL (the
 *   statistics are computed only when one of them is given).
 */
moe_status moe_layer_forward(const moe_config* cfg, int32_t T, const void* x,
                             const moe_weights* w, void* out, int32_t* counts, float* lb_z,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Device-level and communication balance losses ([P3] DeepSeek-v1 "设备级负载loss", DeepSeek-v2
 * "通信负载均衡loss"; the page describes them without formulas, so the expert-level loss of
 * moe_load_stats is taken with the n_groups devices as its units, expert e on device e/(N/G)):
 *   f'_d = sum_{e on d} counts[e] / (T K);   P'_d = sum_{e on d} P[e];
 *   L_dev = G sum_d f'_d P'_d;
 *   R_d = tokens with at least one chosen expert on d (tokens d receives);
 *   L_comm = G sum_d (R_d / sum R) P'_d.
 * Both are 1 when routing is uniform; with one expert per device L_dev is the expert-level L_B.
 *   logits [T, N] fp32, topk_idx [T, K] int32 (from moe_route); losses [2] fp32 out:
 *   {L_dev, L_comm}.
 */
moe_status moe_group_balance_losses(const moe_config* cfg, int32_t T, const float* logits,
                                    const int32_t* topk_idx, float* losses, void* ws,
                                    size_t ws_bytes, moe_stream_t stream);

/*
 * Sequence-wise balance loss ([P3] DeepSeek-v3, "sequence粒度的负载均衡loss"): the expert-level
 * balance loss of moe_load_stats computed within each sequence instead of over the batch, and
 * averaged over the sequences. The page gives no formula; this is the plain reading:
 *   L_b = N sum_e f_e^b P_e^b with f_e^b = (assignments of sequence b to e) / (seq_len K) and
 *   P_e^b = (sum of e's scores over b's tokens) / (sum of all scores over b's tokens);
 *   loss = (1/B) sum_b L_b over the B = T / seq_len sequences of seq_len consecutive tokens.
 * It equals 1 when routing is uniform inside every sequence and N / K when every sequence
 * collapses onto K experts, even if the batch as a whole is balanced.
 *   logits [T, N] fp32 and topk_idx [T, K] int32 (from moe_route); per_seq [T / seq_len] fp32
 *   out or NULL; loss [1] fp32 out. seq_len must divide T.
 */
moe_status moe_seq_balance_loss(const moe_config* cfg, int32_t T, int32_t seq_len,
                                const float* logits, const int32_t* topk_idx, float* per_seq,
                                float* loss, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Auxiliary-loss-free balancing bias update ([P3] DeepSeek-v3, "Auxiliary-Loss-Free load
 * balancing"): after a batch, each expert's selection bias moves by `rate` against its load:
 *   e_i = mean_j counts[j] - counts[i];  select_bias[i] += rate * sign(e_i)
 * (overloaded experts lose rate, underloaded ones gain it, an expert exactly at the mean keeps
 * its bias). The sign is decided exactly in integers; the addition is one fp32 add.
 *   counts [N] int32 (from moe_load_stats or moe_layer_forward), select_bias [N] fp32 in/out,
 *   rate >= 0 (the page's bias update rate u).
 */
moe_status moe_bias_update(const moe_config* cfg, const int32_t* counts, float rate,
                           float* select_bias, moe_stream_t stream);

/*
 * Optional per-stage timing of moe_layer_forward (measurement aid; not thread-safe, one host
 * thread). Between start and stop, each of the first `max_calls` moe_layer_forward calls of
 * this process records a CUDA event on its stream at the start of every stage and at its end;
 * nothing synchronises inside the calls. Stages, in order:
 *   0 gate GEMM, 1 routing, 2 load statistics (zero when not requested), 3 permutation
 *   (drop thresholds, histogram, scan, scatter), 4 row dispatch (x -> x_perm; empty on the
 *   bf16 path, where the up GEMM gathers its rows from x), 5 expert up GEMM (routed + shared,
 *   SwiGLU), 6 expert down GEMM, 7 combine.
 * Calls captured into a CUDA graph record their events as graph nodes, which record each time
 * the graph runs; stop then reads the last run's times.
 * moe_stage_timing_start creates the events (host resources only, no device memory).
 * moe_stage_timing_stop waits for the recorded events, writes the summed milliseconds of the
 * first n_stages stages over the recorded calls to stage_ms (may be NULL), the number of
 * recorded calls to *calls (may be NULL), and destroys the events.
 */
#define MOE_N_STAGES 8
moe_status moe_stage_timing_start(int32_t max_calls);
moe_status moe_stage_timing_stop(float* stage_ms, int32_t n_stages, int32_t* calls);

/* Synchronises `stream`, then returns and clears the current device's error word
 * (MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_CHECK), or MOE_ERR_CUDA if the sync failed. */
moe_status moe_get_error(moe_stream_t stream);

/* Self-test of the kernels' bounded waits: launches one CTA that waits on an mbarrier nothing
 * will ever arrive on, with a limit of `timeout_us` microseconds (1 .. 10,000,000). The wait
 * gives up, records MOE_ERR_TIMEOUT in the device error word and the kernel returns; read it
 * with moe_get_error(). No fault, no trap, the context stays usable. */
moe_status moe_selftest_wait_timeout(int32_t timeout_us, moe_stream_t stream);

/*
 * Redundant-expert placement planner (host only, no GPU; [P4] sections 2 and 4: replicate hot
 * experts, place the replicas on the GPUs of an expert-parallel deployment). From each expert's
 * measured load (e.g. moe_load_stats counts summed over a serving window):
 *   replicate: the n_gpus * slots_per_gpu - n_experts extra replicas go, one at a time, to the
 *     expert with the largest load per replica (ties: lower expert) among the experts with fewer
 *     replicas than there are GPUs (while any remains); a replica carries load / replicas;
 *   place: replicas by decreasing load (ties: lower expert, lower replica) onto the least-loaded
 *     GPU with a free slot that does not host that expert yet (ties: lower GPU), else onto the
 *     least-loaded GPU with a free slot;
 *   n_nodes > 1 (hierarchical, [P4] section 2): expert groups (n_groups of consecutive experts)
 *     first go, heaviest first, to the least-loaded node with room (n_groups / n_nodes groups
 *     per node); then each node replicates and places its own experts on its n_gpus / n_nodes
 *     GPUs (GPU g is on node g / (n_gpus / n_nodes)).
 *   load [n_experts] (>= 0); replicas [n_experts] out; gpu_expert [n_gpus * slots_per_gpu] out:
 *   the experts each GPU hosts (-1 = empty slot); gpu_load [n_gpus] out (may be NULL).
 */
typedef struct {
  int32_t n_experts;
  int32_t n_gpus;
  int32_t slots_per_gpu;
  int32_t n_nodes;   /* <= 1: global placement */
  int32_t n_groups;  /* hierarchical placement only */
} moe_placement_config;
moe_status moe_plan_placement(const moe_placement_config* pc, const int64_t* load,
                              int32_t* replicas, int32_t* gpu_expert, double* gpu_load);

/* Number of kernels this library has launched in this process so far (all devices, all
 * streams; a launch made while a stream is captured into a CUDA graph counts once, at capture).
 * Host-only counter, for measurement. */
unsigned long long moe_kernel_launches(void);

/* Static text for a status code. */
const char* moe_status_string(moe_status s);

/* Text of the last argument error raised on this host thread ("" if none). */
const char* moe_last_error_detail(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H_ */
