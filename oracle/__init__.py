"""fp64 CPU oracle of the DeepSeekMoE layer forward.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the benchmark's CPU-baseline
leg may import this; the library path never does. It shares no code with the CUDA kernels.
The arithmetic lives in ``moe_oracle.cpp`` (plain fp64 loops); this wrapper marshals numpy
arrays and orders the steps of one layer forward:

  gate logits -> scores -> (group / device limited) top-K -> [stats] -> [v2 drop]
  -> permutation -> per-expert SwiGLU rows + shared experts -> weighted combine

Page citations sit on each C function. Parity of the layer output at full size has no
closed form; what pins each step is listed in the oracle pin tests.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with g++ (OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
               _SRC, "-o", tmp, "-lquadmath"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


class OracleCfg(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int),
                ("G", ctypes.c_int), ("Gk", ctypes.c_int), ("K", ctypes.c_int),
                ("topn", ctypes.c_int), ("score_fn", ctypes.c_int), ("norm_topk", ctypes.c_int),
                ("routed_scale", ctypes.c_double), ("S", ctypes.c_int), ("I", ctypes.c_int),
                ("capacity_drop", ctypes.c_int)]


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        assert _lib.oracle_abi_version() == 2
    return _lib


def _p(a: np.ndarray | None, ct=ctypes.c_double):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle wants contiguous arrays"
    return a.ctypes.data_as(ctypes.POINTER(ct))


def _cfg(cfg, T: int | None = None) -> OracleCfg:
    return OracleCfg(T=cfg.T if T is None else T, H=cfg.hidden, N=cfg.n_routed, G=cfg.n_groups,
                     Gk=cfg.topk_groups, K=cfg.top_k, topn=cfg.group_score_topn,
                     score_fn=1 if cfg.score_fn == "sigmoid" else 0,
                     norm_topk=int(bool(cfg.norm_topk)), routed_scale=float(cfg.routed_scale),
                     S=cfg.n_shared, I=cfg.inter, capacity_drop=int(bool(cfg.capacity_drop)))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


# ---------------------------------------------------------------- step functions
def gate_logits(x, w_gate, gate_bias=None) -> np.ndarray:
    x, w_gate = _f64(x), _f64(w_gate)
    T, H = x.shape
    N = w_gate.shape[0]
    gb = None if gate_bias is None else _f64(gate_bias)
    u = np.empty((T, N), np.float64)
    lib().oracle_gate_logits(T, H, N, _p(x), _p(w_gate), _p(gb), _p(u))
    return u


def scores(u, score_fn: str) -> np.ndarray:
    u = _f64(u)
    T, N = u.shape
    s = np.empty_like(u)
    lib().oracle_scores(T, N, 1 if score_fn == "sigmoid" else 0, _p(u), _p(s))
    return s


def route(cfg, s, select_bias=None, u=None):
    """-> (idx [T,K] int32 ascending expert id, w [T,K] f64, margin [T] f64).

    s: the fp64 scores. u (optional): the logits they came from. With u, two keys (or group
    scores) whose fp64 values lie within 1e-14 * max(1, |a|, |b|) of each other are ordered by
    their real values, evaluated in quad precision from u (values within 2^-80 * max(|a|, |b|)
    count as equal: lower index first); without u the fp64 values decide alone."""
    s = _f64(s)
    T = s.shape[0]
    c = _cfg(cfg, T)
    b = None if select_bias is None else _f64(select_bias)
    uu = None if u is None else _f64(u)
    if uu is not None:
        assert uu.shape == s.shape
    idx = np.empty((T, cfg.top_k), np.int32)
    w = np.empty((T, cfg.top_k), np.float64)
    margin = np.empty((T,), np.float64)
    lib().oracle_route(ctypes.byref(c), _p(s), _p(uu), _p(b), _p(idx, ctypes.c_int32), _p(w),
                       _p(margin))
    return idx, w, margin


@dataclass
class LoadStats:
    counts: np.ndarray
    f: np.ndarray
    P: np.ndarray
    lb: float
    zloss: float
    lse_mean: float


def load_stats(cfg, u, s, idx) -> LoadStats:
    u, s = _f64(u), _f64(s)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T = u.shape[0]
    c = _cfg(cfg, T)
    N = cfg.n_routed
    counts = np.empty(N, np.int64)
    f = np.empty(N, np.float64)
    P = np.empty(N, np.float64)
    out3 = np.empty(3, np.float64)
    lib().oracle_load_stats(ctypes.byref(c), _p(u), _p(s), _p(idx, ctypes.c_int32),
                            _p(counts, ctypes.c_int64), _p(f), _p(P), _p(out3))
    return LoadStats(counts, f, P, float(out3[0]), float(out3[1]), float(out3[2]))


def seq_balance_loss(cfg, u, s, idx, seq_len: int):
    """Sequence-wise balance loss ("DeepSeek MoE：从v1到v3的演进", DeepSeek-v3, sequence粒度的
    负载均衡loss): the expert-level balance loss of the ST-MoE section, computed within each
    sequence instead of over the batch, averaged over the sequences. The page prints no formula;
    the reading taken is L_seq = (1/B) sum_b L_B(tokens of sequence b), with f and P of each
    sequence defined as for the batch. The batch is B = T / seq_len consecutive sequences.
    -> (per-sequence losses [B], their mean)."""
    u, s = _f64(u), _f64(s)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T = u.shape[0]
    assert seq_len > 0 and T % seq_len == 0
    per = np.array([load_stats(cfg, u[b:b + seq_len], s[b:b + seq_len], idx[b:b + seq_len]).lb
                    for b in range(0, T, seq_len)], dtype=np.float64)
    return per, float(per.mean())


def group_balance_losses(cfg, u, s, idx):
    """Device-level and communication balance losses ("DeepSeek MoE：从v1到v3的演进",
    DeepSeek-v1 设备级负载loss and DeepSeek-v2 通信负载均衡loss). The page describes them in words
    only; the reading taken follows the expert-level loss of the ST-MoE section with the
    n_groups devices (expert e on device e / (N / G)) as the units:
      f'_d = sum over e on d of f_e   (share of the batch's assignments d computes),
      P'_d = sum over e on d of P_e   (share of the router score d receives),
      L_dev = G * sum_d f'_d P'_d;
      R_d  = number of tokens with at least one chosen expert on d (tokens d receives),
      f''_d = R_d / sum_d' R_d',  L_comm = G * sum_d f''_d P'_d.
    Both are 1 when routing is uniform. -> (L_dev, L_comm)."""
    st = load_stats(cfg, u, s, idx)
    G, N = cfg.n_groups, cfg.n_routed
    per = N // G
    dev_of = np.arange(N) // per
    f_dev = np.zeros(G)
    p_dev = np.zeros(G)
    for e in range(N):
        f_dev[dev_of[e]] += st.f[e]
        p_dev[dev_of[e]] += st.P[e]
    recv = np.zeros(G)
    idx = np.asarray(idx)
    for t in range(idx.shape[0]):
        for d in sorted(set(int(e) // per for e in idx[t])):
            recv[d] += 1
    l_dev = G * float(np.sum(f_dev * p_dev))
    l_comm = G * float(np.sum(recv / recv.sum() * p_dev))
    return l_dev, l_comm


def capacity_drop(cfg, idx, w) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = _f64(w)
    T = idx.shape[0]
    c = _cfg(cfg, T)
    kept = np.empty(idx.shape, np.uint8)
    lib().oracle_capacity_drop(ctypes.byref(c), _p(idx, ctypes.c_int32), _p(w),
                               _p(kept, ctypes.c_uint8))
    return kept


def permute(cfg, idx, kept=None):
    """-> (offsets [N+1], row_token [R], slot_row [T,K]) as int32."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T = idx.shape[0]
    c = _cfg(cfg, T)
    R = int(idx.size if kept is None else int(np.count_nonzero(kept)))
    offsets = np.empty(cfg.n_routed + 1, np.int32)
    row_token = np.empty(max(R, 1), np.int32)
    slot_row = np.empty(idx.shape, np.int32)
    kp = None if kept is None else np.ascontiguousarray(kept, dtype=np.uint8)
    lib().oracle_permute(ctypes.byref(c), _p(idx, ctypes.c_int32), _p(kp, ctypes.c_uint8),
                         _p(offsets, ctypes.c_int32), _p(row_token, ctypes.c_int32),
                         _p(slot_row, ctypes.c_int32))
    return offsets, row_token[:R], slot_row


def swiglu_rows(x_rows, w13, w2) -> np.ndarray:
    """SwiGLU expert on rows. Weights: float arrays, or bf16 torch tensors (widened exactly)."""
    x_rows = _f64(x_rows)
    n, H = x_rows.shape
    y = np.empty((n, H), np.float64)
    if _is_bf16_tensor(w13):
        I = int(w2.shape[1])
        assert tuple(w13.shape) == (2 * I, H) and tuple(w2.shape) == (H, I)
        b13 = _bf16_bits(w13)
        b2 = _bf16_bits(w2)
        if n:
            lib().oracle_swiglu_rows_bf16w(n, H, I, _p(x_rows), _p(b13, ctypes.c_uint16),
                                           _p(b2, ctypes.c_uint16), _p(y))
        return y
    w13, w2 = _f64(w13), _f64(w2)
    I = w2.shape[1]
    assert w13.shape == (2 * I, H) and w2.shape == (H, I)
    if n:
        lib().oracle_swiglu_rows(n, H, I, _p(x_rows), _p(w13), _p(w2), _p(y))
    return y


def _is_bf16_tensor(t) -> bool:
    try:
        import torch
    except ImportError:  # pragma: no cover
        return False
    return isinstance(t, torch.Tensor) and t.dtype == torch.bfloat16


def _bf16_bits(t) -> np.ndarray:
    import torch
    return np.ascontiguousarray(t.detach().to("cpu").contiguous().view(torch.int16).numpy()
                                .view(np.uint16))


def combine(y_rows, slot_row, w, y_shared=None) -> np.ndarray:
    y_rows = _f64(y_rows)
    slot_row = np.ascontiguousarray(slot_row, dtype=np.int32)
    w = _f64(w)
    T, K = slot_row.shape
    H = y_rows.shape[1] if y_rows.ndim == 2 and y_rows.shape[0] else (
        y_shared.shape[1] if y_shared is not None else 0)
    ys = None if y_shared is None else _f64(y_shared)
    out = np.empty((T, H), np.float64)
    if y_rows.shape[0] == 0:
        y_rows = np.zeros((1, H), np.float64)
    lib().oracle_combine(T, H, K, _p(y_rows), _p(slot_row, ctypes.c_int32), _p(w), _p(ys), _p(out))
    return out


def bias_update(counts, rate: float, b) -> np.ndarray:
    counts = np.ascontiguousarray(counts, dtype=np.int64)
    b = _f64(b).copy()
    lib().oracle_bias_update(len(b), _p(counts, ctypes.c_int64), ctypes.c_double(float(rate)), _p(b))
    return b


# ---------------------------------------------------------------- whole layer
def layer_forward(cfg, x, w_gate, gate_bias, select_bias, expert_weights, shared_weights,
                  tokens=None, u=None):
    """One layer forward in fp64.

    x [T,H] (any float array), w_gate [N,H]; expert_weights(e) -> (W13 [2I,H], W2 [H,I]) and
    shared_weights(s) -> the same for shared expert s, both as float64 arrays (fetched one
    expert at a time so full-size layers fit in host memory).
    tokens: optional sorted token subset whose outputs are computed. Routing always covers
    the tokens the result depends on: every token when the v2 drop is on (the drop ranks the
    whole batch), only the subset otherwise.
    u: optional precomputed logits [T,N] for the routed tokens (tests feed identical logits).
    Returns a dict with u, s, idx, w, margin, kept, offsets/row_token/slot_row (full batch
    only), the token list and out [len(tokens), H].
    """
    T = x.shape[0]  # x: an array, or any object giving rows through x[row_indices]
    all_tokens = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    route_tokens = np.arange(T) if (cfg.capacity_drop or tokens is None) else all_tokens
    if u is None:
        u_r = gate_logits(x[route_tokens], w_gate, gate_bias)
    else:
        u_r = _f64(u)[route_tokens]
    s_r = scores(u_r, cfg.score_fn)
    idx_r, w_r, margin_r = route(cfg, s_r, select_bias, u=u_r)
    kept_r = capacity_drop(cfg.replace(T=len(route_tokens)), idx_r, w_r) if cfg.capacity_drop \
        else np.ones(idx_r.shape, np.uint8)
    res = dict(route_tokens=route_tokens, u=u_r, s=s_r, idx=idx_r, w=w_r, margin=margin_r,
               kept=kept_r)
    if tokens is None:
        offs, row_token, slot_row = permute(cfg, idx_r, kept_r)
        res.update(offsets=offs, row_token=row_token, slot_row=slot_row)

    # position of each output token inside the routed arrays
    pos = np.searchsorted(route_tokens, all_tokens)
    idx_o, w_o, kept_o = idx_r[pos], w_r[pos], kept_r[pos]
    xo = _f64(x[all_tokens])
    n, H, K = len(all_tokens), cfg.hidden, cfg.top_k
    # rows of this output subset, one per kept assignment, grouped by expert
    slot = -np.ones((n, K), np.int32)
    y_rows = np.zeros((int(kept_o.sum()), H), np.float64)
    r0 = 0
    for e in np.unique(idx_o[kept_o.astype(bool)]):
        tt, kk = np.nonzero((idx_o == e) & kept_o.astype(bool))
        w13, w2 = expert_weights(int(e))
        y_rows[r0:r0 + len(tt)] = swiglu_rows(xo[tt], w13, w2)
        slot[tt, kk] = np.arange(r0, r0 + len(tt), dtype=np.int32)
        r0 += len(tt)
    y_sh = np.zeros((n, H), np.float64)
    for s_ in range(cfg.n_shared):
        w13, w2 = shared_weights(s_)
        y_sh += swiglu_rows(xo, w13, w2)
    res["tokens"] = all_tokens
    res["out"] = combine(y_rows, slot, w_o, y_sh)
    return res


# ---------------------------------------------------------------- expert placement planner
def plan_placement(load, n_gpus: int, slots: int, n_nodes: int = 1, n_groups: int = 0):
    """Redundant-expert placement ("DeepSeek-V3的Group-Limited Expert Routing与负载均衡优化实践",
    sections 2 and 4: give hot experts replicas, place replicas on GPUs; hierarchically for
    prefill: expert groups to nodes first). The pages name the steps; the rules taken:
      replicate: one extra replica at a time to the expert with the largest load per replica
        (ties: lower expert), among experts with fewer replicas than GPUs while any remains;
      place: replicas by decreasing load per replica (ties: lower expert, lower replica) onto the
        least-loaded GPU with a free slot not yet hosting that expert (ties: lower GPU), else
        onto the least-loaded GPU with a free slot;
      groups (n_nodes > 1): by decreasing load (ties: lower group) onto the least-loaded node
        with room for one more group.
    Plain loops, fractions for the replication comparisons.
    -> (replicas [N], gpu_expert [n_gpus][slots] with -1 for empty slots, gpu_load [n_gpus])."""
    from fractions import Fraction
    load = [int(v) for v in load]
    N = len(load)
    reps = [0] * N
    hosted = [[] for _ in range(n_gpus)]
    gload = [0.0] * n_gpus

    def replicate(ids, total, cap):
        for e in ids:
            reps[e] = 1
        for _ in range(total - len(ids)):
            below = [e for e in ids if reps[e] < cap]
            cand = below if below else list(ids)
            best = max(cand, key=lambda e: (Fraction(load[e], reps[e]), -e))
            reps[best] += 1

    def place(ids, gpus):
        items = [(load[e] / reps[e], e, j) for e in ids for j in range(reps[e])]
        items.sort(key=lambda it: (-it[0], it[1], it[2]))
        for w, e, _ in items:
            free = [g for g in gpus if len(hosted[g]) < slots]
            fresh = [g for g in free if e not in hosted[g]]
            pool = fresh if fresh else free
            g = min(pool, key=lambda g: (gload[g], g))
            hosted[g].append(e)
            gload[g] += w

    if n_nodes <= 1:
        replicate(list(range(N)), n_gpus * slots, n_gpus)
        place(list(range(N)), list(range(n_gpus)))
    else:
        gpn, per, gpnode = n_gpus // n_nodes, N // n_groups, n_groups // n_nodes
        gl = [sum(load[g * per:(g + 1) * per]) for g in range(n_groups)]
        order = sorted(range(n_groups), key=lambda g: (-gl[g], g))
        nl, nc, node_groups = [0] * n_nodes, [0] * n_nodes, [[] for _ in range(n_nodes)]
        for g in order:
            n = min((n for n in range(n_nodes) if nc[n] < gpnode), key=lambda n: (nl[n], n))
            node_groups[n].append(g)
            nc[n] += 1
            nl[n] += gl[g]
        for n in range(n_nodes):
            ids = [e for g in sorted(node_groups[n]) for e in range(g * per, (g + 1) * per)]
            replicate(ids, gpn * slots, gpn)
            place(ids, list(range(n * gpn, (n + 1) * gpn)))
    ge = np.full((n_gpus, slots), -1, np.int32)
    for g in range(n_gpus):
        ge[g, :len(hosted[g])] = hosted[g]
    return np.array(reps, np.int32), ge, np.array(gload, np.float64)
