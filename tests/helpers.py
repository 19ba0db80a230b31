"""Shared helpers of the GPU parity tests: buffers, C-ABI calls, comparisons."""
from __future__ import annotations

import numpy as np
import torch

from moe_inputs import CONFIGS, LayerConfig

# Small bf16 layers that still span several tiles, ragged segment tails, empty experts,
# a partial 256-column output tile and a K loop longer than the smem ring.
MID_A = CONFIGS["v3_prefill"].replace(
    name="mid_a", T=300, hidden=512, n_routed=16, n_groups=4, topk_groups=2, top_k=4,
    group_score_topn=2, n_shared=2, inter=256, w_std=0.05, gate_std=0.06,
    logit_offset="zipf")
MID_B = CONFIGS["v1"].replace(
    name="mid_b", T=517, hidden=384, n_routed=32, top_k=6, n_shared=1, inter=384, w_std=0.05,
    gate_std=0.05, logit_offset="normal")
MID_V2 = CONFIGS["v2"].replace(name="mid_v2", T=640, hidden=256, n_routed=40, n_groups=8,
                               topk_groups=3, top_k=6, n_shared=1, inter=128, w_std=0.05,
                               gate_std=0.06)
# K = hidden = 320 is an odd multiple of 64: the router and up-projection GEMMs' last k block
# holds one 64-element unit (and the router's split K range ends in it at small T)
MID_ODD = CONFIGS["v3_prefill"].replace(
    name="mid_odd", T=333, hidden=320, n_routed=24, n_groups=4, topk_groups=2, top_k=4,
    group_score_topn=2, n_shared=2, inter=256, w_std=0.05, gate_std=0.06,
    logit_offset="zipf")


def rel_frob(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def tol_for(cfg: LayerConfig) -> float:
    """Layer-output tolerance (relative Frobenius): 1e-2 for bf16, 1e-5 for fp32."""
    return 1e-2 if cfg.dtype == "bf16" else 1e-5


def dev_weights(w: dict, device="cuda") -> dict:
    return {k: (None if v is None else v.to(device).contiguous()) for k, v in w.items()}


def workspace(cfg, T, device="cuda"):
    import mixture_experts_routing_sigmoid_b300 as moe
    n = moe.moe_workspace_size(cfg, T)
    assert n > 0
    return torch.empty(n, dtype=torch.uint8, device=device)


def gpu_route(cfg, T, logits=None, x=None, weights=None, ws=None):
    import mixture_experts_routing_sigmoid_b300 as moe
    idx = torch.empty((T, cfg.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, cfg.top_k), dtype=torch.float32, device="cuda")
    lo = None if logits is not None else torch.empty((T, cfg.n_routed), dtype=torch.float32,
                                                    device="cuda")
    if ws is None:
        ws = workspace(cfg, T)
    moe.moe_route(cfg, T, x, weights, logits, lo, idx, w, ws)
    assert moe.moe_get_error() == 0
    return idx, w, lo


def gpu_permute(cfg, T, idx, w, x=None, ws=None, row_w=None):
    import mixture_experts_routing_sigmoid_b300 as moe
    A = T * cfg.top_k
    offsets = torch.empty(cfg.n_routed + 1, dtype=torch.int32, device="cuda")
    row_token = torch.full((max(A, 1),), -7, dtype=torch.int32, device="cuda")
    slot_row = torch.empty((max(A, 1),), dtype=torch.int32, device="cuda")
    x_perm = None
    if x is not None:
        x_perm = torch.zeros((max(A, 1), cfg.hidden), dtype=x.dtype, device="cuda")
    if ws is None:
        ws = workspace(cfg, T)
    moe.moe_permute(cfg, T, idx, w, x, offsets, row_token, slot_row, x_perm, ws, row_w=row_w)
    assert moe.moe_get_error() == 0
    return offsets, row_token, slot_row, x_perm


def sample_tokens(T: int, n: int, seed: int = 0) -> np.ndarray:
    if n >= T:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    s = np.sort(rng.choice(T, size=n, replace=False))
    # always include the first and last token (tile edges)
    return np.unique(np.concatenate([[0, T - 1], s]))



def gemm_tiles(cfg: LayerConfig, offs, mode: str):
    """The expert GEMM's tiles in the kernel's order, restated from its tile rule: problems by
    decreasing rows (ties: lower index; the shared experts are problem n_routed with T rows),
    then feature tiles (up: 128 intermediate features, down: 256 hidden features), then token
    tiles (a segment's rows cut into equal tiles of at most 256, multiples of 16).
    Returns [(problem, first feature, end feature, first row, end row)], rows relative to the
    problem's segment."""
    rows = [int(r) for r in np.diff(np.asarray(offs))]
    if cfg.n_shared > 0:
        rows.append(cfg.T)
    order = sorted(range(len(rows)), key=lambda q: (-rows[q], q))
    out = []
    for q in order:
        r = rows[q]
        if r <= 0:
            continue
        shared = q == cfg.n_routed
        if mode == "up":
            feats, per_tile = (cfg.n_shared * cfg.inter if shared else cfg.inter), 128
        else:
            feats, per_tile = cfg.hidden, 256
        ntt = -(-r // 256)
        per = (-(-r // ntt) + 15) // 16 * 16
        for ft in range(-(-feats // per_tile)):
            for tt in range(ntt):
                out.append((q, ft * per_tile, min(feats, (ft + 1) * per_tile), tt * per,
                            min(r, (tt + 1) * per)))
    return out


def gemm_tail_split(cfg: LayerConfig, offs, mode: str, pairs: int = 74):
    """The up projection's tail split (the down projection cuts nothing), restated from the
    kernel's rule to tell the tests which tiles it cuts along K: with W tiles (gemm_tiles) on
    `pairs` CTA pairs, the last R = W mod pairs tiles (all W when W < pairs) are cut into
    S = min(pairs // R, 8, routed k blocks // 8, 80 // R) pieces when R <= pairs / 2, R <= 40
    and S >= 2. Returns (W, R, S), with R = S = 0 when nothing is split."""
    W = len(gemm_tiles(cfg, offs, mode))
    if mode != "up":
        return W, 0, 0
    k_routed = cfg.hidden if mode == "up" else cfg.inter
    kb = -(-(k_routed // 64) // 2)
    if W <= 0 or pairs <= 1:
        return W, 0, 0
    R = W % pairs
    if R == 0 or 2 * R > pairs or R > 40:
        return W, 0, 0
    S = min(pairs // R, 8, kb // 8, 80 // R)
    return (W, R, S) if S >= 2 else (W, 0, 0)
