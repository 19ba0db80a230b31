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
