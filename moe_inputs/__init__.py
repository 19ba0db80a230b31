"""Seeded synthetic inputs for the DeepSeekMoE layer forward.

This module is shared by the CUDA path's tests/bench and by the fp64 oracle.
It holds layer shapes and random draws only: no step of the method (no gate,
no routing, no expert math) is computed here.

Shapes follow the model descriptions on the pages:
  * "DeepSeek MoE：从v1到v3的演进" (wln20.github.io), DeepSeek-v2 / v3 sections:
    160 routed experts / 6 active (v2), 256 routed / 8 active (v3).
  * "DeepSeek-V3的Group-Limited Expert Routing与负载均衡优化实践" (mhpn.cn), section 1:
    256 experts in 8 groups of 32, keep 4 groups, pick 8.
Everything else (hidden sizes, intermediate sizes, init std, offsets) is the
synthetic workload recipe of this library; nothing is a trained weight.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass

import torch

__all__ = ["LayerConfig", "CONFIGS", "make_weights", "make_router", "make_x", "make_logits",
           "expert_weights_f64", "to_f64"]


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int                  # tokens in the batch
    hidden: int             # H
    n_routed: int           # N routed experts
    n_groups: int           # G expert groups (v3) or virtual devices (v2); 1 = no limit
    topk_groups: int        # groups (or devices, M) each token may use
    top_k: int              # K routed experts per token
    group_score_topn: int   # group score = sum of its top-n selection scores (1 = max)
    score_fn: str           # "softmax" | "sigmoid"
    norm_topk: bool         # renormalise the K weights to sum 1
    routed_scale: float     # multiply routed weights by this
    n_shared: int           # S always-on shared experts
    inter: int              # I, intermediate size of one (fine-grained) expert
    capacity_drop: bool     # v2 device-level token drop
    dtype: str              # "f32" | "bf16"
    w_std: float            # std of expert weights
    gate_std: float         # std of the router weight W_g
    select_bias_std: float  # std of the v3 selection bias b (0 = zero bias vector)
    has_select_bias: bool   # pass a selection bias vector at all
    logit_offset: str       # "none" | "normal" (N(0,1) per expert) | "zipf"
    zipf_s: float = 1.2

    def replace(self, **kw) -> "LayerConfig":
        return dataclasses.replace(self, **kw)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


_V3 = dict(hidden=7168, n_routed=256, n_groups=8, topk_groups=4, top_k=8, group_score_topn=2,
           score_fn="sigmoid", norm_topk=True, routed_scale=2.5, n_shared=1, inter=2048,
           capacity_drop=False, dtype="bf16", w_std=0.006, gate_std=0.006, select_bias_std=0.1,
           has_select_bias=True)

CONFIGS: dict[str, LayerConfig] = {
    # Tiny oracle layer, fp32.
    "tiny": LayerConfig("tiny", T=64, hidden=128, n_routed=16, n_groups=4, topk_groups=2,
                        top_k=4, group_score_topn=2, score_fn="sigmoid", norm_topk=True,
                        routed_scale=1.0, n_shared=1, inter=64, capacity_drop=False, dtype="f32",
                        w_std=0.02, gate_std=0.02, select_bias_std=0.0, has_select_bias=True,
                        logit_offset="none"),
    # DeepSeekMoE (v1) style: softmax gate, 64 fine-grained experts, top-6, no group limit.
    "v1": LayerConfig("v1", T=4096, hidden=2048, n_routed=64, n_groups=1, topk_groups=1, top_k=6,
                      group_score_topn=1, score_fn="softmax", norm_topk=False, routed_scale=1.0,
                      n_shared=2, inter=1408, capacity_drop=False, dtype="bf16", w_std=0.02,
                      gate_std=0.02, select_bias_std=0.0, has_select_bias=False,
                      logit_offset="none"),
    # DeepSeek-V2 style: 160 experts on 8 virtual devices of 20, M=3 devices, top-6, drop.
    "v2": LayerConfig("v2", T=8192, hidden=5120, n_routed=160, n_groups=8, topk_groups=3, top_k=6,
                      group_score_topn=1, score_fn="softmax", norm_topk=False, routed_scale=1.0,
                      n_shared=2, inter=1536, capacity_drop=True, dtype="bf16", w_std=0.02,
                      gate_std=0.02, select_bias_std=0.0, has_select_bias=False,
                      logit_offset="normal"),
    # DeepSeek-V3 style prefill.
    "v3_prefill": LayerConfig("v3_prefill", T=16384, logit_offset="none", **_V3),
    # DeepSeek-V3 style decode steps, Zipf(1.2) expert popularity through a logit offset.
    "v3_decode_32": LayerConfig("v3_decode_32", T=32, logit_offset="zipf", **_V3),
    "v3_decode_128": LayerConfig("v3_decode_128", T=128, logit_offset="zipf", **_V3),
    "v3_decode_512": LayerConfig("v3_decode_512", T=512, logit_offset="zipf", **_V3),
    # Profiling case of the V3 prefill GEMMs: the same shapes and per-expert load (512 rows per
    # expert on average) with 1/8 of the experts and tokens, so that a detailed profiler
    # capture holds about 3 GB on the device while its operands still exceed L2.
    "v3_prefill_e32": LayerConfig("v3_prefill_e32", T=2048, logit_offset="none",
                                  **{**_V3, "n_routed": 32}),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, std, g, device, dtype):
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(dtype)


def logit_offset(cfg: LayerConfig, g: torch.Generator, device) -> torch.Tensor | None:
    """Per-expert additive logit offset that skews expert popularity.

    normal: offset_e ~ N(0, 1).
    zipf:   offset_e = -s * ln(rank_e) with rank a seeded permutation of 1..N, so that
            exp(offset) follows a Zipf(s) popularity law over experts.
    """
    N = cfg.n_routed
    if cfg.logit_offset == "none":
        return None
    if cfg.logit_offset == "normal":
        return torch.randn((N,), generator=g, device=device, dtype=torch.float32)
    if cfg.logit_offset == "zipf":
        perm = torch.randperm(N, generator=g, device=device)
        rank = (perm + 1).to(torch.float64)
        return (-cfg.zipf_s * torch.log(rank)).to(torch.float32)
    raise ValueError(cfg.logit_offset)


def _router_draws(cfg: LayerConfig, g: torch.Generator, device) -> dict:
    out = {"w_gate": _randn((cfg.n_routed, cfg.hidden), cfg.gate_std, g, device,
                            cfg.torch_dtype)}
    out["gate_logit_bias"] = logit_offset(cfg, g, device)
    if cfg.has_select_bias:
        if cfg.select_bias_std > 0:
            out["select_bias"] = torch.randn((cfg.n_routed,), generator=g, device=device,
                                             dtype=torch.float32) * cfg.select_bias_std
        else:
            out["select_bias"] = torch.zeros((cfg.n_routed,), device=device, dtype=torch.float32)
    else:
        out["select_bias"] = None
    return out


def make_router(cfg: LayerConfig, device="cpu", seed: int = 0) -> dict:
    """w_gate, gate_logit_bias, select_bias: the first draws of make_weights (same values)."""
    return _router_draws(cfg, _gen(device, seed + 1), device)


def make_weights(cfg: LayerConfig, device="cpu", seed: int = 0) -> dict:
    """All layer parameters, in the config dtype (router bias and selection bias in fp32).

    Draw order: x is drawn first by make_x with the same seed; here W_g, gate_logit_bias,
    select_bias, shared W13/W2, then routed W13/W2 expert by expert.
      w_gate            [N, H]
      gate_logit_bias   [N] fp32 or None  (router linear bias; carries the skew offsets)
      select_bias       [N] fp32 or None  (v3 selection-only bias b_i)
      w13_shared        [S, 2I, H]  rows 0..I-1 gate projection, I..2I-1 up projection
      w2_shared         [S, H, I]
      w13               [N, 2I, H]
      w2                [N, H, I]
    """
    dt = cfg.torch_dtype
    H, N, S, I = cfg.hidden, cfg.n_routed, cfg.n_shared, cfg.inter
    g = _gen(device, seed + 1)
    out = _router_draws(cfg, g, device)
    out["w13_shared"] = torch.empty((S, 2 * I, H), device=device, dtype=dt)
    out["w2_shared"] = torch.empty((S, H, I), device=device, dtype=dt)
    for s in range(S):
        out["w13_shared"][s] = _randn((2 * I, H), cfg.w_std, g, device, dt)
        out["w2_shared"][s] = _randn((H, I), cfg.w_std, g, device, dt)
    out["w13"] = torch.empty((N, 2 * I, H), device=device, dtype=dt)
    out["w2"] = torch.empty((N, H, I), device=device, dtype=dt)
    for e in range(N):
        out["w13"][e] = _randn((2 * I, H), cfg.w_std, g, device, dt)
        out["w2"][e] = _randn((H, I), cfg.w_std, g, device, dt)
    return out


def make_x(cfg: LayerConfig, device="cpu", seed: int = 0, T: int | None = None) -> torch.Tensor:
    """Token activations x [T, H] ~ N(0, 1) in the config dtype."""
    T = cfg.T if T is None else T
    g = _gen(device, seed)
    return _randn((T, cfg.hidden), 1.0, g, device, cfg.torch_dtype)


def make_logits(cfg: LayerConfig, seed: int = 0, T: int | None = None,
                device="cpu") -> torch.Tensor:
    """Synthetic router logits u [T, N] fp32 for routing-only parity.

    Distribution of x W_g^T for x ~ N(0,1), W_g ~ N(0, gate_std): N(0, H gate_std^2),
    plus the config's per-expert offset.
    """
    T = cfg.T if T is None else T
    g = _gen(device, seed + 7)
    sd = math.sqrt(cfg.hidden) * cfg.gate_std
    u = torch.randn((T, cfg.n_routed), generator=g, device=device, dtype=torch.float32) * sd
    off = logit_offset(cfg, g, device)
    if off is not None:
        u = u + off[None, :]
    return u


def to_f64(t: torch.Tensor):
    """Widen a tensor (any device, any float dtype) to a contiguous float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).contiguous().numpy()


def expert_weights_f64(w: dict, e: int, shared: bool = False):
    """(W13 [2I,H], W2 [H,I]) of one routed (or shared) expert as float64 numpy arrays."""
    if shared:
        return to_f64(w["w13_shared"][e]), to_f64(w["w2_shared"][e])
    return to_f64(w["w13"][e]), to_f64(w["w2"][e])
