"""The whole layer forward (moe_layer_forward) on the GPU against the fp64 oracle.

The oracle computes its own logits from the same bf16 (or fp32) x and weights. Output rows are
compared by relative Frobenius error (1e-2 bf16, 1e-5 fp32). Tokens whose oracle routing
margin is below 1e-4 (their expert set may legitimately flip under fp32 vs fp64 logits) are
excluded and reported; with the v2 drop, so are tokens holding an assignment whose weight lies
within 1e-4 of its device's capacity cut (the same margin rule applied to the drop decision).
"""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import CONFIGS, make_weights, make_x
from tests.helpers import MID_A, MID_B, MID_ODD, MID_V2, rel_frob, sample_tokens, tol_for, workspace

pytestmark = pytest.mark.gpu

CFGS = {**CONFIGS, "mid_a": MID_A, "mid_b": MID_B, "mid_v2": MID_V2, "mid_odd": MID_ODD}


def _near_cut_tokens(cfg, idx, w, kept, margin=1e-4):
    """Tokens with an assignment whose drop decision has a margin below `margin`: on a device
    that drops, its routing weight lies within `margin` of the cut (the weight of the device's
    last kept assignment). The same rule as for the expert choice: the GPU's logits differ from
    the oracle's fp64 ones by rounding, so such a decision may legitimately flip."""
    per = cfg.n_routed // cfg.n_groups
    dev = (idx // per).ravel()
    wf = w.ravel()
    kf = kept.ravel().astype(bool)
    out = set()
    for d in range(cfg.n_groups):
        a = np.nonzero(dev == d)[0]
        if kf[a].all():
            continue
        w_cut = wf[a][kf[a]].min()
        for r in a[np.abs(wf[a] - w_cut) < margin]:
            out.add(int(r // cfg.top_k))
    return out


def _run(cfg, n_sample):
    import mixture_experts_routing_sigmoid_b300 as moe
    T = cfg.T
    w = make_weights(cfg, device="cuda")
    x = make_x(cfg, device="cuda", seed=2)
    out = torch.full((T, cfg.hidden), float("nan"), dtype=x.dtype, device="cuda")
    counts = torch.empty(cfg.n_routed, dtype=torch.int32, device="cuda")
    lbz = torch.empty(3, dtype=torch.float32, device="cuda")
    ws = workspace(cfg, T)
    moe.moe_layer_forward(cfg, T, x, w, out, counts, lbz, ws)
    assert moe.moe_get_error() == 0
    assert int(counts.sum()) == T * cfg.top_k
    tok = sample_tokens(T, n_sample, seed=4)
    f64 = (lambda t: t.double().cpu().numpy())
    ew = (lambda e: (w["w13"][e], w["w2"][e])) if cfg.dtype == "bf16" else \
        (lambda e: (f64(w["w13"][e]), f64(w["w2"][e])))
    sw = (lambda s: (w["w13_shared"][s], w["w2_shared"][s])) if cfg.dtype == "bf16" else \
        (lambda s: (f64(w["w13_shared"][s]), f64(w["w2_shared"][s])))
    gb = None if w["gate_logit_bias"] is None else f64(w["gate_logit_bias"])
    sb = None if w["select_bias"] is None else f64(w["select_bias"])
    xin = f64(x) if (cfg.capacity_drop or n_sample >= T) else x
    res = oracle.layer_forward(cfg, xin if not isinstance(xin, torch.Tensor) else
                               _RowFetcher(x), f64(w["w_gate"]), gb, sb, ew, sw,
                               tokens=None if n_sample >= T else tok)
    tokens = res["tokens"]
    pos = np.searchsorted(res["route_tokens"], tokens)
    ok = res["margin"][pos] >= 1e-4
    n_margin = int((~ok).sum())
    n_cut = 0
    if cfg.capacity_drop:
        near = _near_cut_tokens(cfg, res["idx"], res["w"], res["kept"])
        cut = np.array([t in near for t in tokens])
        n_cut = int((cut & ok).sum())
        ok &= ~cut
        print(f"{cfg.name}: {len(near)} of {len(res['route_tokens'])} tokens of the batch hold "
              f"an assignment within 1e-4 of a device's cut")
    n_ex = int((~ok).sum())
    print(f"{cfg.name}: {n_ex} of {len(tokens)} compared tokens excluded "
          f"({n_margin} by the routing margin, {n_cut} more by the drop margin)")
    assert n_ex <= max(3, len(tokens) // 10)
    got = out[torch.from_numpy(tokens).long().cuda()].double().cpu().numpy()
    err = rel_frob(got[ok], res["out"][ok])
    print(f"{cfg.name}: relative Frobenius error {err:.3e}")
    assert np.isfinite(got).all()
    assert err <= tol_for(cfg)
    return res


class _RowFetcher:
    """Gives the oracle x rows of a CUDA tensor on demand (as fp64) without copying all of x."""

    def __init__(self, x):
        self.x, self.shape = x, tuple(x.shape)

    def __getitem__(self, rows):
        return self.x[torch.as_tensor(np.asarray(rows)).long().cuda()].double().cpu().numpy()


@pytest.mark.parametrize("name,n_sample", [("tiny", 64), ("mid_a", 300), ("mid_b", 517),
                                           ("mid_v2", 640), ("mid_odd", 333)])
def test_layer_small_whole(name, n_sample):
    _run(CFGS[name], n_sample)


@pytest.mark.parametrize("name,n_sample", [("v1", 48), ("v2", 32), ("v3_prefill", 16),
                                           ("v3_decode_32", 32), ("v3_decode_128", 24),
                                           ("v3_decode_512", 24)])
def test_layer_full_size_sampled(name, n_sample):
    _run(CFGS[name], n_sample)


@pytest.mark.parametrize("T", [1, 2, 33, 64, 65, 128, 129])
def test_layer_odd_token_counts(T):
    _run(MID_A.replace(T=T), T)
    _run(CONFIGS["v3_decode_32"].replace(T=T), min(T, 8))
