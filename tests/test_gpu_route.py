"""Routing and load statistics on the GPU against the fp64 oracle.

Fed identical logits, the chosen experts are bit-exact and the weights agree within 1e-5
(absolute). With the v2 drop on, weights are the correctly rounded fp32 values, so they equal
the oracle's rounded to fp32. End to end (logits from the tensor-core gate GEMM), tokens whose
oracle decision margin is below 1e-4 are excluded from the index comparison and reported.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import CONFIGS, make_logits, make_router, make_x
from tests.helpers import MID_A, MID_B, MID_ODD, MID_V2, gpu_route, sample_tokens, workspace

pytestmark = pytest.mark.gpu

ROUTE_CFGS = {**CONFIGS, "mid_a": MID_A, "mid_b": MID_B, "mid_v2": MID_V2, "mid_odd": MID_ODD,
              "k16": CONFIGS["v1"].replace(name="k16", T=1000, n_routed=64, n_groups=4,
                                           topk_groups=4, top_k=16, group_score_topn=2,
                                           score_fn="sigmoid", norm_topk=True,
                                           routed_scale=1.5, has_select_bias=True,
                                           select_bias_std=0.05),
              # 128 experts: four per lane (the routing and statistics kernels' JM = 4 builds),
              # at a batch above and one below the large-batch routing kernel's threshold
              "n128": CONFIGS["v3_prefill"].replace(name="n128", T=2000, n_routed=128,
                                                    n_groups=8, topk_groups=4, top_k=8),
              "n128_small": CONFIGS["v3_prefill"].replace(name="n128_small", T=300,
                                                          n_routed=128, n_groups=8,
                                                          topk_groups=4, top_k=8)}


def _oracle_route(cfg, u, sb):
    u64 = u.double().numpy()
    s = oracle.scores(u64, cfg.score_fn)
    return oracle.route(cfg, s, None if sb is None else sb.double().numpy(), u=u64)


def _check_route(cfg, u, sb, what=""):
    T = u.shape[0]
    idx_o, w_o, _ = _oracle_route(cfg, u, sb)
    w = {"select_bias": None if sb is None else sb.cuda()}
    idx_g, w_g, _ = gpu_route(cfg, T, logits=u.cuda(), weights=w)
    idx_g, w_g = idx_g.cpu().numpy(), w_g.cpu().numpy()
    bad = np.nonzero((idx_g != idx_o).any(axis=1))[0]
    assert len(bad) == 0, f"{what}: {len(bad)} tokens differ, first {bad[:5]}"
    assert np.abs(w_g - w_o).max() <= 1e-5
    if cfg.capacity_drop:
        np.testing.assert_array_equal(w_g, w_o.astype(np.float32))
    return idx_o, w_o


@pytest.mark.parametrize("name", list(ROUTE_CFGS))
def test_route_identical_logits_bit_exact(name):
    cfg = ROUTE_CFGS[name]
    u = make_logits(cfg, seed=3)
    sb = make_router(cfg)["select_bias"]
    _check_route(cfg, u, sb, name)


@pytest.mark.parametrize("name", ["tiny", "v3_prefill", "v1", "v2", "k16"])
def test_route_ties_and_near_ties(name):
    """Exact ties (equal logits, zero bias), 1-ulp neighbours, and duplicated groups: the
    tie rule (lower group, lower expert) must hold exactly as in the oracle."""
    cfg = ROUTE_CFGS[name]
    N, T = cfg.n_routed, 512
    g = torch.Generator().manual_seed(11)
    u = make_logits(cfg, seed=5, T=T).clone()
    u[0:32] = 0.25                                    # every logit equal
    u[32:64] = torch.round(u[32:64] * 4) / 4          # many exact ties
    base = u[64:128].clone()
    u[64:128] = torch.from_numpy(np.nextafter(base.numpy(), np.float32(np.inf)))  # 1-ulp shifts
    u[64:128, ::2] = base[:, ::2]
    gs = N // cfg.n_groups
    if cfg.n_groups > 1:
        u[128:160, gs:2 * gs] = u[128:160, 0:gs]       # two identical groups
    perm = torch.randperm(N, generator=g)
    u[160:192] = u[160:192, perm]
    sb_zero = None if not cfg.has_select_bias else torch.zeros(N)
    _check_route(cfg, u, sb_zero, name + " zero-bias")
    sb = make_router(cfg)["select_bias"]
    _check_route(cfg, u, sb, name + " bias")


def test_route_single_token_and_tail_sizes():
    cfg = CONFIGS["v3_prefill"]
    for T in (1, 7, 33, 255):
        u = make_logits(cfg, seed=T, T=T)
        _check_route(cfg, u, make_router(cfg)["select_bias"], f"T={T}")


@pytest.mark.parametrize("name", ["tiny", "v1", "v2", "v3_prefill", "mid_a", "n128"])
def test_load_stats(name):
    import mixture_experts_routing_sigmoid_b300 as moe
    cfg = ROUTE_CFGS[name]
    T, N = cfg.T, cfg.n_routed
    u = make_logits(cfg, seed=4)
    sb = make_router(cfg)["select_bias"]
    u64 = u.double().numpy()
    s = oracle.scores(u64, cfg.score_fn)
    idx_o, _, _ = oracle.route(cfg, s, None if sb is None else sb.double().numpy(), u=u64)
    st = oracle.load_stats(cfg, u64, s, idx_o)
    counts = torch.empty(N, dtype=torch.int32, device="cuda")
    f = torch.empty(N, dtype=torch.float32, device="cuda")
    P = torch.empty(N, dtype=torch.float32, device="cuda")
    lbz = torch.empty(3, dtype=torch.float32, device="cuda")
    ws = workspace(cfg, T)
    moe.moe_load_stats(cfg, T, u.cuda(), torch.from_numpy(idx_o).cuda(), counts, f, P, lbz, ws)
    assert moe.moe_get_error() == 0
    np.testing.assert_array_equal(counts.cpu().numpy(), st.counts)
    np.testing.assert_allclose(f.cpu().numpy(), st.f, rtol=1e-6)
    np.testing.assert_allclose(P.cpu().numpy(), st.P, rtol=1e-5, atol=1e-7)
    lb, lz, lm = lbz.cpu().numpy().tolist()
    assert abs(lb - st.lb) <= 1e-5 * abs(st.lb)
    assert abs(lz - st.zloss) <= 1e-5 * abs(st.zloss)
    assert abs(lm - st.lse_mean) <= 1e-5 * abs(st.lse_mean)


@pytest.mark.parametrize("name", ["mid_a", "mid_b", "mid_v2", "v1", "v3_prefill",
                                  "v3_decode_128"])
def test_route_end_to_end_from_x(name):
    """Gate GEMM on the tensor cores + routing, against fp64 logits from the same bf16 x, W_g.
    Logits agree to fp32-accumulation accuracy; idx agree except on tokens whose oracle margin
    is below 1e-4 (excluded and reported)."""
    cfg = ROUTE_CFGS[name]
    T = cfg.T
    x = make_x(cfg, device="cuda", seed=2)
    r = make_router(cfg, device="cuda")
    idx_g, w_g, u_g = gpu_route(cfg, T, x=x, weights=r)
    tok = sample_tokens(T, 512, seed=1)
    u_o = oracle.gate_logits(x[tok].cpu().double().numpy(), r["w_gate"].cpu().double().numpy(),
                             None if r["gate_logit_bias"] is None
                             else r["gate_logit_bias"].cpu().double().numpy())
    u_gs = u_g[tok].cpu().double().numpy()
    assert np.abs(u_gs - u_o).max() <= 1e-4 * max(1.0, np.abs(u_o).max())
    if cfg.capacity_drop:
        return  # weights / drop are checked with identical logits above
    sb = r["select_bias"]
    s = oracle.scores(u_o, cfg.score_fn)
    idx_o, w_o, margin = oracle.route(cfg, s, None if sb is None else sb.cpu().double().numpy(),
                                      u=u_o)
    keep = margin >= 1e-4
    n_ex = int((~keep).sum())
    print(f"{name}: {n_ex} of {len(tok)} sampled tokens excluded (margin < 1e-4)")
    assert n_ex <= max(3, len(tok) // 20)
    np.testing.assert_array_equal(idx_g.cpu().numpy()[tok][keep], idx_o[keep])
    assert np.abs(w_g.cpu().numpy()[tok][keep] - w_o[keep]).max() <= 1e-4


@pytest.mark.parametrize("name,T", [("v3_prefill", 256), ("mid_a", 256), ("k16", 256),
                                    ("v3_prefill", 2048)])
def test_route_dense_near_ties_sigmoid(name, T):
    """Every token's keys sit within a few ulps of each other (one logit per token moved by 0-3
    ulps per expert, a selection bias of 0.1 moved by 0-5 ulps per expert), so every group and
    expert decision lies inside the fp32 error bound and is settled by the exact recheck, with
    bands that hold most groups and experts and exact ties among them. At 2048 tokens the batch
    runs the routing kernel built for large batches (fewer registers: the recheck spills)."""
    cfg = ROUTE_CFGS[name]
    N = cfg.n_routed
    rng = np.random.default_rng(21)
    u0 = rng.standard_normal(T).astype(np.float32)
    steps = rng.integers(0, 4, size=(T, N))
    u = u0[:, None].repeat(N, axis=1)
    for k in range(1, 4):
        u = np.where(steps >= k, np.nextafter(u, np.float32(np.inf)), u)
    b = np.full(N, 0.1, dtype=np.float32)
    bsteps = rng.integers(0, 6, size=N)
    for k in range(1, 6):
        b = np.where(bsteps >= k, np.nextafter(b, np.float32(np.inf)), b)
    _check_route(cfg, torch.from_numpy(u.astype(np.float32)), torch.from_numpy(b), name + " dense ties")
