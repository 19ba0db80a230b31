"""Routed + shared SwiGLU experts and the weighted combine on the GPU against the fp64 oracle.

Inputs (x, weights, the permutation) come from the seeded generators and the oracle, never
from the CUDA path. Expert rows are compared by relative Frobenius error: 1e-2 for bf16
(tensor cores, h rounded to bf16 between the GEMMs), 1e-5 for fp32.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import CONFIGS, make_logits, make_router, make_weights, make_x
from tests.helpers import (MID_A, MID_B, MID_ODD, MID_V2, gemm_tail_split, gemm_tiles, rel_frob,
                           sample_tokens, tol_for, workspace)

pytestmark = pytest.mark.gpu

CFGS = {**CONFIGS, "mid_a": MID_A, "mid_b": MID_B, "mid_v2": MID_V2, "mid_odd": MID_ODD,
        # batches of at most 64 and 128 tokens: tiles of few token rows, whose smaller ring
        # stages run deeper
        "mid_a_t50": MID_A.replace(name="mid_a_t50", T=50),
        "mid_odd_t100": MID_ODD.replace(name="mid_odd_t100", T=100)}


def _perm_inputs(cfg, seed=3):
    T = cfg.T
    u = make_logits(cfg, seed=seed, T=T)
    sb = make_router(cfg)["select_bias"]
    u64 = u.double().numpy()
    s = oracle.scores(u64, cfg.score_fn)
    idx, w, _ = oracle.route(cfg, s, None if sb is None else sb.double().numpy(), u=u64)
    kept = oracle.capacity_drop(cfg, idx, w) if cfg.capacity_drop else None
    offs, row_token, slot_row = oracle.permute(cfg, idx, kept)
    return idx, w, offs, row_token, slot_row


def _expert_of_rows(offs):
    return np.repeat(np.arange(len(offs) - 1), np.diff(offs))


@pytest.mark.parametrize("name", ["tiny", "mid_a", "mid_b", "mid_v2", "mid_odd", "mid_a_t50",
                                  "mid_odd_t100", "v1", "v2", "v3_prefill", "v3_decode_32",
                                  "v3_decode_128", "v3_decode_512"])
def test_expert_ffn(name):
    import mixture_experts_routing_sigmoid_b300 as moe
    cfg = CFGS[name]
    T, H, K = cfg.T, cfg.hidden, cfg.top_k
    # oracle cost of every routed row: 3 H I multiply-adds each
    big = T * K * 3 * H * cfg.inter > 4e9
    dev = "cuda"
    w = make_weights(cfg, device=dev)
    x = make_x(cfg, device=dev, seed=2)
    idx, wt, offs, row_token, slot_row = _perm_inputs(cfg)
    R = int(offs[-1])
    x_perm = torch.zeros((T * K, H), dtype=x.dtype, device=dev)
    x_perm[:R] = x[torch.from_numpy(row_token).long().to(dev)]
    y = torch.full((T * K, H), float("nan"), dtype=x.dtype, device=dev)
    ys = torch.full((T, H), float("nan"), dtype=x.dtype, device=dev) if cfg.n_shared else None
    ws = workspace(cfg, T)
    moe.moe_expert_ffn(cfg, T, x_perm, torch.from_numpy(offs).to(dev), x, w, y, ys, ws)
    assert moe.moe_get_error() == 0

    # routed rows: all of them on small layers, a sample spread over experts on big ones
    exp_of = _expert_of_rows(offs)
    rows = np.arange(R) if not big else np.unique(np.concatenate(
        [offs[:-1][np.diff(offs) > 0],                       # first row of every segment
         offs[1:][np.diff(offs) > 0] - 1,                    # last row (ragged tails)
         np.random.default_rng(0).choice(R, 64, replace=False)]))
    if big:
        # keep the oracle cost bounded: at most 48 distinct experts
        ex = np.unique(exp_of[rows])[:48]
        rows = rows[np.isin(exp_of[rows], ex)]
    got = y[torch.from_numpy(rows).long().to(dev)].double().cpu().numpy()
    want = np.zeros_like(got)
    xr = x_perm[torch.from_numpy(rows).long().to(dev)].double().cpu().numpy()
    for e in np.unique(exp_of[rows]):
        sel = exp_of[rows] == e
        w13, w2 = (w["w13"][e], w["w2"][e]) if cfg.dtype == "bf16" else \
            (w["w13"][e].double().cpu().numpy(), w["w2"][e].double().cpu().numpy())
        want[sel] = oracle.swiglu_rows(xr[sel], w13, w2)
    err = rel_frob(got, want)
    assert err <= tol_for(cfg), f"routed rows: rel err {err:.3g}"

    if cfg.n_shared:
        tok = sample_tokens(T, 32 if big else T, seed=1)
        xs = x[torch.from_numpy(tok).long().to(dev)].double().cpu().numpy()
        want_s = np.zeros((len(tok), H))
        for s_ in range(cfg.n_shared):
            w13, w2 = (w["w13_shared"][s_], w["w2_shared"][s_]) if cfg.dtype == "bf16" else \
                (w["w13_shared"][s_].double().cpu().numpy(), w["w2_shared"][s_].double().cpu().numpy())
            want_s += oracle.swiglu_rows(xs, w13, w2)
        got_s = ys[torch.from_numpy(tok).long().to(dev)].double().cpu().numpy()
        err = rel_frob(got_s, want_s)
        assert err <= tol_for(cfg), f"shared rows: rel err {err:.3g}"


@pytest.mark.parametrize("name", ["tiny", "mid_b", "mid_v2", "v3_prefill"])
def test_combine(name):
    import mixture_experts_routing_sigmoid_b300 as moe
    cfg = CFGS[name]
    T, H, K = cfg.T, cfg.hidden, cfg.top_k
    idx, wt, offs, row_token, slot_row = _perm_inputs(cfg)
    R = int(offs[-1])
    g = torch.Generator(device="cuda").manual_seed(5)
    y = torch.randn((max(R, 1), H), generator=g, device="cuda").to(cfg.torch_dtype)
    ys = torch.randn((T, H), generator=g, device="cuda").to(cfg.torch_dtype)
    w32 = wt.astype(np.float32)
    out = torch.empty((T, H), dtype=cfg.torch_dtype, device="cuda")
    moe.moe_combine(cfg, T, y, torch.from_numpy(slot_row).cuda(), torch.from_numpy(w32).cuda(),
                    ys, out)
    assert moe.moe_get_error() == 0
    tok = sample_tokens(T, 256, seed=2)
    # only the rows the sampled tokens reference, renumbered
    sr = slot_row[tok]
    used = np.unique(sr[sr >= 0])
    remap = -np.ones(max(R, 1), np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    sr_sub = np.where(sr >= 0, remap[np.maximum(sr, 0)], -1).astype(np.int32)
    y_sub = y[torch.from_numpy(used).long().cuda()].double().cpu().numpy()
    want = oracle.combine(y_sub, sr_sub, w32[tok].astype(np.float64),
                          ys[torch.from_numpy(tok).long().cuda()].double().cpu().numpy())
    got = out[torch.from_numpy(tok).long().cuda()].double().cpu().numpy()
    assert rel_frob(got, want) <= (1e-2 if cfg.dtype == "bf16" else 1e-6)
    if cfg.dtype == "bf16":
        # output is the bf16 rounding of an fp32 sum: elementwise within 2^-8 relative + slack
        assert np.all(np.abs(got - want) <= 2 ** -8 * np.abs(want) + 1e-2)


@pytest.mark.parametrize("name", ["mid_a", "mid_a_t50", "mid_odd_t100", "v3_prefill_e32",
                                  "v3_decode_32"])
def test_tile_schedule_does_not_change_results(name):
    """moe_expert_ffn (workspace given: tiles claimed dynamically from a counter, the tail wave's
    tiles cut along K into pieces) and moe_expert_up + moe_expert_down (no workspace: static
    round-robin tiles, nothing cut) compute every uncut tile with the same k order, so those
    outputs are bitwise equal. A cut tile's pieces are added in piece order in fp32: its outputs
    (and, for a cut up-projection tile, the rows of y it feeds) agree within a bf16 rounding,
    and two runs are bitwise equal whichever piece finishes last."""
    import mixture_experts_routing_sigmoid_b300 as moe
    cfg = CFGS[name]
    T, H, K, I, S = cfg.T, cfg.hidden, cfg.top_k, cfg.inter, cfg.n_shared
    dev = "cuda"
    w = make_weights(cfg, device=dev)
    x = make_x(cfg, device=dev, seed=2)
    idx, wt, offs, row_token, slot_row = _perm_inputs(cfg)
    R = int(offs[-1])
    x_perm = torch.zeros((T * K, H), dtype=x.dtype, device=dev)
    x_perm[:R] = x[torch.from_numpy(row_token).long().to(dev)]
    offs_d = torch.from_numpy(offs).to(dev)
    runs = []
    for _ in range(2):
        y_dyn = torch.zeros((T * K, H), dtype=x.dtype, device=dev)
        ys_dyn = torch.zeros((T, H), dtype=x.dtype, device=dev)
        moe.moe_expert_ffn(cfg, T, x_perm, offs_d, x, w, y_dyn, ys_dyn, workspace(cfg, T))
        runs.append((y_dyn, ys_dyn))
    h = torch.zeros((T * K, I), dtype=x.dtype, device=dev)
    h_sh = torch.zeros((T, S * I), dtype=x.dtype, device=dev)
    y_st = torch.zeros_like(runs[0][0])
    ys_st = torch.zeros_like(runs[0][1])
    moe.moe_expert_up(cfg, T, x_perm, offs_d, x, w, h, h_sh)
    moe.moe_expert_down(cfg, T, h, offs_d, h_sh, w, y_st, ys_st)
    torch.cuda.synchronize()
    assert moe.moe_get_error() == 0
    (y_dyn, ys_dyn), (y_dyn2, ys_dyn2) = runs
    assert torch.equal(y_dyn[:R], y_dyn2[:R]) and torch.equal(ys_dyn, ys_dyn2)
    # outputs that a cut tile computes or feeds
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    cut_y = np.zeros((R, H), bool)
    cut_ys = np.zeros((T, H), bool)
    n_cut = 0
    for mode in ("up", "down"):
        _, n_tail, pieces = gemm_tail_split(cfg, offs, mode, pairs)
        if pieces < 2:
            continue
        n_cut += n_tail
        for q, f0, f1, r0, r1 in gemm_tiles(cfg, offs, mode)[-n_tail:]:
            cols = slice(None) if mode == "up" else slice(f0, f1)
            if q == cfg.n_routed:
                cut_ys[r0:r1, cols] = True
            else:
                cut_y[offs[q] + r0:offs[q] + r1, cols] = True
    if name in ("v3_prefill_e32", "v3_decode_32"):
        assert n_cut > 0, "this batch must exercise the tail split"
    for got, want, cut in ((y_dyn[:R], y_st[:R], cut_y), (ys_dyn, ys_st, cut_ys)):
        g = got.float().cpu().numpy()
        e = want.float().cpu().numpy()
        np.testing.assert_array_equal(g[~cut], e[~cut])
        if cut.any():
            assert np.all(np.abs(g[cut] - e[cut]) <= 2 ** -6 * np.abs(e[cut])
                          + 1e-3 * np.abs(e).max())
            assert rel_frob(g[cut], e[cut]) <= 1e-3


@pytest.mark.parametrize("name", ["mid_a", "mid_odd", "mid_v2", "mid_a_t50", "mid_odd_t100",
                                  "v3_decode_32", "v3_decode_512", "v3_prefill_e32", "v1"])
def test_row_gather_equals_permuted_copy(name):
    """The up projection reading its routed rows from x through row_token (tile::gather4 loads,
    what moe_layer_forward runs) gives bitwise the outputs of the same GEMM on the permuted copy
    x_perm = x[row_token]: the gather changes where the token rows come from, not the
    arithmetic. Segments of every length occur (ragged tails, segments shorter than one row
    group of four, empty experts)."""
    import mixture_experts_routing_sigmoid_b300 as moe
    cfg = CFGS[name]
    T, H, K, I, S = cfg.T, cfg.hidden, cfg.top_k, cfg.inter, cfg.n_shared
    dev = "cuda"
    w = make_weights(cfg, device=dev)
    x = make_x(cfg, device=dev, seed=2)
    idx, wt, offs, row_token, slot_row = _perm_inputs(cfg)
    R = int(offs[-1])
    rt = torch.full((T * K,), -3, dtype=torch.int32, device=dev)  # rows past R: not read
    rt[:R] = torch.from_numpy(row_token).to(dev)
    x_perm = torch.zeros((T * K, H), dtype=x.dtype, device=dev)
    x_perm[:R] = x[rt[:R].long()]
    offs_d = torch.from_numpy(offs).to(dev)
    h_ref = torch.zeros((T * K, I), dtype=x.dtype, device=dev)
    hs_ref = torch.zeros((T, max(S, 1) * I), dtype=x.dtype, device=dev) if S else None
    moe.moe_expert_up(cfg, T, x_perm, offs_d, x, w, h_ref, hs_ref)
    h = torch.full_like(h_ref, float("nan"))
    hs = torch.full_like(hs_ref, float("nan")) if S else None
    moe.moe_expert_up_gather(cfg, T, x, rt, offs_d, w, h, hs)
    torch.cuda.synchronize()
    assert moe.moe_get_error() == 0
    assert torch.equal(h[:R], h_ref[:R])
    if S:
        assert torch.equal(hs, hs_ref)
