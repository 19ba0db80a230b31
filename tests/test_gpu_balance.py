"""Auxiliary-loss-free bias update on the GPU against the fp64 oracle.

The direction of every expert's step is an integer decision (its count against the batch
mean) and must match exactly; the new bias is one fp32 addition of values whose exact sum the
oracle's fp64 arithmetic holds, so the fp32 results must match bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import CONFIGS

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,seed", [("tiny", 0), ("v3_prefill", 1), ("v2", 2)])
def test_bias_update_matches_oracle(name, seed):
    import mixture_experts_routing_sigmoid_b300 as moe
    cfg = CONFIGS[name]
    N = cfg.n_routed
    rng = np.random.default_rng(seed)
    counts = rng.integers(0, 2 * cfg.top_k * 64, size=N).astype(np.int32)
    counts[: N // 4] = int(np.round(counts.mean()))      # some experts near the mean
    total = int(counts.sum())
    if total % N == 0:                                     # and, when possible, exactly at it
        counts[0] = total // N
    bias = (rng.normal(0.0, 0.1, N)).astype(np.float32)
    rate = np.float32(1e-3)
    want = oracle.bias_update(counts.astype(np.int64), float(rate),
                              bias.astype(np.float64)).astype(np.float32)
    b_dev = torch.from_numpy(bias.copy()).cuda()
    moe.moe_bias_update(cfg, torch.from_numpy(counts).cuda(), float(rate), b_dev)
    assert moe.moe_get_error() == 0
    got = b_dev.cpu().numpy()
    np.testing.assert_array_equal(np.sign(got - bias), np.sign(want - bias))
    np.testing.assert_array_equal(got, want)


def test_bias_update_from_layer_counts():
    """Counts written by moe_layer_forward drive the update (the training-time loop)."""
    import mixture_experts_routing_sigmoid_b300 as moe
    from moe_inputs import make_weights, make_x
    from tests.helpers import workspace
    cfg = CONFIGS["tiny"]
    w = make_weights(cfg, device="cuda")
    x = make_x(cfg, device="cuda", seed=4)
    out = torch.empty_like(x)
    counts = torch.empty(cfg.n_routed, dtype=torch.int32, device="cuda")
    lbz = torch.empty(3, dtype=torch.float32, device="cuda")
    moe.moe_layer_forward(cfg, cfg.T, x, w, out, counts, lbz, workspace(cfg, cfg.T))
    b_dev = w["select_bias"].clone()
    moe.moe_bias_update(cfg, counts, 0.01, b_dev)
    assert moe.moe_get_error() == 0
    c = counts.cpu().numpy().astype(np.int64)
    assert c.sum() == cfg.T * cfg.top_k
    want = oracle.bias_update(c, float(np.float32(0.01)),
                              w["select_bias"].double().cpu().numpy()).astype(np.float32)
    np.testing.assert_array_equal(b_dev.cpu().numpy(), want)


@pytest.mark.parametrize("name,seq_len", [("tiny", 16), ("tiny", 64), ("v1", 512), ("v3_prefill", 4096),
                                          ("v3_prefill", 1)])
def test_seq_balance_loss_matches_oracle(name, seq_len):
    """Sequence-wise balance loss on identical logits and routing: per-sequence values and their
    mean within 1e-5 relative (fp32 score sums over at most a few thousand tokens)."""
    import mixture_experts_routing_sigmoid_b300 as moe
    from moe_inputs import make_logits, make_router
    from tests.helpers import gpu_route, workspace
    cfg = CONFIGS[name]
    T = cfg.T if seq_len > 1 else 256
    u = make_logits(cfg, seed=11, T=T)
    sb = make_router(cfg)["select_bias"]
    w = {"select_bias": None if sb is None else sb.cuda()}
    idx, _, _ = gpu_route(cfg, T, logits=u.cuda(), weights=w)
    B = T // seq_len
    per = torch.empty(B, dtype=torch.float32, device="cuda")
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    moe.moe_seq_balance_loss(cfg, T, seq_len, u.cuda(), idx, per, loss, workspace(cfg, T))
    assert moe.moe_get_error() == 0
    ud = u.double().numpy()
    want_per, want_mean = oracle.seq_balance_loss(cfg, ud, oracle.scores(ud, cfg.score_fn),
                                                  idx.cpu().numpy(), seq_len)
    np.testing.assert_allclose(per.cpu().numpy(), want_per, rtol=1e-5)
    assert abs(float(loss.item()) - want_mean) <= 1e-5 * abs(want_mean)


def test_seq_balance_loss_rejects_bad_seq_len():
    import mixture_experts_routing_sigmoid_b300 as moe
    from tests.helpers import workspace
    cfg = CONFIGS["tiny"]
    u = torch.zeros((cfg.T, cfg.n_routed), device="cuda")
    idx = torch.zeros((cfg.T, cfg.top_k), dtype=torch.int32, device="cuda")
    loss = torch.empty(1, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_seq_balance_loss(cfg, cfg.T, 7, u, idx, None, loss, workspace(cfg, cfg.T))
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["tiny", "v2", "v3_prefill", "v3_decode_512"])
def test_group_balance_losses_match_oracle(name):
    """Device-level and communication losses on identical logits and routing: within 1e-5
    relative of the fp64 oracle (fp32 score sums)."""
    import mixture_experts_routing_sigmoid_b300 as moe
    from moe_inputs import make_logits, make_router
    from tests.helpers import gpu_route, workspace
    cfg = CONFIGS[name]
    T = cfg.T
    u = make_logits(cfg, seed=13, T=T)
    sb = make_router(cfg)["select_bias"]
    idx, _, _ = gpu_route(cfg, T, logits=u.cuda(),
                          weights={"select_bias": None if sb is None else sb.cuda()})
    out = torch.empty(2, dtype=torch.float32, device="cuda")
    moe.moe_group_balance_losses(cfg, T, u.cuda(), idx, out, workspace(cfg, T))
    assert moe.moe_get_error() == 0
    ud = u.double().numpy()
    want = oracle.group_balance_losses(cfg, ud, oracle.scores(ud, cfg.score_fn),
                                       idx.cpu().numpy())
    np.testing.assert_allclose(out.cpu().numpy(), want, rtol=1e-5)
