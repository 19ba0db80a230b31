"""Runtime behaviour of the layer forward on the GPU: it can be captured into a CUDA graph and
replayed with identical results, its stage timing covers each call, the launch counter counts
what runs, and repeated calls are deterministic."""
import pytest
import torch

from moe_inputs import CONFIGS, make_weights, make_x
from tests.helpers import MID_A, workspace

pytestmark = pytest.mark.gpu


def _layer(cfg, seed=2):
    w = make_weights(cfg, device="cuda")
    x = make_x(cfg, device="cuda", seed=seed)
    return w, x, torch.empty_like(x), workspace(cfg, cfg.T)


@pytest.mark.parametrize("cfg", [MID_A, CONFIGS["tiny"], CONFIGS["v3_decode_32"]],
                         ids=lambda c: c.name)
def test_graph_replay_matches_eager(cfg):
    import mixture_experts_routing_sigmoid_b300 as moe
    w, x, out, ws = _layer(cfg)
    moe.moe_layer_forward(cfg, cfg.T, x, w, out, None, None, ws)
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        moe.moe_layer_forward(cfg, cfg.T, x, w, out, None, None, ws,
                              torch.cuda.current_stream())
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert moe.moe_get_error() == 0
    assert torch.equal(out, eager)


def test_repeated_calls_are_bitwise_deterministic():
    import mixture_experts_routing_sigmoid_b300 as moe
    cfg = MID_A
    w, x, out, ws = _layer(cfg, seed=3)
    moe.moe_layer_forward(cfg, cfg.T, x, w, out, None, None, ws)
    first = out.clone()
    for _ in range(3):
        moe.moe_layer_forward(cfg, cfg.T, x, w, out, None, None, ws)
        assert torch.equal(out, first)


def test_stage_timing_and_launch_count():
    import mixture_experts_routing_sigmoid_b300 as moe
    cfg = CONFIGS["tiny"]   # fp32: gate, route, permutation (one block), dispatch, up, down, combine
    w, x, out, ws = _layer(cfg)
    moe.moe_layer_forward(cfg, cfg.T, x, w, out, None, None, ws)
    torch.cuda.synchronize()
    n0 = moe.moe_kernel_launches()
    moe.moe_stage_timing_start(3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(3):
        moe.moe_layer_forward(cfg, cfg.T, x, w, out, None, None, ws)
    e1.record()
    torch.cuda.synchronize()
    stages, calls = moe.moe_stage_timing_stop()
    assert calls == 3
    assert moe.moe_kernel_launches() - n0 == 3 * 7
    assert set(stages) == set(moe.STAGE_NAMES)
    assert all(v >= 0.0 for v in stages.values())
    assert stages["stats"] < 0.05 * sum(stages.values())       # not requested: empty stage
    assert sum(stages.values()) <= e0.elapsed_time(e1) * 1.05 + 0.05
    with pytest.raises(moe.MoeError):
        moe.moe_stage_timing_stop()                            # not active any more
