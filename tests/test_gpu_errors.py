"""Failure handling on the GPU without faulting it: a bounded wait that runs out reports
MOE_ERR_TIMEOUT through the error word and leaves the context usable; bad arguments with real
device buffers are refused on the host."""
import numpy as np
import pytest
import torch

from moe_inputs import CONFIGS, make_logits
from tests.helpers import gpu_route, workspace

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    import mixture_experts_routing_sigmoid_b300 as moe
    assert moe.moe_get_error() == 0
    moe.moe_selftest_wait_timeout(20000)          # 20 ms wait on a barrier nobody arrives on
    assert moe.moe_get_error() == moe.MOE_ERR_TIMEOUT
    assert moe.moe_get_error() == 0               # read clears it
    cfg = CONFIGS["tiny"]
    idx, w, _ = gpu_route(cfg, cfg.T, logits=make_logits(cfg).cuda(), weights={})
    assert idx.shape == (cfg.T, cfg.top_k) and torch.isfinite(w).all()


def test_workspace_too_small_with_device_buffers():
    import mixture_experts_routing_sigmoid_b300 as moe
    cfg = CONFIGS["v3_decode_32"]
    T = cfg.T
    ws = workspace(cfg, T)[:1024]
    x = torch.zeros((T, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    w = {k: torch.zeros(16, device="cuda") for k in ("w_gate", "w13", "w2", "w13_shared",
                                                        "w2_shared")}
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward(cfg, T, x, w, out, None, None, ws)
    assert ei.value.status == moe.MOE_ERR_WORKSPACE
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward(cfg, T, x[:, 1:], w, out, None, None, workspace(cfg, T))
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG   # misaligned rows pointer
    assert moe.moe_get_error() == 0
