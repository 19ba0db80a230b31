"""moe_permute_static_scratch: the permutation for callers that cannot allocate device memory.

Such callers (an allocator-free runtime, a plugin whose host framework owns every device
allocation, a process that must not grow its device footprint) cannot pass a workspace, so
this entry point keeps its scratch in a 2.5 MiB device array inside the library. Its outputs
must equal moe_permute's bit for bit (integer index work), call after call: the array keeps the
previous call's contents, so two different calls in a row are compared. The largest case is
the documented cap (65536 tokens, 256 experts), where every region of the array is in use; it
permutes indices only.
This file is collected last on purpose; it also passes when run on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from moe_inputs import CONFIGS, make_logits, make_router, make_x
from tests.helpers import MID_A, MID_V2


def _routing(cfg, T, seed):
    u = make_logits(cfg, seed=seed, T=T)
    sb = make_router(cfg)["select_bias"]
    u64 = u.double().numpy()
    s = oracle.scores(u64, cfg.score_fn)
    idx, w, _ = oracle.route(cfg.replace(T=T), s, None if sb is None else sb.double().numpy(),
                             u=u64)
    return torch.from_numpy(idx).cuda(), torch.from_numpy(w.astype(np.float32)).cuda()


def _outputs(cfg, T, with_x):
    A = T * cfg.top_k
    offs = torch.full((cfg.n_routed + 1,), -5, dtype=torch.int32, device="cuda")
    rt = torch.full((A,), -5, dtype=torch.int32, device="cuda")
    sr = torch.full((A,), -5, dtype=torch.int32, device="cuda")
    xp = torch.zeros((A, cfg.hidden), dtype=cfg.torch_dtype, device="cuda") if with_x else None
    return offs, rt, sr, xp


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", [MID_V2, MID_A, CONFIGS["v2"], CONFIGS["v3_prefill"],
                                 CONFIGS["v3_prefill"].replace(name="v3_t65536", T=65536)],
                         ids=lambda c: c.name)
def test_static_scratch_permute_matches_workspace_permute(cfg):
    import mixture_experts_routing_sigmoid_b300 as moe
    T = cfg.T
    with_x = T * cfg.hidden <= 2 ** 27
    ws = torch.empty(moe.moe_workspace_size(cfg, T), dtype=torch.uint8, device="cuda")
    for call, seed in enumerate((21, 22)):  # two different calls in a row
        idx, w = _routing(cfg, T, seed)
        x = make_x(cfg, device="cuda", seed=seed, T=T) if with_x else None
        ref = _outputs(cfg, T, with_x)
        moe.moe_permute(cfg, T, idx, w, x, *ref, ws)
        got = _outputs(cfg, T, with_x)
        moe.moe_permute_static_scratch(cfg, T, idx, w, x, *got)
        assert moe.moe_get_error() == 0
        R = int(ref[0][-1])
        assert torch.equal(got[0], ref[0]), f"offsets differ on call {call}"
        assert torch.equal(got[1][:R], ref[1][:R]), f"row_token differs on call {call}"
        assert torch.equal(got[2], ref[2]), f"slot_row differs on call {call}"
        if with_x:
            assert torch.equal(got[3][:R], ref[3][:R]), f"x_perm differs on call {call}"


def test_static_scratch_rejects_too_many_tokens():
    """Host-side check (no GPU work): more tokens than the static scratch holds is refused."""
    import mixture_experts_routing_sigmoid_b300 as moe
    c = moe.config_of(CONFIGS["v3_prefill"])
    st = moe.lib.moe_permute_static_scratch(ctypes.byref(c), 65537, 0x1000, 0x2000, None,
                                            0x3000, 0x4000, 0x5000, None, None)
    assert st == moe.MOE_ERR_UNSUPPORTED
    assert "65536" in moe.lib.moe_last_error_detail().decode()
