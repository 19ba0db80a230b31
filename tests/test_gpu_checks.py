"""The bounds-checked build (libmoe_b300_checked.so, loaded when MOE_B300_CHECKED=1).

Its kernels check the indices they follow: segment offsets (expert GEMMs), slot rows (row
dispatch, combine) and gathered token rows. An index outside its logical range is reported as
MOE_ERR_DEVICE_CHECK through moe_get_error and the access is skipped ("从零构建DeepSeekMoE",
section 7 lists fault handling among the deployment concerns). Every bad index fed here still
lies inside the buffers the test allocates, so the default build, which has no checks, reads and
writes only memory it owns and reports nothing. Each case runs in a child process (the build is
chosen when the package is imported).
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import json, sys
import numpy as np, torch
sys.path.insert(0, ROOT)
import mixture_experts_routing_sigmoid_b300 as moe
from moe_inputs import make_weights, make_x
from tests.helpers import MID_A, workspace
cfg = MID_A
T, H, K, I, S, N = cfg.T, cfg.hidden, cfg.top_k, cfg.inter, cfg.n_shared, cfg.n_routed
res = {"lib": moe.LIB_PATH}
w = make_weights(cfg, device="cuda"); x = make_x(cfg, device="cuda", seed=2)
ws = workspace(cfg, T)
# a valid routing and permutation first
idx = torch.empty((T, K), dtype=torch.int32, device="cuda"); wt = torch.empty((T, K), device="cuda")
moe.moe_route(cfg, T, x, w, None, None, idx, wt, ws)
offs = torch.empty(N + 1, dtype=torch.int32, device="cuda")
rt = torch.empty(T * K, dtype=torch.int32, device="cuda"); sr = torch.empty(T * K, dtype=torch.int32, device="cuda")
xp = torch.zeros((T * K, H), dtype=x.dtype, device="cuda")
moe.moe_permute(cfg, T, idx, wt, x, offs, rt, sr, xp, ws)
res["valid"] = moe.moe_get_error()
EXTRA = 64  # spare rows behind every buffer a bad index can reach
# 1. combine with slot rows past the T*K rows of y (inside y's allocation)
y = torch.randn((T * K + EXTRA, H), device="cuda").to(x.dtype)
bad = sr.clone(); bad[5] = T * K + 3; bad[17] = T * K + EXTRA - 1
out = torch.empty_like(x)
moe.moe_combine(cfg, T, y, bad, wt, None, out)
res["combine"] = moe.moe_get_error()
# 2. expert GEMMs with a segment ending past the T*K rows (inside the allocations)
bad_offs = offs.clone(); bad_offs[N] = T * K + 8
big_xp = torch.zeros((T * K + EXTRA, H), dtype=x.dtype, device="cuda")
y2 = torch.zeros((T * K + EXTRA, H), dtype=x.dtype, device="cuda")
ys = torch.zeros((T, H), dtype=x.dtype, device="cuda")
moe.moe_expert_ffn(cfg, T, big_xp, bad_offs, x, w, y2, ys, ws)
res["ffn"] = moe.moe_get_error()
# 3. row dispatch (moe_permute) is checked through slot rows the permutation itself writes, so
#    it cannot be fed a bad one; the gathered rows of the up projection are: a token index past T
bad_rt = rt.clone(); bad_rt[0] = T + 5
h = torch.zeros((T * K + EXTRA, I), dtype=x.dtype, device="cuda")
hs = torch.zeros((T, S * I), dtype=x.dtype, device="cuda")
moe.moe_expert_up_gather(cfg, T, x, bad_rt, offs, w, h, hs)
res["gather"] = moe.moe_get_error()
# 4. valid inputs again: no report, and the same layer output as the other build
out2 = torch.empty_like(x)
moe.moe_layer_forward(cfg, T, x, w, out2, None, None, ws)
res["layer"] = moe.moe_get_error()
res["layer_sum"] = float(out2.double().abs().sum())
print(json.dumps(res))
'''


def _child(checked: bool) -> dict:
    env = dict(os.environ)
    env["MOE_B300_CHECKED"] = "1" if checked else "0"
    r = subprocess.run([sys.executable, "-c", CHILD.replace("ROOT", repr(ROOT))], env=env,
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_checked_build_reports_out_of_range_indices():
    import mixture_experts_routing_sigmoid_b300 as moe
    got = _child(True)
    assert got["lib"].endswith("libmoe_b300_checked.so")
    assert got["valid"] == moe.MOE_OK
    assert got["combine"] == moe.MOE_ERR_DEVICE_CHECK
    assert got["ffn"] == moe.MOE_ERR_DEVICE_CHECK
    assert got["gather"] == moe.MOE_ERR_DEVICE_CHECK
    assert got["layer"] == moe.MOE_OK
    plain = _child(False)
    assert plain["lib"].endswith("libmoe_b300.so")
    # the default build checks nothing (and stays in bounds: every bad index is inside a buffer)
    assert plain["valid"] == plain["combine"] == plain["ffn"] == plain["gather"] == moe.MOE_OK
    assert plain["layer"] == moe.MOE_OK
    # on valid inputs both builds compute the same layer
    assert got["layer_sum"] == plain["layer_sum"]
