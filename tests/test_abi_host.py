"""C-ABI library: loads, exports every declared entry point, rejects bad arguments on the host
before anything reaches a GPU (CPU only: no compute call is made)."""
import ctypes
import os
import re

import pytest

from moe_inputs import CONFIGS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import mixture_experts_routing_sigmoid_b300 as m
    return m


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("moe_route", "moe_load_stats", "moe_permute", "moe_expert_ffn", "moe_combine",
              "moe_layer_forward", "moe_workspace_size", "moe_get_error"):
        assert n in names


def test_every_declared_symbol_is_exported(moe):
    raw = ctypes.CDLL(moe.LIB_PATH)
    for n in _declared_functions():
        assert hasattr(raw, n), n
    assert set(moe.EXPORTED_SYMBOLS) <= set(_declared_functions())


def test_workspace_size(moe):
    for name, cfg in CONFIGS.items():
        n = moe.moe_workspace_size(cfg, cfg.T)
        assert n > 0 and n % 256 == 0, name
        assert moe.moe_workspace_size(cfg, 2 * cfg.T) > n
    # x_perm / y_perm share one region: the v3 prefill workspace stays under 5 GB
    assert moe.moe_workspace_size(CONFIGS["v3_prefill"], 16384) < 5 * 2 ** 30


@pytest.mark.parametrize("bad,status", [
    (dict(n_groups=3), -1),             # does not divide n_routed
    (dict(topk_groups=9), -1),          # more than n_groups
    (dict(top_k=200), -1),              # more than the kept groups hold
    (dict(routed_scale=0.0), -1),
    (dict(group_score_topn=3), -2),     # valid for the method, not for the kernels
    (dict(n_routed=512, n_groups=8), -2),
    (dict(inter=100), -2),              # bf16 path wants inter % 128 == 0
])
def test_invalid_config_rejected_on_host(moe, bad, status):
    cfg = CONFIGS["v3_prefill"].replace(**bad)
    c = moe.config_of(cfg)
    assert moe.lib.moe_workspace_size(ctypes.byref(c), 16) == 0
    st = moe.lib.moe_layer_forward(ctypes.byref(c), 16, None, None, None, None, None, None, 0,
                                   None)
    assert st == status
    assert moe.lib.moe_last_error_detail().decode()


def test_null_and_misaligned_pointers_rejected(moe):
    cfg = CONFIGS["v3_prefill"]
    c = moe.config_of(cfg)
    w = moe.MoeWeights()
    st = moe.lib.moe_layer_forward(ctypes.byref(c), 16, None, ctypes.byref(w), None, None, None,
                                   None, 0, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    st = moe.lib.moe_combine(ctypes.byref(c), 4, 0x1001, 0x2000, 0x3000, None, 0x4000, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    assert "aligned" in moe.lib.moe_last_error_detail().decode()
    st = moe.lib.moe_selftest_wait_timeout(0, None)
    assert st == moe.MOE_ERR_INVALID_ARG


def test_workspace_too_small_rejected(moe):
    cfg = CONFIGS["tiny"]
    c = moe.config_of(cfg)
    st = moe.lib.moe_permute(ctypes.byref(c), 8, 0x1000, 0x2000, None, 0x3000, 0x4000, None,
                             0x5000, None, 0x6000, 64, None)
    assert st == moe.MOE_ERR_WORKSPACE


def test_status_strings(moe):
    for s in range(-6, 1):
        assert moe.moe_status_string(s) != "unknown status"


def test_zero_tokens_is_a_no_op(moe):
    cfg = CONFIGS["v3_prefill"]
    c = moe.config_of(cfg)
    w = moe.MoeWeights()
    assert moe.lib.moe_layer_forward(ctypes.byref(c), 0, None, ctypes.byref(w), None, None, None,
                                     None, 0, None) == 0


def test_permute_row_w_alignment_checked(moe):
    cfg = CONFIGS["tiny"]
    c = moe.config_of(cfg)
    st = moe.lib.moe_permute(ctypes.byref(c), 8, 0x1000, 0x2000, None, 0x3000, 0x4000, 0x4004,
                             0x5000, None, 0x6000, 1 << 30, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    assert "row_w" in moe.lib.moe_last_error_detail().decode()
