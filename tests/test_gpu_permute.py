"""Permutation by expert and the v2 device-level drop on the GPU, bit-exact against the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from moe_inputs import CONFIGS, make_logits, make_router, make_x
from tests.helpers import MID_A, MID_B, MID_V2, gpu_permute, gpu_route

pytestmark = pytest.mark.gpu

CFGS = {**CONFIGS, "mid_a": MID_A, "mid_b": MID_B, "mid_v2": MID_V2}


def _oracle_routing(cfg, T, seed=3):
    u = make_logits(cfg, seed=seed, T=T)
    sb = make_router(cfg)["select_bias"]
    u64 = u.double().numpy()
    s = oracle.scores(u64, cfg.score_fn)
    idx, w, _ = oracle.route(cfg, s, None if sb is None else sb.double().numpy(), u=u64)
    return idx, w


def _check(cfg, T, idx, w, with_x=True):
    w32 = w.astype(np.float32)
    kept = oracle.capacity_drop(cfg.replace(T=T), idx, w32.astype(np.float64)) \
        if cfg.capacity_drop else None
    offs_o, rt_o, sr_o = oracle.permute(cfg.replace(T=T), idx, kept)
    x = make_x(cfg, device="cuda", seed=9, T=T) if with_x else None
    row_w = torch.full((max(T * cfg.top_k, 1),), float("nan"), device="cuda")
    offs, rt, sr, xp = gpu_permute(cfg, T, torch.from_numpy(idx).cuda(),
                                   torch.from_numpy(w32).cuda(), x=x, row_w=row_w)
    np.testing.assert_array_equal(offs.cpu().numpy(), offs_o)
    R = int(offs_o[-1])
    np.testing.assert_array_equal(rt.cpu().numpy()[:R], rt_o)
    np.testing.assert_array_equal(sr.cpu().numpy()[:T * cfg.top_k], sr_o.ravel())
    if with_x and R:
        assert torch.equal(xp[:R], x[torch.from_numpy(rt_o).long().cuda()])
    # row_w[r] is the routing weight of the assignment placed at row r
    sr_flat = sr_o.ravel()
    want = np.full(R, np.nan, dtype=np.float32)
    want[sr_flat[sr_flat >= 0]] = w32.ravel()[sr_flat >= 0]
    np.testing.assert_array_equal(row_w.cpu().numpy()[:R], want)
    return offs_o, kept


@pytest.mark.parametrize("name", ["tiny", "v1", "v2", "v3_prefill", "v3_decode_32",
                                  "v3_decode_512", "mid_a", "mid_b", "mid_v2"])
def test_permute_bit_exact(name):
    cfg = CFGS[name]
    idx, w = _oracle_routing(cfg, cfg.T)
    offs, kept = _check(cfg, cfg.T, idx, w, with_x=cfg.T * cfg.hidden <= 2 ** 27)
    if cfg.capacity_drop:
        C = math.ceil(cfg.T * cfg.top_k / cfg.n_groups)
        loads = np.bincount(idx.ravel() // (cfg.n_routed // cfg.n_groups), minlength=cfg.n_groups)
        assert loads.max() > C, "the skewed v2 workload must exercise the drop"


def test_drop_ties_and_uniform_load():
    cfg = MID_V2
    T, K = cfg.T, cfg.top_k
    per = cfg.n_routed // cfg.n_groups
    # all assignments on device 0 with equal weights: keeps the first C in (token, slot) order
    idx = np.tile(np.arange(K, dtype=np.int32), (T, 1))
    w = np.full((T, K), 0.125)
    _check(cfg, T, idx, w)
    # balanced load: nothing dropped
    idx = np.array([[((t + j) % 8) * per + (t // 8 + i) % per for j in range(3) for i in range(2)]
                    for t in range(T)], np.int32)
    w = np.random.default_rng(0).random((T, K))
    _, kept = _check(cfg, T, idx, w)
    assert kept.all()


def test_permute_one_hot_expert_and_empty_experts():
    """Every token routed to expert 3 (a segment of T rows over several 128-row tiles);
    most experts get no rows at all."""
    cfg = MID_B
    T, K = cfg.T, cfg.top_k
    idx = np.tile(np.array([3, 5, 8, 13, 21, 30], np.int32), (T, 1))
    w = np.full((T, K), 0.1)
    offs, _ = _check(cfg, T, idx, w)
    assert offs[4] - offs[3] == T


def test_permute_end_to_end_from_gpu_route():
    """GPU route -> GPU permute equals oracle route -> drop -> permute on identical logits."""
    cfg = CONFIGS["v2"]
    T = cfg.T
    u = make_logits(cfg, seed=8)
    idx_g, w_g, _ = gpu_route(cfg, T, logits=u.cuda(), weights={})
    offs, rt, sr, _ = gpu_permute(cfg, T, idx_g, w_g)
    s = oracle.scores(u.double().numpy(), "softmax")
    idx_o, w_o, _ = oracle.route(cfg, s, u=u.double().numpy())
    kept = oracle.capacity_drop(cfg, idx_o, w_o)
    offs_o, rt_o, sr_o = oracle.permute(cfg, idx_o, kept)
    np.testing.assert_array_equal(offs.cpu().numpy(), offs_o)
    np.testing.assert_array_equal(sr.cpu().numpy(), sr_o.ravel())
    np.testing.assert_array_equal(rt.cpu().numpy()[:offs_o[-1]], rt_o)


@pytest.mark.parametrize("T", [1, 255, 257, 1023, 1024, 1025])
def test_permute_single_block_boundaries(T):
    """One CTA takes batches of up to 1024 tokens, more go through the three-kernel path: both
    sides of the boundary are bit-exact."""
    cfg = MID_A.replace(T=T)
    idx, w = _oracle_routing(cfg, T)
    _check(cfg, T, idx, w, with_x=True)


@pytest.mark.parametrize("per_dev0", [2, 4])
def test_drop_device_with_more_keys_than_shared_memory(per_dev0):
    """The drop's radix select keeps up to 20480 keys of a device in shared memory and streams
    them from global memory beyond that: a v2-sized batch (T = 8192, K = 6) putting 2 of each
    token's 6 slots on device 0 (16384 keys: shared memory) or 4 (32768 keys: streamed), with
    random weights and ties, drops bit-exactly as the oracle does."""
    cfg = CONFIGS["v2"]
    T, K, N, G = cfg.T, cfg.top_k, cfg.n_routed, cfg.n_groups
    per = N // G
    rng = np.random.default_rng(per_dev0)
    idx = np.empty((T, K), np.int32)
    for t in range(T):
        dev0 = rng.choice(per, size=per_dev0, replace=False)
        rest = rng.choice(np.arange(per, N), size=K - per_dev0, replace=False)
        idx[t] = np.sort(np.concatenate([dev0, rest]))
    w = np.round(rng.random((T, K)) * 64) / 64  # many exact ties
    _check(cfg, T, idx, w, with_x=False)
