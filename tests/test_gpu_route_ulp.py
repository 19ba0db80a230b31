"""Routing decisions one or two fp64 units apart, on the GPU against the fp64 oracle.

The routing kernel evaluates keys (sigmoid(u) + b, "DeepSeek MoE：从v1到v3的演进", DeepSeek-v3)
in fp32 and settles a token whose decision margin lies within the fp32 error bound by rescoring
the experts (or groups) inside that bound in fp64, with the same operations as the oracle:
1 / (1 + exp(-u)) + b. The chosen set then matches the oracle's bit for bit only if the GPU's
fp64 exp and the host's agree on those arguments. These tests put the K-th and (K+1)-th keys
(and, separately, the topk_groups-th and next group scores) 0, 1 or 2 fp64 units apart
(tests/golden/sigmoid_near_ties.txt, written from the oracle) and require identical choices.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from moe_inputs import CONFIGS
from tests.helpers import gpu_route

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "sigmoid_near_ties.txt")


def _pairs():
    out = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        ua, ub, D, d = line.split()
        out.append((float.fromhex(ua), float.fromhex(ub), float.fromhex(D), int(d)))
    return out


def _compare(cfg, u, sb):
    s = oracle.scores(u.astype(np.float64), "sigmoid")
    idx_o, w_o, _ = oracle.route(cfg, s, sb.astype(np.float64))
    idx_g, w_g, _ = gpu_route(cfg, u.shape[0], logits=torch.from_numpy(u).cuda(),
                              weights={"select_bias": torch.from_numpy(sb).cuda()})
    idx_g = idx_g.cpu().numpy()
    bad = np.nonzero((idx_g != idx_o).any(axis=1))[0]
    assert len(bad) == 0, f"{len(bad)} of {u.shape[0]} tokens differ, first {bad[:5]}"
    assert np.abs(w_g.cpu().numpy() - w_o).max() <= 1e-5
    return idx_o


def test_expert_decision_within_two_fp64_units():
    """No group limit, K = 8: seven clear winners, then experts A (key sigmoid(u_a)) and
    B (key sigmoid(u_b) + D) a few fp64 units apart compete for the last place."""
    cfg = CONFIGS["v3_prefill"].replace(name="ulp_e", n_groups=1, topk_groups=1, top_k=8)
    N = cfg.n_routed
    pairs = _pairs()
    rng = np.random.default_rng(5)
    per_batch = (N - 7) // 2
    chosen_a = chosen_b = 0
    for b0 in range(0, len(pairs), per_batch):
        batch = pairs[b0:b0 + per_batch]
        T = len(batch)
        u = np.full((T, N), -6.0, np.float32)
        u[:, :7] = 4.0
        sb = np.zeros(N, np.float32)
        for t, (ua, ub, D, _) in enumerate(batch):
            ea, eb = 7 + 2 * t, 8 + 2 * t
            if rng.random() < 0.5:      # B below A in index half of the time
                ea, eb = eb, ea
            u[t, ea], u[t, eb], sb[eb] = ua, ub, D
        idx = _compare(cfg, u, sb)
        for t, (ua, ub, D, _) in enumerate(batch):
            last = set(idx[t]) - set(range(7))
            assert len(last) == 1
            e = last.pop()
            if sb[e] == 0:
                chosen_a += 1
            else:
                chosen_b += 1
    assert chosen_a > 0 and chosen_b > 0


def test_group_decision_within_two_fp64_units():
    """8 groups of 32, keep 4, group score = sum of the top-2 keys: groups 0-2 are clearly in;
    group 3 (top-2: A and a key of 0.982) and group 4 (B and the same 0.982 key) compete for the
    4th place with scores a few fp64 units apart; the kept group's two experts complete K = 8."""
    cfg = CONFIGS["v3_prefill"].replace(name="ulp_g")
    N, gs = cfg.n_routed, cfg.n_routed // cfg.n_groups
    pairs = _pairs()
    rng = np.random.default_rng(6)
    per_batch = gs - 1
    for b0 in range(0, len(pairs), per_batch):
        batch = pairs[b0:b0 + per_batch]
        T = len(batch)
        u = np.full((T, N), -6.0, np.float32)
        for g in range(3):
            u[:, g * gs:g * gs + 2] = 4.0
        sb = np.zeros(N, np.float32)
        for t, (ua, ub, D, _) in enumerate(batch):
            ga, gb = (3, 4) if rng.random() < 0.5 else (4, 3)
            ea, eb = ga * gs + 1 + t, gb * gs + 1 + t
            u[t, ga * gs] = 4.0
            u[t, gb * gs] = 4.0
            u[t, ea], u[t, eb], sb[eb] = ua, ub, D
        _compare(cfg, u, sb)


def test_fp64_sigmoid_matches_the_oracle_bit_for_bit():
    """The premise of the exact recheck: CUDA's fp64 1 / (1 + exp(-u)) equals the oracle's (host
    libm) on fp32 logits. Checked on every fp32 value of the near-tie range and on 2^20 random
    logits over [-30, 30]."""
    lo, hi = np.float32(-0.504), np.float32(-0.5)
    near = np.arange(lo.view(np.int32), hi.view(np.int32), -1, dtype=np.int32).view(np.float32)
    rng = np.random.default_rng(7)
    wide = rng.uniform(-30, 30, size=1 << 20).astype(np.float32)
    u = np.concatenate([near, wide]).astype(np.float64)
    want = oracle.scores(u[None, :], "sigmoid")[0]
    ud = torch.from_numpy(u).cuda()
    got = (1.0 / (1.0 + torch.exp(-ud))).cpu().numpy()
    diff = np.nonzero(got != want)[0]
    assert len(diff) == 0, (f"{len(diff)} of {len(u)} logits differ, e.g. u={u[diff[:3]]}: "
                            f"{got[diff[:3]]} vs {want[diff[:3]]}")
