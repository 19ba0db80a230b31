"""Routing decisions one or two fp64 units apart, on the GPU against the oracle.

The method ranks experts by the real numbers key = sigmoid(u) + b ("DeepSeek MoE：从v1到v3的演进",
DeepSeek-v3) and groups by real sums of keys. fp64 cannot always order keys a few units apart
(CUDA's fp64 exp and the host's differ in the last bit for a few percent of arguments), so both
sides settle such decisions by the real order: the oracle in quad precision from the logits, the
routing kernel by rescoring the keys inside its fp32 error band in double-double arithmetic;
values within 2^-80 of their size count as equal and go to the lower index. These tests put the
K-th and (K+1)-th keys (and, separately, the topk_groups-th and next group scores) 0, 1 or 2
fp64 units apart (tests/golden/sigmoid_near_ties.txt, written from the oracle), and build group
scores that are equal as real numbers, and require identical choices.
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
    u64 = u.astype(np.float64)
    s = oracle.scores(u64, "sigmoid")
    idx_o, w_o, _ = oracle.route(cfg, s, sb.astype(np.float64), u=u64)
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


def test_real_ties_of_group_scores_go_to_the_lower_group():
    """sigmoid(a) + sigmoid(-a) = 1 exactly, so groups whose top-2 keys are such pairs have equal
    real scores (their fp32 and fp64 sums may still differ by a unit): the lower group is kept."""
    cfg = CONFIGS["v3_prefill"].replace(name="ulp_tie")
    N, gs = cfg.n_routed, cfg.n_routed // cfg.n_groups
    rng = np.random.default_rng(8)
    T = 256
    u = np.full((T, N), -6.0, np.float32)
    for t in range(T):
        g = rng.choice(cfg.n_groups, size=5, replace=False)
        for h in g:
            a = np.float32(rng.uniform(0.05, 4.0))
            u[t, h * gs + 3], u[t, h * gs + 7] = a, -a
    idx = _compare(cfg, u, np.zeros(N, np.float32))
    for t in range(T):
        kept = sorted({int(e) // gs for e in idx[t]})
        g = sorted(int(h) for h in np.nonzero((u[t].reshape(cfg.n_groups, gs) > -6).any(1))[0])
        assert kept == g[:cfg.topk_groups]
