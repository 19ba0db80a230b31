"""Redundant-expert placement planner: the oracle against brute force and invariants, the
library's C++ planner against the oracle (identical plans), and the plan quality on the skewed
(Zipf) expert loads of the decode workload, in the prefill (hierarchical, EP32 with 32 redundant
experts) and decode (global, EP144 with 2 experts per GPU) deployment shapes of
"DeepSeek-V3的Group-Limited Expert Routing与负载均衡优化实践", sections 2-4. Host only."""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import oracle
from moe_inputs import CONFIGS, make_logits, make_router


def _zipf_counts(name="v3_decode_512", seed=0):
    cfg = CONFIGS[name]
    u = make_logits(cfg, seed=seed, T=cfg.T).double().numpy()
    sb = make_router(cfg)["select_bias"].double().numpy()
    idx, _, _ = oracle.route(cfg, oracle.scores(u, cfg.score_fn), sb)
    return np.bincount(idx.ravel(), minlength=cfg.n_routed)


def _check_plan(load, reps, ge, gl, n_gpus, slots):
    load = np.asarray(load)
    N = len(load)
    assert reps.sum() == n_gpus * slots and reps.min() >= 1
    assert np.all(ge >= 0)                                   # every slot used
    hosted = np.bincount(ge.ravel(), minlength=N)
    np.testing.assert_array_equal(hosted, reps)              # each replica placed once
    for e in range(N):
        gpus = np.nonzero((ge == e).any(axis=1))[0]
        if reps[e] <= n_gpus:
            assert len(gpus) == reps[e]                      # replicas on distinct GPUs
    assert abs(gl.sum() - load.sum()) <= 1e-9 * max(1, load.sum())
    lower = max(load.sum() / n_gpus, max(load[e] / reps[e] for e in range(N)))
    assert gl.max() >= lower - 1e-9


def test_replication_is_optimal_on_small_cases():
    """The replica counts minimise the largest per-replica load (brute force over all splits of
    the extra replicas, each expert capped at the number of GPUs)."""
    rng = np.random.default_rng(0)
    for _ in range(40):
        N = int(rng.integers(2, 6))
        n_gpus = int(rng.integers(2, 4))
        slots = int(rng.integers(-(-N // n_gpus), -(-N // n_gpus) + 3))
        load = rng.integers(0, 50, N)
        total = n_gpus * slots
        reps, _, _ = oracle.plan_placement(load, n_gpus, slots)
        best = None
        for split in itertools.product(range(1, n_gpus + 1), repeat=N):
            if sum(split) != total:
                continue
            v = max(Fraction(int(load[e]), split[e]) for e in range(N))
            best = v if best is None else min(best, v)
        if best is None:   # every expert at the cap still leaves slots: caps lifted
            continue
        got = max(Fraction(int(load[e]), int(reps[e])) for e in range(N))
        assert got == best


def test_uniform_loads_balance_perfectly():
    reps, ge, gl = oracle.plan_placement([7] * 16, n_gpus=4, slots=4)
    assert np.all(reps == 1) and np.all(gl == 28.0)


@pytest.mark.parametrize("nodes,groups", [(1, 0), (4, 8)])
def test_oracle_invariants_random(nodes, groups):
    rng = np.random.default_rng(1)
    for _ in range(10):
        load = rng.integers(0, 1000, 64)
        reps, ge, gl = oracle.plan_placement(load, n_gpus=16, slots=5, n_nodes=nodes,
                                             n_groups=groups)
        _check_plan(load, reps, ge, gl, 16, 5)
        if nodes > 1:   # each node hosts exactly the experts of its groups
            for n in range(nodes):
                experts = set(ge[n * 4:(n + 1) * 4].ravel().tolist())
                grp = {e // 8 for e in experts}
                assert len(grp) == groups // nodes
                assert experts == {e for g in grp for e in range(g * 8, (g + 1) * 8)}


@pytest.mark.parametrize("nodes,groups,n_gpus,slots", [(1, 0, 144, 2), (4, 8, 32, 9),
                                                      (1, 0, 16, 3), (2, 4, 8, 5)])
def test_library_planner_matches_oracle(nodes, groups, n_gpus, slots):
    import mixture_experts_routing_sigmoid_b300 as moe
    rng = np.random.default_rng(2)
    N = 256 if n_gpus * slots >= 256 else 32
    for load in (_zipf_counts(), rng.integers(0, 5000, 256), np.zeros(256, np.int64)):
        load = np.asarray(load[:N])
        got = moe.moe_plan_placement(load, n_gpus, slots, nodes, groups)
        want = oracle.plan_placement(load, n_gpus, slots, nodes, groups)
        for a, b in zip(got, want):
            np.testing.assert_array_equal(a, b)


def test_plan_reduces_imbalance_on_zipf_loads():
    """Decode routing with Zipf(1.2) popularity (21 of 256 experts take all 4096 assignments):
    with 32 redundant experts the busiest GPU carries less than the hottest expert alone, and in
    the prefill shape (32 GPUs) less than the same placement with one replica per expert."""
    load = _zipf_counts()
    # decode: 144 GPUs x 2 slots = 256 experts + 32 replicas
    reps, ge, gl = oracle.plan_placement(load, 144, 2)
    _check_plan(load, reps, ge, gl, 144, 2)
    assert gl.max() < load.max()
    # prefill: 4 nodes x 8 GPUs, 8 slots (no redundancy) against 9 slots (32 replicas)
    _, _, gl0 = oracle.plan_placement(load, 32, 8, 4, 8)
    reps, ge, gl1 = oracle.plan_placement(load, 32, 9, 4, 8)
    _check_plan(load, reps, ge, gl1, 32, 9)
    assert gl1.max() < 0.6 * gl0.max()
