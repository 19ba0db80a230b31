"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: a hand-worked example,
a closed form, an invariant stated on the pages, brute-force enumeration on tiny inputs,
or a special case that reduces to a library routine (numpy / scipy / torch on CPU).
"""
import itertools
import os
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from moe_inputs import CONFIGS
from tests.conftest import read_golden

TINY = CONFIGS["tiny"]


def _cfg8(**kw):
    base = dict(T=1, hidden=4, n_routed=8, n_groups=4, topk_groups=2, top_k=3,
                group_score_topn=2, score_fn="sigmoid", norm_topk=True, routed_scale=1.0,
                n_shared=0, inter=2, capacity_drop=False)
    base.update(kw)
    return TINY.replace(**base)


# ------------------------------------------------------------------ routing
def test_route_golden_group_limited():
    gd = read_golden("route_group_limited.txt")
    s = np.array([gd["scores"]])
    idx, w, _ = oracle.route(_cfg8(group_score_topn=2), s)
    assert idx[0].tolist() == [int(v) for v in gd["topn2"]]
    np.testing.assert_array_equal(w[0], np.array(gd["topn2_w"]))
    idx, _, _ = oracle.route(_cfg8(group_score_topn=1), s)
    assert idx[0].tolist() == [int(v) for v in gd["topn1"]]
    idx, _, _ = oracle.route(_cfg8(n_groups=1, topk_groups=1), s)
    assert idx[0].tolist() == [int(v) for v in gd["nolimit"]]
    idx, _, _ = oracle.route(_cfg8(), np.full((1, 8), 0.5))
    assert idx[0].tolist() == [int(v) for v in gd["ties"]]


def _group_scores(key, G, topn):
    gs = len(key) // G
    return [sum(sorted(key[g * gs:(g + 1) * gs], reverse=True)[:topn]) for g in range(G)]


@pytest.mark.parametrize("topn", [1, 2])
def test_route_bruteforce_tiny_group_limited(topn):
    """Tiny-layer shape: 16 experts, 4 groups, keep 2, top-4. Enumerate all 6 group pairs and
    all 70 expert subsets inside the winning pair."""
    rng = np.random.default_rng(1)
    cfg = TINY.replace(T=200, group_score_topn=topn)
    s = rng.random((200, 16))
    b = rng.normal(0, 0.1, 16)
    idx, _, _ = oracle.route(cfg, s, b)
    for t in range(200):
        key = s[t] + b
        gsc = _group_scores(key, 4, topn)
        best_pair = max(itertools.combinations(range(4), 2), key=lambda p: gsc[p[0]] + gsc[p[1]])
        elig = [e for e in range(16) if e // 4 in best_pair]
        best = max(itertools.combinations(elig, 4), key=lambda c: sum(key[e] for e in c))
        assert idx[t].tolist() == sorted(best)
        assert len({e // 4 for e in idx[t]}) <= 2


def test_route_bruteforce_no_group_limit():
    rng = np.random.default_rng(2)
    cfg = TINY.replace(T=40, n_groups=1, topk_groups=1)
    s = rng.random((40, 16))
    idx, _, _ = oracle.route(cfg, s)
    for t in range(40):
        best = max(itertools.combinations(range(16), 4), key=lambda c: sum(s[t, e] for e in c))
        assert idx[t].tolist() == sorted(best)


@pytest.mark.parametrize("G,Gk", [(1, 1), (8, 8), (4, 4)])
def test_route_reduces_to_topk(G, Gk):
    """No group limit (G=1) or keeping every group equals plain top-K (torch.topk, fp64)."""
    rng = np.random.default_rng(3)
    cfg = CONFIGS["v3_prefill"].replace(T=64, n_groups=G, topk_groups=Gk)
    s = rng.random((64, 256))
    b = rng.normal(0, 0.1, 256)
    idx, _, _ = oracle.route(cfg, s, b)
    ref = torch.topk(torch.from_numpy(s + b), 8, dim=1).indices.sort(dim=1).values.numpy()
    np.testing.assert_array_equal(idx, ref)


def test_sigmoid_zero_bias_topk_of_logits():
    """sigmoid is monotone, so with b = 0 the chosen set is the top-K of the logits."""
    rng = np.random.default_rng(4)
    cfg = CONFIGS["v3_prefill"].replace(T=64, n_groups=1, topk_groups=1)
    u = rng.normal(0, 1, (64, 256))
    idx, _, _ = oracle.route(cfg, oracle.scores(u, "sigmoid"), np.zeros(256))
    ref = torch.topk(torch.from_numpy(u), 8, dim=1).indices.sort(dim=1).values.numpy()
    np.testing.assert_array_equal(idx, ref)


def test_device_limited_literal_walk():
    """v2 device-limited routing, stated as a walk: go down the experts in score order until
    the experts seen span M devices; those are the devices; then top-K over their experts."""
    rng = np.random.default_rng(5)
    cfg = CONFIGS["v2"].replace(T=300)
    u = rng.normal(0, 1.4, (300, 160)) + rng.normal(0, 1, 160)
    s = oracle.scores(u, "softmax")
    idx, _, _ = oracle.route(cfg, s)
    for t in range(300):
        order = np.argsort(-s[t], kind="stable")
        devs = []
        for e in order:
            d = e // 20
            if d not in devs:
                devs.append(d)
            if len(devs) == 3:
                break
        elig = [e for e in range(160) if e // 20 in devs]
        top = sorted(sorted(elig, key=lambda e: -s[t, e])[:6])
        assert idx[t].tolist() == top
        assert len({e // 20 for e in idx[t]}) <= 3


@pytest.mark.parametrize("name", ["tiny", "v1", "v2", "v3_prefill"])
def test_route_invariants(name):
    cfg = CONFIGS[name].replace(T=257)
    rng = np.random.default_rng(6)
    u = rng.normal(0, 1, (257, cfg.n_routed))
    s = oracle.scores(u, cfg.score_fn)
    b = rng.normal(0, 0.1, cfg.n_routed) if cfg.has_select_bias else None
    idx, w, margin = oracle.route(cfg, s, b)
    gs = cfg.n_routed // cfg.n_groups
    for t in range(257):
        assert len(set(idx[t].tolist())) == cfg.top_k
        assert np.all(np.diff(idx[t]) > 0)
        assert len({e // gs for e in idx[t]}) <= cfg.topk_groups
        if cfg.norm_topk:
            assert math.isclose(w[t].sum(), cfg.routed_scale, rel_tol=1e-12)
            ratio = w[t] / s[t, idx[t]]
            np.testing.assert_allclose(ratio, ratio[0], rtol=1e-12)
        else:
            np.testing.assert_allclose(w[t], s[t, idx[t]] * cfg.routed_scale, rtol=1e-15)
    assert np.all(margin >= 0)
    st = oracle.load_stats(cfg, u, s, idx)
    assert st.counts.sum() == 257 * cfg.top_k


def _near_tie_pairs():
    out = []
    for line in open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                                  "sigmoid_near_ties.txt")):
        if line.startswith("#") or not line.strip():
            continue
        ua, ub, D, d = line.split()
        out.append((float.fromhex(ua), float.fromhex(ub), float.fromhex(D), int(d)))
    return out


def test_route_near_ties_follow_the_real_order():
    """Keys a few fp64 units apart ("DeepSeek MoE：从v1到v3的演进", DeepSeek-v3: rank by
    sigmoid(u) + b): given the logits, the oracle orders them as the real numbers are ordered,
    checked against mpmath at 60 significant digits (independent of the oracle and of any
    libm exp). Real ties (differences below 2^-80 relative) go to the lower expert."""
    import mpmath
    mpmath.mp.dps = 60
    cfg = CONFIGS["v3_prefill"].replace(n_groups=1, topk_groups=1, top_k=1, n_routed=4)
    sig = lambda v: 1 / (1 + mpmath.exp(-mpmath.mpf(v)))
    n_flip = 0
    for ua, ub, D, _ in _near_tie_pairs():
        ka, kb = sig(ua), sig(ub) + mpmath.mpf(D)
        want_a = ka > kb or (abs(ka - kb) <= mpmath.mpf(2) ** -80 * max(ka, kb))  # A: lower index
        u = np.array([[ua, ub, -8.0, -8.0]])
        b = np.array([0.0, D, 0.0, 0.0])
        s = oracle.scores(u, "sigmoid")
        idx, _, _ = oracle.route(cfg, s, b, u=u)
        assert idx[0, 0] == (0 if want_a else 1), (ua, ub, D)
        idx64, _, _ = oracle.route(cfg, s, b)
        n_flip += int(idx64[0, 0] != idx[0, 0])
    # fp64 alone is not enough to order these keys: it gets some of them wrong
    assert n_flip > 0


def test_route_real_ties_of_group_scores_go_to_the_lower_group():
    """sigmoid(u) + sigmoid(-u) = 1 exactly: two groups whose top-2 keys are such pairs tie in
    the reals (their fp64 sums may differ by a unit), and the lower group wins as for any tie."""
    cfg = CONFIGS["v3_prefill"].replace(n_routed=8, n_groups=4, topk_groups=1, top_k=2,
                                        group_score_topn=2)
    rng = np.random.default_rng(3)
    for _ in range(200):
        a, c = rng.uniform(0.1, 3.0, size=2).astype(np.float32)
        u = np.array([[-8, -8, a, -a, c, -c, -8, -8]], np.float64)
        b = np.zeros(8)
        s = oracle.scores(u, "sigmoid")
        idx, _, _ = oracle.route(cfg, s, b, u=u)
        assert list(idx[0]) == [2, 3]


def test_scores_match_scipy():
    rng = np.random.default_rng(7)
    u = rng.normal(0, 3, (50, 64))
    np.testing.assert_allclose(oracle.scores(u, "sigmoid"), scipy.special.expit(u), rtol=1e-14)
    np.testing.assert_allclose(oracle.scores(u, "softmax"), scipy.special.softmax(u, axis=1),
                               rtol=1e-13)


def test_gate_logits_match_numpy():
    rng = np.random.default_rng(8)
    x, wg, gb = rng.normal(size=(9, 33)), rng.normal(size=(7, 33)), rng.normal(size=7)
    np.testing.assert_allclose(oracle.gate_logits(x, wg, gb), x @ wg.T + gb, rtol=1e-12)


# ------------------------------------------------------------------ load statistics
def test_lb_uniform_routing_is_one():
    """Token t sees a base logit vector rotated by t (T a multiple of N): every expert gets
    T K / N assignments and the same score mass, so L_B = 1 exactly."""
    gd = read_golden("load_balance_closed_forms.txt")
    for fn in ("softmax", "sigmoid"):
        cfg = TINY.replace(T=64, n_groups=1, topk_groups=1, score_fn=fn)
        base = np.linspace(-1, 1, 16) ** 3 + np.arange(16) * 1e-3
        u = np.stack([np.roll(base, t) for t in range(64)])
        s = oracle.scores(u, fn)
        idx, _, _ = oracle.route(cfg, s)
        st = oracle.load_stats(cfg, u, s, idx)
        assert np.all(st.counts == 64 * 4 // 16)
        assert math.isclose(st.lb, gd["uniform_lb"][0], rel_tol=1e-12)


def test_lb_collapse_is_n_over_k():
    gd = read_golden("load_balance_closed_forms.txt")
    N, K = int(gd["collapse_N"][0]), int(gd["collapse_K"][0])
    cfg = TINY.replace(T=32, n_groups=1, topk_groups=1, score_fn="softmax", top_k=K)
    u = np.full((32, N), -2000.0)
    u[:, [1, 5, 9, 14]] = 0.0  # same K experts for every token, equal probability 1/K
    s = oracle.scores(u, "softmax")
    idx, _, _ = oracle.route(cfg, s)
    assert np.all(idx == [1, 5, 9, 14])
    st = oracle.load_stats(cfg, u, s, idx)
    assert math.isclose(st.lb, gd["collapse_lb"][0], rel_tol=1e-12)


def test_zloss_constant_logits():
    gd = read_golden("load_balance_closed_forms.txt")
    c, N = gd["const_c"][0], int(gd["const_N"][0])
    cfg = TINY.replace(T=5, n_groups=1, topk_groups=1)
    u = np.full((5, N), c)
    s = oracle.scores(u, "sigmoid")
    idx, _, _ = oracle.route(cfg, s)
    st = oracle.load_stats(cfg, u, s, idx)
    assert math.isclose(st.lse_mean, gd["const_lse"][0], rel_tol=1e-14)
    assert math.isclose(st.zloss, gd["const_lz"][0], rel_tol=1e-14)


def test_zloss_and_P_match_library():
    rng = np.random.default_rng(9)
    cfg = CONFIGS["v1"].replace(T=100)
    u = rng.normal(0, 2, (100, 64))
    s = oracle.scores(u, "softmax")
    idx, _, _ = oracle.route(cfg, s)
    st = oracle.load_stats(cfg, u, s, idx)
    lse = scipy.special.logsumexp(u, axis=1)
    assert math.isclose(st.zloss, float(np.mean(lse ** 2)), rel_tol=1e-12)
    assert math.isclose(st.lse_mean, float(np.mean(lse)), rel_tol=1e-12)
    # softmax: the page's two statements of P_i agree (score share = mean probability)
    np.testing.assert_allclose(st.P, s.mean(axis=0), rtol=1e-12)
    np.testing.assert_array_equal(st.counts, np.bincount(idx.ravel(), minlength=64))
    np.testing.assert_allclose(st.f, st.counts / (100 * 6), rtol=1e-15)


# ------------------------------------------------------------------ v2 device-level drop
def _drop_case(T=600, skew=2.0, seed=10):
    rng = np.random.default_rng(seed)
    cfg = CONFIGS["v2"].replace(T=T)
    u = rng.normal(0, 1.4, (T, 160)) + rng.normal(0, skew, 160)
    s = oracle.scores(u, "softmax")
    idx, w, _ = oracle.route(cfg, s)
    return cfg, idx, w


def test_drop_invariants():
    cfg, idx, w = _drop_case()
    kept = oracle.capacity_drop(cfg, idx, w).astype(bool)
    C = math.ceil(cfg.T * cfg.top_k / 8)
    dev = idx // 20
    dropped_any = False
    for d in range(8):
        m = dev == d
        Td = int(m.sum())
        assert int(kept[m].sum()) == min(Td, C)
        if Td > C:
            dropped_any = True
            assert w[m & ~kept].max() <= w[m & kept].min()
    assert dropped_any


def test_drop_uniform_load_keeps_everything():
    cfg = CONFIGS["v2"].replace(T=160)
    # token t's experts: device (t mod 8) gets two, the next two devices two each -> balanced
    idx = np.array([[((t + j) % 8) * 20 + (t // 8 + i) % 20 for j in range(3) for i in range(2)]
                    for t in range(160)], np.int32)
    w = np.random.default_rng(11).random(idx.shape)
    loads = np.bincount((idx // 20).ravel(), minlength=8)
    assert np.all(loads == 160 * 6 // 8)
    assert oracle.capacity_drop(cfg, idx, w).all()


def test_drop_ties_keep_lower_token_then_slot():
    cfg = CONFIGS["v2"].replace(T=16)
    idx = np.tile(np.array([0, 1, 2, 3, 4, 5], np.int32), (16, 1))  # everything on device 0
    w = np.full(idx.shape, 0.25)
    kept = oracle.capacity_drop(cfg, idx, w)
    C = math.ceil(16 * 6 / 8)
    assert kept.ravel().tolist() == [1] * C + [0] * (16 * 6 - C)


# ------------------------------------------------------------------ permutation
def test_permute_matches_stable_argsort():
    cfg, idx, w = _drop_case(T=333, seed=12)
    kept = oracle.capacity_drop(cfg, idx, w)
    offs, row_token, slot_row = oracle.permute(cfg, idx, kept)
    flat_e = idx.ravel()
    keep = kept.ravel().astype(bool)
    a_ids = np.nonzero(keep)[0]
    order = a_ids[np.argsort(flat_e[a_ids], kind="stable")]
    np.testing.assert_array_equal(row_token, order // cfg.top_k)
    expect_slot = -np.ones(idx.size, np.int64)
    expect_slot[order] = np.arange(len(order))
    np.testing.assert_array_equal(slot_row.ravel(), expect_slot)
    np.testing.assert_array_equal(offs, np.concatenate([[0], np.cumsum(
        np.bincount(flat_e[keep], minlength=160))]))


# ------------------------------------------------------------------ expert FFN and combine
def test_swiglu_golden():
    gd = read_golden("swiglu_closed_form.txt")
    y = oracle.swiglu_rows(np.array([gd["x"]]), np.array(gd["w13"]).reshape(2, 2),
                           np.array(gd["w2"]).reshape(2, 1))
    np.testing.assert_allclose(y[0], gd["y"], rtol=1e-15, atol=0)


def test_swiglu_matches_numpy_matmul():
    rng = np.random.default_rng(13)
    x, w13, w2 = rng.normal(size=(5, 48)), rng.normal(size=(2 * 24, 48)), rng.normal(size=(48, 24))
    a, g = x @ w13[:24].T, x @ w13[24:].T
    ref = (a * scipy.special.expit(a) * g) @ w2.T
    np.testing.assert_allclose(oracle.swiglu_rows(x, w13, w2), ref, rtol=1e-11, atol=1e-12)


def _small_layer(cfg, seed=14):
    rng = np.random.default_rng(seed)
    H, N, I, S = cfg.hidden, cfg.n_routed, cfg.inter, cfg.n_shared
    x = rng.normal(size=(cfg.T, H))
    wg = rng.normal(0, 0.3, (N, H))
    w13 = rng.normal(0, 0.2, (N, 2 * I, H))
    w2 = rng.normal(0, 0.2, (N, H, I))
    w13s = rng.normal(0, 0.2, (S, 2 * I, H))
    w2s = rng.normal(0, 0.2, (S, H, I))
    return x, wg, w13, w2, w13s, w2s


def test_layer_single_expert_is_dense_swiglu():
    """N = 1, K = 1, softmax: every token goes to the one expert with weight 1, so the layer is
    routed SwiGLU + shared SwiGLU, written here with numpy matmuls."""
    cfg = TINY.replace(T=7, hidden=16, n_routed=1, n_groups=1, topk_groups=1, top_k=1,
                       score_fn="softmax", norm_topk=False, n_shared=1, inter=8)
    x, wg, w13, w2, w13s, w2s = _small_layer(cfg)
    res = oracle.layer_forward(cfg, x, wg, None, None, lambda e: (w13[e], w2[e]),
                               lambda s: (w13s[s], w2s[s]))

    def dense(w13_, w2_):
        a, g = x @ w13_[:8].T, x @ w13_[8:].T
        return (a * scipy.special.expit(a) * g) @ w2_.T
    np.testing.assert_allclose(res["out"], dense(w13[0], w2[0]) + dense(w13s[0], w2s[0]),
                               rtol=1e-11, atol=1e-12)


def test_layer_token_permutation_equivariance():
    cfg = TINY.replace(T=24, hidden=32, inter=16)
    x, wg, w13, w2, w13s, w2s = _small_layer(cfg, seed=15)
    ew, sw = (lambda e: (w13[e], w2[e])), (lambda s: (w13s[s], w2s[s]))
    out = oracle.layer_forward(cfg, x, wg, None, None, ew, sw)["out"]
    perm = np.random.default_rng(16).permutation(24)
    out_p = oracle.layer_forward(cfg, x[perm], wg, None, None, ew, sw)["out"]
    np.testing.assert_allclose(out_p, out[perm], rtol=1e-12, atol=1e-13)


def test_layer_subset_equals_full_rows():
    cfg = TINY.replace(T=30, hidden=32, inter=16)
    x, wg, w13, w2, w13s, w2s = _small_layer(cfg, seed=17)
    ew, sw = (lambda e: (w13[e], w2[e])), (lambda s: (w13s[s], w2s[s]))
    full = oracle.layer_forward(cfg, x, wg, None, None, ew, sw)
    sub = oracle.layer_forward(cfg, x, wg, None, None, ew, sw, tokens=[2, 3, 11, 29])
    np.testing.assert_allclose(sub["out"], full["out"][[2, 3, 11, 29]], rtol=1e-13, atol=1e-14)


def test_layer_combine_is_weighted_sum_of_expert_outputs():
    """out_t - shared_t equals sum_k w_tk * SwiGLU_{e_k}(x_t), each expert applied alone."""
    cfg = TINY.replace(T=6, hidden=32, inter=16)
    x, wg, w13, w2, w13s, w2s = _small_layer(cfg, seed=18)
    res = oracle.layer_forward(cfg, x, wg, None, None, lambda e: (w13[e], w2[e]),
                               lambda s: (w13s[s], w2s[s]))
    for t in range(6):
        acc = oracle.swiglu_rows(x[t:t + 1], w13s[0], w2s[0])[0]
        for k in range(cfg.top_k):
            e = res["idx"][t, k]
            acc = acc + res["w"][t, k] * oracle.swiglu_rows(x[t:t + 1], w13[e], w2[e])[0]
        np.testing.assert_allclose(res["out"][t], acc, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ bias update (v3)
def test_bias_update_sign_rule():
    """Overloaded experts (count above the mean) lose u, underloaded gain u, exact mean: 0."""
    counts = np.array([10, 2, 6, 6])  # mean 6
    b = oracle.bias_update(counts, 0.001, np.zeros(4))
    np.testing.assert_array_equal(b, [-0.001, 0.001, 0.0, 0.0])


def test_bias_update_fractional_mean_and_balance():
    """A fractional mean leaves no expert at it; a perfectly balanced batch changes nothing;
    every step is exactly +u, -u or 0 and moves each bias against its expert's load."""
    b0 = np.array([0.5, -0.25, 0.125])
    b = oracle.bias_update(np.array([3, 4, 4]), 0.25, b0)     # mean 11/3
    np.testing.assert_array_equal(b - b0, [0.25, -0.25, -0.25])
    np.testing.assert_array_equal(oracle.bias_update(np.full(8, 7), 0.5, np.arange(8.0)),
                                  np.arange(8.0))
    rng = np.random.default_rng(3)
    c = rng.integers(0, 100, 64)
    d = oracle.bias_update(c, 0.125, np.zeros(64))
    assert set(np.unique(d)) <= {-0.125, 0.0, 0.125}
    assert np.all((d > 0) == (c * 64 < c.sum())) and np.all((d < 0) == (c * 64 > c.sum()))


def test_swiglu_bf16_weights_equal_widened_f64():
    """The bf16-weight entry widens exactly: same result as the fp64 entry on the same values."""
    g = torch.Generator().manual_seed(19)
    x = torch.randn((3, 64), generator=g, dtype=torch.float64).numpy()
    w13 = (torch.randn((2 * 32, 64), generator=g) * 0.1).to(torch.bfloat16)
    w2 = (torch.randn((64, 32), generator=g) * 0.1).to(torch.bfloat16)
    a = oracle.swiglu_rows(x, w13, w2)
    b = oracle.swiglu_rows(x, w13.to(torch.float64).numpy(), w2.to(torch.float64).numpy())
    np.testing.assert_array_equal(a, b)


# ------------------------------------------------------------------ sequence-wise balance loss
def _uniform_stats_inputs(N, K, T, shift0=0):
    """Logits whose routing gives every expert exactly T K / N assignments and P_e = 1/N:
    token t's logit vector is a fixed base vector cyclically shifted by (shift0 + t K) mod N."""
    base = np.linspace(3.0, -3.0, N)
    u = np.stack([np.roll(base, (shift0 + t * K) % N) for t in range(T)])
    return u


def test_seq_balance_one_sequence_is_batch_loss():
    cfg = CONFIGS["tiny"]
    rng = np.random.default_rng(5)
    u = rng.normal(0, 1, (cfg.T, cfg.n_routed))
    s = oracle.scores(u, cfg.score_fn)
    idx, _, _ = oracle.route(cfg, s, np.zeros(cfg.n_routed))
    per, mean = oracle.seq_balance_loss(cfg, u, s, idx, cfg.T)
    assert per.shape == (1,)
    assert mean == oracle.load_stats(cfg, u, s, idx).lb


def test_seq_balance_uniform_sequences_give_one():
    """Routing uniform inside every sequence: each sequence's loss is 1, so is the mean."""
    cfg = CONFIGS["v1"].replace(T=256, n_routed=16, top_k=4)
    N, K, L = 16, 4, 64
    u = _uniform_stats_inputs(N, K, cfg.T)
    s = oracle.scores(u, "softmax")
    idx, _, _ = oracle.route(cfg, s, None)
    per, mean = oracle.seq_balance_loss(cfg, u, s, idx, L)
    np.testing.assert_allclose(per, 1.0, rtol=1e-12)
    assert abs(mean - 1.0) < 1e-12


def test_seq_balance_sees_imbalance_the_batch_loss_hides():
    """Each sequence sends all its tokens to its own K experts with equal scores there: every
    sequence is collapsed (loss N / K) while the batch as a whole is perfectly balanced
    (loss 1). The sequence-wise loss must report the collapse."""
    N, K, L = 16, 4, 32
    cfg = CONFIGS["v1"].replace(T=L * (N // K), n_routed=N, top_k=K)
    u = np.full((cfg.T, N), -40.0)
    for b in range(N // K):
        u[b * L:(b + 1) * L, b * K:(b + 1) * K] = 0.0
    s = oracle.scores(u, "softmax")
    idx, _, _ = oracle.route(cfg, s, None)
    per, mean = oracle.seq_balance_loss(cfg, u, s, idx, L)
    np.testing.assert_allclose(per, N / K, rtol=1e-12)
    assert abs(oracle.load_stats(cfg, u, s, idx).lb - 1.0) < 1e-12


# ------------------------------------------------------------------ device / communication losses
def _route(cfg, u, sb=None):
    s = oracle.scores(u, cfg.score_fn)
    idx, _, _ = oracle.route(cfg, s, sb)
    return s, idx


def test_group_losses_one_expert_per_device_is_expert_loss():
    """With as many devices as experts, the device-level loss is the expert-level L_B."""
    cfg = CONFIGS["v1"].replace(T=128, n_routed=16, top_k=4, n_groups=16, topk_groups=16)
    u = np.random.default_rng(8).normal(0, 1, (cfg.T, 16))
    s, idx = _route(cfg, u)
    l_dev, _ = oracle.group_balance_losses(cfg, u, s, idx)
    assert abs(l_dev - oracle.load_stats(cfg, u, s, idx).lb) < 1e-12


def test_group_losses_top1_communication_equals_device_loss():
    """With one expert per token each token reaches exactly one device, so the received-token
    shares equal the assignment shares and the two losses coincide."""
    cfg = CONFIGS["v1"].replace(T=200, n_routed=16, top_k=1, n_groups=4, topk_groups=4)
    u = np.random.default_rng(9).normal(0, 1, (cfg.T, 16))
    s, idx = _route(cfg, u)
    l_dev, l_comm = oracle.group_balance_losses(cfg, u, s, idx)
    assert abs(l_dev - l_comm) < 1e-12


def test_group_losses_uniform_routing_gives_one():
    N, K, G = 16, 4, 4
    cfg = CONFIGS["v1"].replace(T=64, n_routed=N, top_k=K, n_groups=G, topk_groups=G)
    u = _uniform_stats_inputs(N, K, cfg.T)
    s, idx = _route(cfg, u)
    l_dev, l_comm = oracle.group_balance_losses(cfg, u, s, idx)
    assert abs(l_dev - 1.0) < 1e-12 and abs(l_comm - 1.0) < 1e-12


def test_group_losses_collapse_onto_one_device():
    """Every token sends all its assignments and (almost) all its score to device 0: both losses
    approach G, the number of devices."""
    N, K, G = 16, 4, 4
    cfg = CONFIGS["v1"].replace(T=32, n_routed=N, top_k=K, n_groups=G, topk_groups=G)
    u = np.full((cfg.T, N), -60.0)
    u[:, :4] = 0.0
    s, idx = _route(cfg, u)
    l_dev, l_comm = oracle.group_balance_losses(cfg, u, s, idx)
    np.testing.assert_allclose([l_dev, l_comm], [G, G], rtol=1e-12)
