"""Pins of the oracle's adaptive-verification (AV) pruning and of pruned
(ragged) verification.

"Verificación Adaptativa sin una cabeza de confianza": AV verifies a subset of
the drafts ("Antecedentes"); survival is the running product of the
confidences, the drafts are ranked by it over the batch, and the budget
maximises the expected emitted tokens per measured cost ("Otras
Características Consideradas"). Pruning on the draft distribution's q_max,
never on the sampled token, keeps speculative decoding lossless (footnote 1
shows the bias of pruning on q(x)). Each test ties the oracle to a hand
computation, brute force over subsets, the unpruned oracle on a truncated
problem, closed forms, or a Monte Carlo chi-square. CPU only.
"""
import itertools

import numpy as np
import pytest
from scipy import special, stats

import oracle


def _costs(N, a=1.0, b=0.2, rng=None):
    v = a + b * np.arange(N + 1)
    if rng is not None:
        v = v * rng.uniform(0.9, 1.1, N + 1)
    return np.zeros(N + 1, np.float32), v.astype(np.float32)


def test_budget_hand_case():
    # survival [[.9, .45], [.6, .06]]; ranked .9, .6, .45, .06; S_k = 0, .9,
    # 1.5, 1.95, 2.01; (2 + S_k) / cost_k with cost 1, 1.2, 1.4, 1.6, 1.8 =
    # 2, 2.4167, 2.5, 2.4688, 2.2333: budget 2, the first draft of each
    conf = np.array([[0.9, 0.5], [0.6, 0.1]], np.float32)
    dc = np.zeros(5, np.float32)
    vc = np.array([1.0, 1.2, 1.4, 1.6, 1.8], np.float32)
    r = oracle.av_budget(conf, dc, vc)
    assert r["budget"] == 2
    np.testing.assert_array_equal(r["draft_len"], [1, 1])
    np.testing.assert_allclose(r["survival"], [[0.9, 0.45], [0.6, 0.06]], rtol=1e-6)
    np.testing.assert_allclose(r["objective"], [2.0, 2.9 / 1.2, 3.5 / 1.4, 3.95 / 1.6, 4.01 / 1.8], rtol=1e-6)


@pytest.mark.parametrize("seed", range(8))
def test_budget_against_brute_force_over_subsets(seed):
    rng = np.random.default_rng(seed)
    B, K = int(rng.integers(1, 4)), int(rng.integers(1, 4))
    conf = rng.uniform(0.05, 0.99, (B, K)).astype(np.float32)
    N = B * K
    dc, vc = _costs(N, 1.0, float(rng.uniform(0.05, 0.6)), rng)
    r = oracle.av_budget(conf, dc, vc)
    surv = np.cumprod(conf.astype(np.float64), axis=1).ravel()
    cost = dc.astype(np.float64) + vc.astype(np.float64)
    best = max((B + surv[list(sub)].sum()) / cost[len(sub)]
               for k in range(N + 1) for sub in itertools.combinations(range(N), k))
    np.testing.assert_allclose(r["objective"][r["budget"]], best, rtol=1e-6)
    # the winners are a prefix of each sequence and attain the best objective
    win = np.concatenate([np.arange(b * K, b * K + r["draft_len"][b]) for b in range(B)]).astype(int)
    assert r["draft_len"].sum() == r["budget"]
    np.testing.assert_allclose((B + surv[win].sum()) / cost[len(win)], best, rtol=1e-6)


def test_ties_keep_prefixes_and_bad_costs_are_ineligible():
    conf = np.array([[1.0, 1.0, 0.5], [1.0, 0.0, 1.0]], np.float32)   # ties in survival
    dc = np.zeros(7, np.float32)
    vc = np.array([1, 1, 1, 1, 1, 1, 1], np.float32)
    r = oracle.av_budget(conf, dc, vc)
    # ranked: (0,0) (0,1) (1,0) all 1.0, then (0,2) .5, then the zeros
    assert r["budget"] == 4 and list(r["draft_len"]) == [3, 1]
    vc2 = np.array([1, -1, 0, np.nan, 1, 1, 1], np.float32)
    r2 = oracle.av_budget(conf, dc, vc2)
    assert np.isneginf(r2["objective"][1:4]).all() and r2["budget"] == 4
    r3 = oracle.av_budget(conf, dc, np.zeros(7, np.float32))
    assert r3["budget"] == 0 and list(r3["draft_len"]) == [0, 0]


def test_cross_sequence_ties_rank_by_index():
    # Equal survival in different sequences, with a budget that cuts through
    # the tie: the reading ranks ties by ascending flat index b*K + i, so the
    # lower sequence gets the draft. Objectives (B + S_k) / cost_k with
    # survival .5 everywhere: K = 1, costs 1, 1, 2 give 2, 2.5, 1.5.
    conf = np.array([[0.5], [0.5]], np.float32)
    r = oracle.av_budget(conf, np.zeros(3, np.float32), np.array([1, 1, 2], np.float32))
    assert r["budget"] == 1 and list(r["draft_len"]) == [1, 0]
    # three sequences, two drafts each, all survival .25 after the first:
    # costs make a budget of 4 best; ranked (0,0) (1,0) (2,0) at .5, then
    # (0,1) at .25 -- the lowest sequence takes the tied second draft
    conf = np.array([[0.5, 0.5], [0.5, 0.5], [0.5, 0.5]], np.float32)
    vc = np.array([1, 1, 1, 1, 1, 4, 4], np.float32)
    r = oracle.av_budget(conf, np.zeros(7, np.float32), vc)
    assert r["budget"] == 4 and list(r["draft_len"]) == [2, 1, 1]


def _problem(seed, B=6, K=5, V=64):
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    zd = (zt[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
    q = special.softmax(zd.astype(np.float64), axis=-1)
    x = np.array([[rng.choice(V, p=q[b, i]) for i in range(K)] for b in range(B)], np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    return zt, zd, x, u


@pytest.mark.parametrize("mode", [oracle.STOCHASTIC, oracle.GREEDY, oracle.FLY])
def test_full_draft_length_is_the_unpruned_verify(mode):
    zt, zd, x, u = _problem(1)
    B, K = x.shape
    a = oracle.verify(zt, zd, x, u, mode=mode, fly_theta=0.5, fly_window=2, est_params=np.ones(K + 1))
    b = oracle.verify(zt, zd, x, u, mode=mode, fly_theta=0.5, fly_window=2, est_params=np.ones(K + 1),
                      draft_len=np.full(B, K))
    for k in ("out_tokens", "accepted_len", "flags"):
        np.testing.assert_array_equal(a[k], b[k])
    for k in ("pos_stats", "feature", "conf"):
        np.testing.assert_array_equal(a[k], b[k])


@pytest.mark.parametrize("mode", [oracle.STOCHASTIC, oracle.GREEDY, oracle.FLY])
def test_pruned_sequence_equals_the_truncated_problem(mode):
    zt, zd, x, u = _problem(2, B=8, K=5)
    B, K = x.shape
    dl = np.array([5, 4, 3, 2, 1, 1, 3, 5], np.int32)
    est = np.linspace(0.5, 1.5, K + 1)
    r = oracle.verify(zt, zd, x, u, mode=mode, fly_theta=0.5, fly_window=2, est_params=est, draft_len=dl)
    for b in range(B):
        kb = int(dl[b])
        ub = np.concatenate([u[b, :kb], u[b, K:]])[None]
        t = oracle.verify(zt[b:b + 1, :kb + 1], zd[b:b + 1, :kb], x[b:b + 1, :kb], ub, mode=mode,
                          fly_theta=0.5, fly_window=2, est_params=est[:kb + 1])
        assert r["accepted_len"][b] == t["accepted_len"][0]
        np.testing.assert_array_equal(r["out_tokens"][b, :kb + 1], t["out_tokens"][0])
        assert (r["out_tokens"][b, kb + 1:] == -1).all()
        np.testing.assert_array_equal(r["pos_stats"][b, :kb + 1, :2], t["pos_stats"][0, :, :2])
        np.testing.assert_array_equal(r["feature"][b, :kb], t["feature"][0])
        assert np.isnan(r["feature"][b, kb:]).all() and np.isnan(r["pos_stats"][b, kb + 1:]).all()


def test_nothing_verified_draws_from_the_first_target_row():
    zt, zd, x, u = _problem(3, B=5, K=3)
    B, K = x.shape
    r = oracle.verify(zt, zd, x, u, draft_len=np.zeros(B, np.int32))
    p = special.softmax(zt[:, 0].astype(np.float64), axis=-1)
    for b in range(B):
        c = np.cumsum(p[b])
        tok = int(np.argmax(c > u[b, K] * c[-1]))      # smallest v with running sum > u * Z
        assert r["accepted_len"][b] == 0 and r["out_tokens"][b, 0] == tok
        assert (r["out_tokens"][b, 1:] == -1).all()


def test_pruned_labels():
    rng = np.random.default_rng(4)
    B, K = 40, 5
    f = rng.normal(0, 2, (B, K))
    dl = rng.integers(0, K + 1, B).astype(np.int32)
    n = np.array([rng.integers(0, d + 1) for d in dl], np.int32)
    _, _, cnt = oracle.estimator_update(f, n, np.zeros(K + 1), 0.0, draft_len=dl)
    # positions 0..n labelled, except position n when all K_b verified drafts were accepted
    expect = sum(min(int(a), int(d) - 1) + 1 for a, d in zip(n, dl) if d > 0)
    assert cnt[0] == expect
    st = oracle.irls_zero(K)
    oracle.irls_accumulate(f, n, np.zeros(K + 1), st, draft_len=dl)
    assert st[2][0] == expect
    with pytest.raises(ValueError):
        oracle.estimator_update(f, np.full(B, K, np.int32), np.zeros(K + 1), 0.0, draft_len=np.zeros(B, np.int32))


def test_pruning_on_q_max_stays_lossless():
    # tiny vocabulary: prune with the budget on confidences from logit(q_max),
    # which does not look at the sampled draft token; the first emitted token
    # must still follow the target row 0
    rng = np.random.default_rng(5)
    V, K, B, reps = 4, 3, 4000, 25
    pt = np.array([[0.1, 0.2, 0.3, 0.4], [0.4, 0.3, 0.2, 0.1], [0.25, 0.25, 0.25, 0.25],
                   [0.7, 0.1, 0.1, 0.1]])
    pd = np.array([[0.3, 0.3, 0.2, 0.2], [0.1, 0.2, 0.3, 0.4], [0.6, 0.2, 0.1, 0.1]])
    zt = np.broadcast_to(np.log(pt).astype(np.float32), (B, K + 1, V)).copy()
    zd = np.broadcast_to(np.log(pd).astype(np.float32), (B, K, V)).copy()
    counts = np.zeros(V)
    for _ in range(reps):
        # per-sequence draft distributions vary through a random temperature
        tau = rng.uniform(0.5, 2.0, B).astype(np.float32)
        zdb = (zd / tau[:, None, None]).astype(np.float32)
        q = special.softmax(zdb.astype(np.float64), axis=-1)
        x = (q.cumsum(-1) > rng.random((B, K, 1))).argmax(-1).astype(np.int32)
        u = rng.random((B, K + 1)).astype(np.float32)
        fq = np.log(q.max(-1)) - np.log1p(-q.max(-1))
        conf = special.expit(0.5 * fq + 0.2).astype(np.float32)
        dc, vc = _costs(B * K, 1.0, 0.3 / B)
        dl = oracle.av_budget(conf, dc, vc)["draft_len"]
        assert 0 < dl.sum() < B * K
        r = oracle.verify(zt, zdb, x, u, draft_len=dl)
        counts += np.bincount(r["out_tokens"][:, 0], minlength=V)
    _, pval = stats.chisquare(counts, pt[0] * counts.sum())
    assert pval > 1e-3, (counts / counts.sum(), pval)


def test_pruning_on_the_sampled_token_is_caught():
    # negative control for the test above: pruning on q(x_0) (footnote 1's
    # rule) biases the first token, and the same chi-square detects it
    rng = np.random.default_rng(6)
    V, K, B = 4, 1, 40000
    pt = np.array([[0.5, 0.5, 0.0, 0.0], [0.25, 0.25, 0.25, 0.25]]) + 1e-9
    pd = np.array([[0.2, 0.8, 0.0, 0.0]]) + 1e-9
    zt = np.broadcast_to(np.log(pt).astype(np.float32), (B, K + 1, V)).copy()
    zd = np.broadcast_to(np.log(pd).astype(np.float32), (B, K, V)).copy()
    q = special.softmax(zd.astype(np.float64), axis=-1)
    x = (q.cumsum(-1) > rng.random((B, K, 1))).argmax(-1).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    dl = (q[np.arange(B), 0, x[:, 0]] >= 0.5).astype(np.int32)      # verify only if q(x) >= 0.5
    r = oracle.verify(zt, zd, x, u, draft_len=dl)
    counts = np.bincount(r["out_tokens"][:, 0], minlength=V)[:2]
    np.testing.assert_allclose(counts / counts.sum(), [0.4, 0.6], atol=0.01)   # footnote 1's [0.4, 0.6]
    _, pval = stats.chisquare(counts, np.array([0.5, 0.5]) * counts.sum())
    assert pval < 1e-6
