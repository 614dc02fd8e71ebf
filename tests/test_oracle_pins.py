"""Pins of the fp64 oracle against facts the pages and mathematics fix.

Each test ties an oracle function to something other than its own code: the
worked example printed in the pages, the losslessness theorem (Monte Carlo
chi-square), closed forms, library routines (scipy's logsumexp and entropy),
and brute force over tiny vocabularies. CPU only.
"""
import json
import os

import numpy as np
import pytest
from scipy import special, stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _softmax64(z):
    z = np.asarray(z, np.float64)
    return np.exp(z - special.logsumexp(z, axis=-1, keepdims=True))


def _rows(p):
    """fp32 logits whose softmax is (to fp32 rounding) the rows p."""
    return np.log(np.asarray(p, np.float64)).astype(np.float32)


# ---------------------------------------------------------------------------
# Worked example: "Verificación Adaptativa sin una cabeza de confianza",
# footnote 1 (p = [.5,.5], q = [.2,.8]).
# ---------------------------------------------------------------------------

def test_footnote_two_token_example():
    g = json.load(open(os.path.join(GOLDEN, "two_token_footnote.json")))
    p, q = np.array(g["p"]), np.array(g["q"])
    N = 20000
    uu = (np.arange(N) + 0.5) / N                     # midpoint grid on [0,1)
    zt = np.repeat(_rows([p, p])[None], N, 0)          # K = 1: rows 0 and 1 (bonus)
    zd = np.repeat(_rows([q])[None], N, 0)

    # draft token b: the ratio p(b)/q(b) and the acceptance frequency
    x = np.ones((N, 1), np.int32)
    u = np.stack([uu, np.full(N, 0.5)], 1).astype(np.float32)
    r = oracle.verify(zt, zd, x, u)
    ratio = np.exp(r["pos_stats"][:, 0, 2])
    np.testing.assert_allclose(ratio, g["accept_prob_b"], rtol=1e-6)
    acc_freq = r["accepted_len"].mean()
    assert abs(acc_freq - g["accept_prob_b"]) <= 1.0 / N
    # every rejection draws from the residual [1, 0]: always token a
    rej = r["accepted_len"] == 0
    assert (r["out_tokens"][rej, 0] == 0).all()
    # a residual draw across the whole u grid stays on the residual's support
    u2 = np.stack([np.full(N, 0.999999), uu], 1).astype(np.float32)
    r2 = oracle.verify(zt, zd, x, u2)
    assert (r2["accepted_len"] == 0).all() and (r2["out_tokens"][:, 0] == 0).all()

    # draft token a: ratio 2.5 -> always accepted
    xa = np.zeros((N, 1), np.int32)
    ra = oracle.verify(zt, zd, xa, u)
    assert (ra["accepted_len"] == 1).all()

    # composition over x ~ q: without pruning the first token follows p
    p_rej_b = 1.0 - acc_freq
    out_a = q[0] * 1.0 + q[1] * p_rej_b * 1.0
    np.testing.assert_allclose([out_a, 1 - out_a], g["output_without_pruning"], atol=2.0 / N)
    # with pruning of drafts whose q(x) < 0.5 the target draws x=a's slot from p
    out_a_pruned = q[0] * p[0] + q[1] * p_rej_b
    np.testing.assert_allclose([out_a_pruned, 1 - out_a_pruned], g["output_with_pruning"],
                               atol=2.0 / N)


# ---------------------------------------------------------------------------
# Losslessness ("Speculative Decoding: ...", "Математика верификации": the
# emitted token is distributed exactly as p). Monte Carlo chi-square, 1e6 trials.
# ---------------------------------------------------------------------------

def _chi2_pvalue(counts, probs):
    n = counts.sum()
    expct = probs * n
    keep = expct > 0
    assert counts[~keep].sum() == 0, "token drawn outside the support of p"
    chi2 = ((counts[keep] - expct[keep]) ** 2 / expct[keep]).sum()
    return stats.chi2.sf(chi2, keep.sum() - 1)


@pytest.mark.parametrize("V,K", [(2, 1), (4, 2), (8, 4), (16, 1), (16, 2), (16, 4)])
def test_lossless_chi_square(V, K):
    rng = np.random.default_rng(1000 + 31 * V + K)
    zt1 = rng.normal(0, 1.5, (K + 1, V)).astype(np.float32)
    zd1 = (zt1[:K] + rng.normal(0, 1.0, (K, V))).astype(np.float32)
    p = _softmax64(zt1)
    q = _softmax64(zd1)
    trials, chunk = 1_000_000, 100_000
    first = np.zeros(V, np.int64)
    second = np.zeros(V, np.int64)
    acc0 = 0
    for c in range(trials // chunk):
        x = np.stack([rng.choice(V, size=chunk, p=q[i]) for i in range(K)], 1).astype(np.int32)
        u = rng.random((chunk, K + 1), dtype=np.float32)
        r = oracle.verify(np.broadcast_to(zt1, (chunk, K + 1, V)),
                          np.broadcast_to(zd1, (chunk, K, V)), x, u)
        first += np.bincount(r["out_tokens"][:, 0], minlength=V)
        sel = r["accepted_len"] >= 1
        acc0 += sel.sum()
        second += np.bincount(r["out_tokens"][sel, 1], minlength=V)
    assert _chi2_pvalue(first, p[0]) > 1e-4
    assert _chi2_pvalue(second, p[1]) > 1e-4
    # closed form of the acceptance probability at position 0: sum_v min(p, q)
    a = np.minimum(p[0], q[0]).sum()
    assert abs(acc0 / trials - a) < 5 * np.sqrt(a * (1 - a) / trials)


def test_p_equals_q_accepts_everything():
    rng = np.random.default_rng(7)
    B, K, V = 64, 5, 300
    zt = rng.normal(0, 3, (B, K + 1, V)).astype(np.float32)
    zd = zt[:, :K].copy()
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1), dtype=np.float32)
    r = oracle.verify(zt, zd, x, u)
    assert (r["accepted_len"] == K).all()
    assert (r["out_tokens"][:, :K] == x).all()
    np.testing.assert_allclose(r["pos_stats"][:, :K, 2], 0.0, atol=1e-12)


def test_bonus_draw_follows_last_target_row():
    # all K drafts accepted (p == q): the bonus token is an inverse-CDF draw from p_K
    rng = np.random.default_rng(11)
    V, K, N = 6, 2, 30000
    zt1 = rng.normal(0, 1, (K + 1, V)).astype(np.float32)
    pK = _softmax64(zt1[K])
    uu = (np.arange(N) + 0.5) / N
    u = np.stack([np.zeros(N), np.zeros(N), uu], 1).astype(np.float32)
    x = np.zeros((N, K), np.int32)
    r = oracle.verify(np.broadcast_to(zt1, (N, K + 1, V)),
                      np.broadcast_to(zt1[:K], (N, K, V)), x, u)
    assert (r["accepted_len"] == K).all()
    freq = np.bincount(r["out_tokens"][:, K], minlength=V) / N
    np.testing.assert_allclose(freq, pK, atol=1.5 / N)
    # brute force: the token is the interval of the cumulative sum that holds u
    cum = np.cumsum(pK)
    expect = np.searchsorted(cum, uu.astype(np.float32).astype(np.float64), side="right")
    assert (r["out_tokens"][:, K] == expect).all()


def test_residual_inverse_cdf_brute_force():
    # forced rejection at position 0; the correction follows norm(max(0, p - q))
    rng = np.random.default_rng(5)
    for V in (3, 7, 16):
        zt1 = rng.normal(0, 1.5, (2, V)).astype(np.float32)
        zd1 = rng.normal(0, 1.5, (1, V)).astype(np.float32)
        p, q = _softmax64(zt1[0]), _softmax64(zd1[0])
        xr = int(np.argmin(p / q))                    # a token with p/q < 1
        assert p[xr] / q[xr] < 0.99
        N = 20000
        uu = (np.arange(N) + 0.5) / N
        u = np.stack([np.full(N, 0.999999), uu], 1).astype(np.float32)
        r = oracle.verify(np.broadcast_to(zt1, (N, 2, V)), np.broadcast_to(zd1, (N, 1, V)),
                          np.full((N, 1), xr, np.int32), u)
        assert (r["accepted_len"] == 0).all()
        res = np.maximum(p - q, 0.0)
        Z = res.sum()
        cum = np.cumsum(res)
        expect = np.array([np.flatnonzero(cum > t * Z)[0] for t in u[:, 1].astype(np.float64)])
        assert (r["out_tokens"][:, 0] == expect).all()
        freq = np.bincount(r["out_tokens"][:, 0], minlength=V) / N
        np.testing.assert_allclose(freq, res / Z, atol=1.5 / N)
        assert (freq[res == 0] == 0).all()


def test_uniform_at_exact_boundary_takes_next_token():
    # strict '>' on the running sum: u*Z equal to a boundary selects the next token
    zt = np.zeros((1, 2, 4), np.float32)              # exact uniform rows, p = q
    for uK, expect in [(0.0, 0), (0.25, 1), (0.5, 2), (0.75, 3), (0.9999, 3)]:
        r = oracle.verify(zt, zt[:, :1].copy(), np.zeros((1, 1), np.int32),
                          np.array([[0.0, uK]], np.float32))
        assert r["accepted_len"][0] == 1 and r["out_tokens"][0, 1] == expect
        if uK in (0.25, 0.5, 0.75):
            assert r["margin"][0] == 0.0               # boundary cases are flagged


# ---------------------------------------------------------------------------
# Greedy exact match ("Training-Free Loosely Speculative Decoding", section 1;
# "Speculative Decoding: ...", "Проверка результата").
# ---------------------------------------------------------------------------

def test_greedy_is_argmax_match_with_ties():
    rng = np.random.default_rng(3)
    B, K, V = 200, 6, 50
    # coarse values make ties frequent; bf16 storage
    zt = rng.integers(-3, 4, (B, K + 1, V)).astype(np.float32)
    import torch
    ztb = torch.from_numpy(zt).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    am = zt.argmax(-1)                                # numpy: first maximal index
    x = np.where(rng.random((B, K)) < 0.8, am[:, :K], rng.integers(0, V, (B, K))).astype(np.int32)
    r = oracle.verify(ztb, None, x, None, mode=oracle.GREEDY)
    for b in range(B):
        mism = np.flatnonzero(x[b] != am[b, :K])
        n = mism[0] if len(mism) else K
        assert r["accepted_len"][b] == n
        assert (r["out_tokens"][b, :n] == x[b, :n]).all()
        assert r["out_tokens"][b, n] == am[b, n]
        assert (r["out_tokens"][b, n + 1:] == -1).all()


# ---------------------------------------------------------------------------
# Row statistics against library routines and closed forms.
# ---------------------------------------------------------------------------

def test_row_stats_against_scipy():
    rng = np.random.default_rng(9)
    z = rng.normal(0, 3, (40, 777)).astype(np.float32)
    z[3, ::5] = -np.inf                               # masked logits
    lse, h, am, fq = oracle.row_stats(z)
    z64 = z.astype(np.float64)
    np.testing.assert_allclose(lse, special.logsumexp(z64, axis=-1), rtol=1e-13)
    p = _softmax64(z64)
    np.testing.assert_allclose(h, stats.entropy(p, axis=-1) / np.log(777), rtol=1e-12)
    assert (am == z.argmax(-1)).all()
    pm = p.max(-1)
    np.testing.assert_allclose(fq, special.logit(pm), rtol=1e-9)


def test_entropy_closed_forms():
    V = 64
    uni = np.zeros((1, V), np.float32)
    onehot = np.full((1, V), -np.inf, np.float32)
    onehot[0, 17] = 2.0
    _, h, am, _ = oracle.row_stats(np.concatenate([uni, onehot]))
    np.testing.assert_allclose(h[0], 1.0, rtol=1e-14)
    assert h[1] == 0.0 and am[1] == 17
    for a in (0.5, 0.1, 0.9, 1e-4):
        _, h2, _, f2 = oracle.row_stats(_rows([[a, 1 - a]]))
        z = _rows([[a, 1 - a]]).astype(np.float64)
        pa = 1.0 / (1.0 + np.exp(z[0, 1] - z[0, 0]))  # exact softmax of the stored values
        H = -(pa * np.log(pa) + (1 - pa) * np.log(1 - pa)) / np.log(2)
        np.testing.assert_allclose(h2[0], H, rtol=1e-12)
        # logit(q_max) of a two-token row: ln(q_max / (1 - q_max))
        qm = max(pa, 1 - pa)
        np.testing.assert_allclose(f2[0], np.log(qm / (1 - qm)), rtol=1e-12, atol=1e-15)


def test_logit_qmax_clamps_when_complement_vanishes():
    z = np.full((1, 8), -np.inf, np.float32)
    z[0, 2] = 0.0
    _, _, _, fq = oracle.row_stats(z)
    assert fq[0] == 30.0


@pytest.mark.parametrize("gap", [5.0, 29.5, 30.5, 100.0, 800.0])
def test_logit_qmax_is_capped_at_30(gap):
    # a two-token row (0, -gap): q_max / (1 - q_max) = e^gap exactly, so
    # logit(q_max) = gap; the reading caps it at 30 (and flags the cap)
    z = np.array([[0.0, -gap]], np.float32)
    _, _, _, fq = oracle.row_stats(z)
    assert abs(fq[0] - min(gap, 30.0)) < 1e-9


def test_log_ratio_matches_logsumexp():
    rng = np.random.default_rng(21)
    B, K, V = 8, 3, 500
    zt = rng.normal(0, 3, (B, K + 1, V)).astype(np.float32)
    zd = (zt[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1), dtype=np.float32)
    r = oracle.verify(zt, zd, x, u)
    t64, d64 = zt.astype(np.float64), zd.astype(np.float64)
    lp = np.take_along_axis(t64[:, :K], x[..., None], 2)[..., 0] - special.logsumexp(t64[:, :K], axis=-1)
    lq = np.take_along_axis(d64, x[..., None], 2)[..., 0] - special.logsumexp(d64, axis=-1)
    np.testing.assert_allclose(r["pos_stats"][:, :K, 2], lp - lq, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(r["pos_stats"][:, :, 0], special.logsumexp(t64, axis=-1), rtol=1e-13)
    assert np.isnan(r["pos_stats"][:, K, 2:]).all()
    # accept decisions against the rule u < min(1, p/q), first rejection stops
    for b in range(B):
        ok = u[b, :K] < np.minimum(1.0, np.exp(lp[b] - lq[b]))
        n = K if ok.all() else int(np.argmin(ok))
        assert r["accepted_len"][b] == n


# ---------------------------------------------------------------------------
# Acceptance estimator ("Verificación Adaptativa sin una cabeza de confianza").
# ---------------------------------------------------------------------------

def test_confidence_is_sigmoid_of_affine_feature():
    rng = np.random.default_rng(4)
    B, K, V = 16, 4, 200
    zd = rng.normal(0, 2, (B, K, V)).astype(np.float32)
    zt = np.concatenate([zd, rng.normal(0, 2, (B, 1, V)).astype(np.float32)], 1)
    est = np.array([0.53, 0.4, 0.1, -0.2, -0.5])
    feat, conf, _ = oracle.confidence(zd, est)
    q = _softmax64(zd.astype(np.float64))
    np.testing.assert_allclose(feat, special.logit(q.max(-1)), rtol=1e-9)
    np.testing.assert_allclose(conf, special.expit(est[0] * feat + est[1:][None, :]), rtol=1e-13)
    r = oracle.verify(zt, zd, np.zeros((B, K), np.int32), rng.random((B, K + 1), dtype=np.float32),
                      est_params=est)
    np.testing.assert_allclose(r["feature"], feat, rtol=1e-14)
    np.testing.assert_allclose(r["conf"], conf, rtol=1e-14)


def test_estimator_hand_cases():
    g = json.load(open(os.path.join(GOLDEN, "estimator_hand_cases.json")))
    for c in g["cases"]:
        K = c["K"]
        f = np.array(c["feature"], np.float64).reshape(-1, K)
        n = np.array(c["accepted_len"], np.int32)
        newp, grad, cnt = oracle.estimator_update(f, n, c["params"], c["lr"])
        np.testing.assert_allclose(grad, c["grad"], atol=1e-15)
        assert list(cnt) == c["counts"]
        np.testing.assert_allclose(newp, c["new_params"], atol=1e-15)


def test_estimator_loss_and_gradient_by_finite_differences():
    assert abs(oracle.estimator_loss(np.zeros((1, 1)), np.array([1], np.int32), [0.0, 0.0])
               - np.log(2.0)) < 1e-15
    rng = np.random.default_rng(8)
    B, K = 50, 6
    f = rng.normal(-2, 1.5, (B, K))
    n = rng.integers(0, K + 1, B).astype(np.int32)
    params = rng.normal(0, 0.5, K + 1)
    _, grad, _ = oracle.estimator_update(f, n, params, 0.0)
    eps = 1e-6
    for k in range(K + 1):
        dp = np.zeros(K + 1)
        dp[k] = eps
        fd = (oracle.estimator_loss(f, n, params + dp) - oracle.estimator_loss(f, n, params - dp)) / (2 * eps)
        assert abs(fd - grad[k]) < 1e-8
    # a small step lowers the loss
    newp, _, _ = oracle.estimator_update(f, n, params, 0.05)
    assert oracle.estimator_loss(f, n, newp) < oracle.estimator_loss(f, n, params)


# ---------------------------------------------------------------------------
# FLy entropy gate and deferral window ("Training-Free Loosely Speculative
# Decoding", 2.A.1 and 2.A.2). Exhaustive over deviation patterns and gate bits.
# ---------------------------------------------------------------------------

def _fly_truth(d, gate_open, W):
    """n_acc from the rule as stated: the first deviation that is not excused.
    A deviation at j is excused only if the target is uncertain there, the next
    W draft positions exist, and none of them deviates."""
    K = len(d)
    for j in range(K):
        if not d[j]:
            continue
        excused = gate_open[j] and (j + W <= K - 1) and not any(d[j + 1:j + W + 1])
        if not excused:
            return j
    return K


@pytest.mark.parametrize("K", [1, 2, 3, 5, 6])
def test_fly_truth_table_exhaustive(K):
    V = 16
    theta = 0.3
    hi = np.zeros(V, np.float32)
    lo = np.full(V, -20.0, np.float32)
    cases = []
    for W in range(1, K + 2):
        for dbits in range(1 << K):
            for gbits in range(1 << K):
                if gbits & ~dbits:
                    continue                            # gate bits only matter at deviations
                cases.append((W, dbits, gbits))
    B = len(cases)
    zt = np.empty((B, K + 1, V), np.float32)
    x = np.empty((B, K), np.int32)
    expect_n = np.empty(B, np.int32)
    Ws = np.empty(B, np.int32)
    for b, (W, dbits, gbits) in enumerate(cases):
        d = [(dbits >> j) & 1 for j in range(K)]
        gate = [(gbits >> j) & 1 for j in range(K)]
        for j in range(K + 1):
            a = (3 * j + 1) % V                        # target argmax of row j
            row = (hi if (j < K and gate[j]) else lo).copy()
            row[a] = 0.05 if (j < K and gate[j]) else 0.0
            zt[b, j] = row
            if j < K:
                x[b, j] = (a + 1) % V if d[j] else a
        expect_n[b] = _fly_truth(d, gate, W)
        Ws[b] = W
    for W in range(1, K + 2):
        sel = Ws == W
        r = oracle.verify(zt[sel], None, x[sel], None, mode=oracle.FLY, fly_theta=theta, fly_window=W)
        n = r["accepted_len"]
        assert (n == expect_n[sel]).all()
        idx = np.arange(sel.sum())
        assert (r["out_tokens"][idx, n] == (3 * n + 1) % V).all()
        for i in np.flatnonzero(n > 0)[:50]:
            assert (r["out_tokens"][i, :n[i]] == x[sel][i, :n[i]]).all()
    # sanity of the row construction: gate-open rows are near-uniform, closed rows peaked
    peaked = lo.copy()
    peaked[1] = 0.0
    _, h, _, _ = oracle.row_stats(np.stack([hi + np.eye(V, dtype=np.float32)[1] * 0.05, peaked]))
    assert h[0] > 0.99 and h[1] < 1e-6


def test_fly_with_a_closed_gate_is_greedy():
    """Normalised entropy never exceeds 1, so at theta > 1 no deviation is
    deferred and FLy reduces to greedy exact match, whatever the window."""
    rng = np.random.default_rng(23)
    B, K, V = 64, 5, 32
    zt = rng.normal(0, 1.5, (B, K + 1, V)).astype(np.float32)
    am = zt.argmax(-1)
    # drafts that match the target's argmax often, so prefixes of every length occur
    x = np.where(rng.random((B, K)) < 0.7, am[:, :K], rng.integers(0, V, (B, K))).astype(np.int32)
    g = oracle.verify(zt, None, x, None, mode=oracle.GREEDY)
    for W in (1, 2, 4):
        f = oracle.verify(zt, None, x, None, mode=oracle.FLY, fly_theta=1.5, fly_window=W)
        np.testing.assert_array_equal(f["accepted_len"], g["accepted_len"])
        np.testing.assert_array_equal(f["out_tokens"], g["out_tokens"])
    assert len(np.unique(g["accepted_len"])) >= 4


def test_fly_gate_tie_defers():
    # h == theta defers (the gate reads h_j >= theta). A two-token uniform row
    # has normalised entropy exactly 1 in fp64; theta = 1 puts it on the tie.
    V, K = 2, 3
    zt = np.zeros((1, K + 1, V), np.float32)
    _, h, am, _ = oracle.row_stats(zt[0])
    assert (h == 1.0).all() and (am == 0).all()
    x = np.array([[1, 0, 0]], np.int32)               # deviation at 0, matches after
    r = oracle.verify(zt, None, x, None, mode=oracle.FLY, fly_theta=1.0, fly_window=2)
    assert r["accepted_len"][0] == 3 and r["margin"][0] == 0.0
    zt[0, 0, 0] = 1e-3                                # h just below theta: rejected
    r = oracle.verify(zt, None, x, None, mode=oracle.FLY, fly_theta=1.0, fly_window=2)
    assert r["accepted_len"][0] == 0 and r["out_tokens"][0, 0] == 0


def test_cdf_output_brackets_every_draw():
    # the normalised running sum the oracle reports for its final draw ends at 1
    # and u[b, K] falls inside the drawn token's interval
    rng = np.random.default_rng(17)
    B, K, V = 300, 3, 40
    zt = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    zd = (zt[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1), dtype=np.float32)
    r = oracle.verify(zt, zd, x, u, want_cdf=True)
    c = r["cdf"]
    np.testing.assert_allclose(c[:, -1], 1.0, rtol=1e-13)
    assert (np.diff(c, axis=1) >= 0).all()
    for b in range(B):
        v = r["out_tokens"][b, r["accepted_len"][b]]
        lo = c[b, v - 1] if v > 0 else 0.0
        assert lo <= u[b, K] < c[b, v]
        assert r["margin_cdf"][b] == min(u[b, K] - lo, c[b, v] - u[b, K]) or abs(
            r["margin_cdf"][b] - min(u[b, K] - lo, c[b, v] - u[b, K])) < 1e-12
    assert np.isinf(oracle.verify(zt, None, x, None, mode=oracle.GREEDY)["margin_cdf"]).all()
