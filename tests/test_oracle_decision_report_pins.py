"""Pins of the oracle's per-position decision report and its overrides.

The GPU decides in fp32 and the oracle in fp64, so where a decision of the
rule lies within the flag margin of its threshold the two may go different
ways ("Speculative Decoding: ...", "Математика верификации": accept x_i iff
u_i < min(1, p(x_i)/q(x_i)); "Training-Free Loosely Speculative Decoding",
2.A.1: the gate reads h_j >= theta). To check such a GPU result completely,
the parity tests re-run the oracle with the GPU's decisions imposed at the
positions in doubt, and with a nucleus boundary placed one tie group off
where top-p leaves it in doubt. These pins tie that report and those
overrides to computations written here from scipy and numpy: softmax, the
accept test, the inverse CDF by searchsorted, the FLy window rule as stated,
and a nucleus built on argsort. CPU only.
"""
import numpy as np
import pytest
from scipy import special

import oracle
from test_oracle_pins import _fly_truth


def _softmax64(z):
    z = np.asarray(z, np.float64)
    return np.exp(z - special.logsumexp(z, axis=-1, keepdims=True))


def _draw(w, u):
    """Inverse CDF written independently: the smallest v whose running sum of
    the weights w exceeds u * sum(w)."""
    c = np.cumsum(w)
    return int(np.searchsorted(c, u * c[-1], side="right"))


def _stochastic_batch(seed, B=200, K=4, V=30):
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    zd = (zt[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1), dtype=np.float32)
    return zt, zd, x, u


def test_stochastic_report_against_scipy():
    zt, zd, x, u = _stochastic_batch(1)
    B, K1, V = zt.shape
    K = K1 - 1
    r = oracle.verify(zt, zd, x, u)
    p, q = _softmax64(zt), _softmax64(zd)
    for b in range(B):
        n = K
        for i in range(K):
            acc = min(1.0, p[b, i, x[b, i]] / q[b, i, x[b, i]])
            take = float(u[b, i]) < acc
            assert r["natural_pos"][b, i] == int(take)
            np.testing.assert_allclose(r["margin_pos"][b, i], abs(float(u[b, i]) - acc), rtol=1e-12, atol=1e-15)
            if not take:
                n = i
                break
        assert r["accepted_len"][b] == n
        assert (r["natural_pos"][b, n + 1:] == -1).all() and np.isinf(r["margin_pos"][b, n + 1:]).all()
        assert r["margin_acc"][b] == r["margin_pos"][b, :min(n + 1, K)].min()


def test_imposing_the_rule_changes_nothing():
    zt, zd, x, u = _stochastic_batch(2)
    a = oracle.verify(zt, zd, x, u, est_params=np.r_[1.0, np.zeros(4)], want_cdf=True)
    b = oracle.verify(zt, zd, x, u, est_params=np.r_[1.0, np.zeros(4)], want_cdf=True, force=a["natural_pos"])
    for k in ("out_tokens", "accepted_len", "pos_stats", "feature", "conf", "margin_pos", "natural_pos",
              "margin_acc", "margin_cdf", "cdf"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def test_imposed_acceptance_draws_the_bonus_from_the_last_row():
    zt, zd, x, u = _stochastic_batch(3)
    B, K1, V = zt.shape
    r = oracle.verify(zt, zd, x, u, force=np.ones((B, K1 - 1), np.int32), want_cdf=True)
    assert (r["accepted_len"] == K1 - 1).all()
    p = _softmax64(zt[:, -1])
    for b in range(B):
        assert r["out_tokens"][b, -1] == _draw(p[b], float(u[b, -1]))
        np.testing.assert_allclose(r["cdf"][b], np.cumsum(p[b]) / p[b].sum(), rtol=1e-12)
    # the report still gives the rule's own decisions at every position
    nat = oracle.verify(zt, zd, x, u)
    reached = nat["natural_pos"] >= 0
    np.testing.assert_array_equal(r["natural_pos"][reached], nat["natural_pos"][reached])


@pytest.mark.parametrize("i", [0, 1, 3])
def test_imposed_rejection_draws_the_residual_of_that_row(i):
    zt, zd, x, u = _stochastic_batch(4 + i)
    B, K1, V = zt.shape
    K = K1 - 1
    force = np.full((B, K), -1, np.int32)
    force[:, :i] = 1
    force[:, i] = 0
    r = oracle.verify(zt, zd, x, u, force=force, want_cdf=True)
    assert (r["accepted_len"] == i).all()
    p, q = _softmax64(zt[:, i]), _softmax64(zd[:, i])
    for b in range(B):
        w = np.maximum(p[b] - q[b], 0.0)
        assert r["out_tokens"][b, i] == _draw(w, float(u[b, K]))
        assert (r["out_tokens"][b, :i] == x[b, :i]).all() and (r["out_tokens"][b, i + 1:] == -1).all()


def _fly_batch(seed, B=300, K=6, V=24):
    rng = np.random.default_rng(seed)
    # rows of mixed entropy: some near-uniform, some peaked
    scale = np.where(rng.random((B, K + 1, 1)) < 0.5, 0.3, 4.0)
    zt = (rng.normal(0, 1, (B, K + 1, V)) * scale).astype(np.float32)
    am = zt.argmax(-1)
    x = np.where(rng.random((B, K)) < 0.6, am[:, :K], rng.integers(0, V, (B, K))).astype(np.int32)
    return zt, x


@pytest.mark.parametrize("W", [1, 2, 4])
def test_fly_imposed_gates_follow_the_window_rule(W):
    zt, x = _fly_batch(10 + W)
    B, K1, V = zt.shape
    K = K1 - 1
    am = zt.argmax(-1)
    d = x != am[:, :K]
    for gate in (0, 1):
        r = oracle.verify(zt, None, x, None, mode=oracle.FLY, fly_theta=0.5, fly_window=W,
                          force=np.full((B, K), gate, np.int32))
        for b in range(B):
            n = _fly_truth(list(d[b]), [gate] * K, W)
            assert r["accepted_len"][b] == n
            assert r["out_tokens"][b, n] == am[b, n]


def test_fly_report_against_scipy():
    zt, x = _fly_batch(20)
    B, K1, V = zt.shape
    K = K1 - 1
    theta, W = 0.5, 2
    r = oracle.verify(zt, None, x, None, mode=oracle.FLY, fly_theta=theta, fly_window=W)
    p = _softmax64(zt)
    h = -(p * np.log(p)).sum(-1) / np.log(V)
    am = zt.argmax(-1)
    for b in range(B):
        n = r["accepted_len"][b]
        for j in range(K):
            gated = j <= min(n, K - 1) and x[b, j] != am[b, j]
            if gated:
                assert r["natural_pos"][b, j] == int(h[b, j] >= theta)
                np.testing.assert_allclose(r["margin_pos"][b, j], abs(h[b, j] - theta), rtol=1e-10, atol=1e-14)
            else:
                assert r["natural_pos"][b, j] == -1 and np.isinf(r["margin_pos"][b, j])


# ---------------------------------------------------------------------------
# top-p: which way a boundary is in doubt, and the boundary placed one tie
# group off ("Verificación Adaptativa sin una cabeza de confianza",
# "Benchmarks": serving samples with top-p 0.95)
# ---------------------------------------------------------------------------

def _groups_desc(z):
    return np.unique(z.astype(np.float64))[::-1]


def _nucleus_threshold(z, top_p, shift=0):
    """Independent boundary: distinct logit values in descending order, the
    first whose upper mass reaches top_p, moved by `shift` groups."""
    z = z.astype(np.float64)
    p = _softmax64(z)
    vals = _groups_desc(z)
    k = 0
    while k < len(vals) - 1 and p[z >= vals[k]].sum() < top_p:
        k += 1
    k = min(max(k + shift, 0), len(vals) - 1)
    return vals[k]


@pytest.mark.parametrize("shift", [-1, 0, 1])
def test_nucleus_shift_moves_the_boundary_one_group(shift):
    rng = np.random.default_rng(30)
    B, K, V = 40, 3, 50
    zt = np.round(rng.normal(0, 2, (B, K + 1, V)) * 4).astype(np.float32) / 4   # ties on a 1/4 grid
    zd = (zt[:, :K] + np.round(rng.normal(0, 1, (B, K, V)) * 4) / 4).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1), dtype=np.float32)
    top_p = 0.8
    ns = np.full((B, 2 * K + 1), shift, np.int32)
    r = oracle.verify(zt, zd, x, u, top_p=top_p, nuc_shift=ns, est_params=np.r_[1.0, np.zeros(K)])
    for b in range(B):
        for j in range(K + 1):
            zs = _nucleus_threshold(zt[b, j], top_p, shift)
            m = zt[b, j].astype(np.float64) >= zs
            np.testing.assert_allclose(r["pos_stats"][b, j, 0], special.logsumexp(zt[b, j][m].astype(np.float64)),
                                       rtol=1e-12)
        for j in range(K):
            zs = _nucleus_threshold(zd[b, j], top_p, shift)
            qm = _softmax64(np.where(zd[b, j] >= zs, zd[b, j].astype(np.float64), -np.inf))
            a = int(np.argmax(qm))
            f = np.log(qm[a]) - np.log(qm.sum() - qm[a]) if qm.sum() - qm[a] > 0 else 30.0
            np.testing.assert_allclose(r["feature"][b, j], min(f, 30.0), rtol=1e-9)


def test_nucleus_doubt_bits():
    # p = (.5, .3, .15, .05) as fp32 logits; masses in fp64 of those logits
    row = np.log(np.array([0.5, 0.3, 0.15, 0.05])).astype(np.float32)
    pf = _softmax64(row)
    zt = np.stack([row, row])[None]
    zd = row[None, None]
    x = np.array([[3]], np.int32)         # a draft token outside every group in doubt
    u = np.array([[0.5, 0.5]], np.float32)

    def doubt(top_p):
        return oracle.verify(zt, zd, x, u, top_p=top_p)["nuc_doubt"][0]

    # top_p at the upper mass of the first two groups: the next group down may be added
    assert (doubt(pf[0] + pf[1]) == 2).all()
    # top_p just above the first group's mass: the group at z* may be dropped
    assert (doubt(pf[0] * (1 + 1e-7)) == 1).all()
    # far from any boundary: no doubt
    assert (doubt(0.7) == 0).all()
