"""Pins of the oracle's temperature-processed verification.

"Verificación Adaptativa sin una cabeza de confianza", "Benchmarks": the pages
serve at a sampling temperature; speculative sampling stays lossless for the
processed distributions p = softmax(z/T), q = softmax(y/T) ("Speculative
Decoding: ...", "Математика верификации"). Pinned by exact rescaling (an
inverse temperature of 2^k equals logits scaled by 2^k, exactly representable
in fp32), the low-temperature limit (stochastic becomes greedy), and a Monte
Carlo chi-square of the emitted token against softmax(z/T). CPU only.
"""
import numpy as np
import pytest
from scipy import special, stats

import oracle


def _problem(seed, B=8, K=4, V=48):
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    zd = (zt[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    return zt, zd, x, u


def _same(a, b):
    for k in ("out_tokens", "accepted_len", "flags"):
        np.testing.assert_array_equal(a[k], b[k])
    for k in ("pos_stats", "feature", "conf", "margin_acc", "margin_cdf"):
        np.testing.assert_array_equal(a[k], b[k])


@pytest.mark.parametrize("mode", [oracle.STOCHASTIC, oracle.GREEDY, oracle.FLY])
def test_unit_temperature_is_the_default(mode):
    zt, zd, x, u = _problem(1)
    kw = dict(mode=mode, fly_theta=0.5, fly_window=1, est_params=np.linspace(0.5, 1.5, 5))
    _same(oracle.verify(zt, zd, x, u, **kw), oracle.verify(zt, zd, x, u, inv_temp=np.ones(8, np.float32), **kw))


@pytest.mark.parametrize("s", [2.0, 0.5, 4.0])
@pytest.mark.parametrize("mode", [oracle.STOCHASTIC, oracle.GREEDY, oracle.FLY])
def test_power_of_two_temperature_equals_scaled_logits(s, mode):
    zt, zd, x, u = _problem(2)
    kw = dict(mode=mode, fly_theta=0.5, fly_window=1, est_params=np.linspace(0.5, 1.5, 5))
    a = oracle.verify(zt, zd, x, u, inv_temp=np.full(8, s, np.float32), **kw)
    b = oracle.verify((zt * np.float32(s)).astype(np.float32), (zd * np.float32(s)).astype(np.float32), x, u, **kw)
    _same(a, b)


def test_per_sequence_temperatures_apply_per_sequence():
    zt, zd, x, u = _problem(3)
    it = np.array([1, 2, 0.5, 4, 1, 0.25, 2, 8], np.float32)
    a = oracle.verify(zt, zd, x, u, inv_temp=it)
    for b in range(8):
        r = oracle.verify(zt[b:b + 1] * it[b], zd[b:b + 1] * it[b], x[b:b + 1], u[b:b + 1])
        np.testing.assert_array_equal(a["out_tokens"][b], r["out_tokens"][0])
        np.testing.assert_array_equal(a["pos_stats"][b], r["pos_stats"][0])


def test_low_temperature_is_greedy():
    rng = np.random.default_rng(4)
    B, K, V = 64, 4, 32
    zt = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    zd = (zt[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
    # as T -> 0 the draft's sample is its argmax; off-distribution drafts have
    # no greedy limit (a draft token that both models give ~0 mass leaves a
    # residual on the target's tail)
    x = zd.argmax(-1).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    s = oracle.verify(zt, zd, x, u, inv_temp=np.full(B, 1e4, np.float32))
    g = oracle.verify(zt, zd, x, None, mode=oracle.GREEDY)
    np.testing.assert_array_equal(s["accepted_len"], g["accepted_len"])
    np.testing.assert_array_equal(s["out_tokens"], g["out_tokens"])


def test_lossless_at_a_temperature():
    rng = np.random.default_rng(5)
    V, K, B, reps, it = 5, 2, 20000, 10, 0.6
    pt = np.log(np.array([[0.1, 0.2, 0.3, 0.25, 0.15], [0.3, 0.1, 0.2, 0.2, 0.2], [0.2] * 5]))
    pd = np.log(np.array([[0.3, 0.3, 0.1, 0.2, 0.1], [0.1, 0.4, 0.2, 0.2, 0.1]]))
    zt = np.broadcast_to(pt.astype(np.float32), (B, K + 1, V)).copy()
    zd = np.broadcast_to(pd.astype(np.float32), (B, K, V)).copy()
    q = special.softmax(pd * it, axis=-1)
    counts = np.zeros(V)
    for _ in range(reps):
        x = (q.cumsum(-1)[None] > rng.random((B, K, 1))).argmax(-1).astype(np.int32)   # drafts from the processed q
        u = rng.random((B, K + 1)).astype(np.float32)
        r = oracle.verify(zt, zd, x, u, inv_temp=np.full(B, it, np.float32))
        counts += np.bincount(r["out_tokens"][:, 0], minlength=V)
    p0 = special.softmax(pt[0] * it)
    _, pval = stats.chisquare(counts, p0 * counts.sum())
    assert pval > 1e-3, (counts / counts.sum(), p0, pval)
