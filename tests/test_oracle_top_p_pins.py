"""Pins of the oracle's top-p (nucleus) processed verification.

"Verificación Adaptativa sin una cabeza de confianza", "Benchmarks": serving
samples with top-p 0.95; "Speculative Decoding: ...", "Математика
верификации": the rule is lossless for the processed p and q. Reading: the
nucleus keeps every token whose logit is at least z*, the largest logit
value whose upper mass reaches top_p (ties at z* all kept). Pinned by closed
forms, the tie rule, an independent nucleus built on numpy's argsort and
cumsum, the tiny-top_p limit (greedy), and a Monte Carlo chi-square of the
emitted token. CPU only.
"""
import numpy as np
import pytest
from scipy import special, stats

import oracle


def _ref_nucleus(z, s, top_p):
    """Independent nucleus of one row: (mask, lse of the processed row, margin)."""
    z = z.astype(np.float64)
    p = special.softmax(s * z)
    order = np.argsort(-z, kind="stable")
    cum = np.cumsum(p[order])
    k = int(np.searchsorted(cum, top_p - 1e-300, side="left"))   # first cum >= top_p
    k = min(k, len(z) - 1)
    zs = z[order[k]]
    mask = z >= zs
    above = p[z > zs].sum()
    margin = min(p[mask].sum() - top_p, top_p - above)
    lse = special.logsumexp(s * z[mask])
    return mask, lse, margin


def _one_step(zt, zd, x, u, **kw):
    return oracle.verify(zt[None], zd[None], np.array([x], np.int32), np.array([u], np.float32), **kw)


def test_top_p_one_is_the_default():
    rng = np.random.default_rng(1)
    zt = rng.normal(0, 2, (6, 5, 40)).astype(np.float32)
    zd = (zt[:, :4] + rng.normal(0, 1, (6, 4, 40))).astype(np.float32)
    x = rng.integers(0, 40, (6, 4)).astype(np.int32)
    u = rng.random((6, 5)).astype(np.float32)
    a = oracle.verify(zt, zd, x, u, est_params=np.ones(5))
    b = oracle.verify(zt, zd, x, u, est_params=np.ones(5), top_p=1.0)
    for k in ("out_tokens", "accepted_len", "pos_stats", "feature", "flags"):
        np.testing.assert_array_equal(a[k], b[k])


def test_closed_form_four_tokens():
    # p = (.5, .3, .15, .05): top_p .7 keeps {0, 1}, renormalised (.625, .375)
    pr = np.array([0.5, 0.3, 0.15, 0.05])
    row = np.log(pr).astype(np.float32)
    zt = np.stack([row, row])                 # target rows 0 and 1 (bonus row)
    zd = row[None]
    r = _one_step(zt, zd, [0], [0.1, 0.9], top_p=0.7, est_params=[1.0, 0.0])
    pf = special.softmax(row.astype(np.float64))
    keep = pf[:2].sum()
    assert r["accepted_len"][0] == 1          # x = 0 with p' = q': accepted
    assert r["out_tokens"][0, 1] == 1         # u = .9 falls in token 1 of p' = (.625, .375)
    lse = special.logsumexp(row.astype(np.float64)) + np.log(keep)
    np.testing.assert_allclose(r["pos_stats"][0, 0, 0], lse, rtol=1e-14)
    pp = pf[:2] / keep
    np.testing.assert_allclose(r["pos_stats"][0, 0, 1], -(pp * np.log(pp)).sum() / np.log(4), rtol=1e-13)
    np.testing.assert_allclose(r["feature"][0, 0], np.log(pp[0] / pp[1]), rtol=1e-13)
    # without top-p the same u draws token 2 (cumulative .5, .8, .95)
    r1 = _one_step(zt, zd, [0], [0.1, 0.9], est_params=[1.0, 0.0])
    assert r1["out_tokens"][0, 1] == 2


def test_ties_at_the_boundary_are_all_kept():
    row = np.array([1.0, 1.0, 1.0, 0.0, -1.0], np.float32)
    zt = np.stack([row, row])
    zd = row[None]
    # the three tied tokens hold 3e/(3e + 1 + 1/e) = .85 > top_p = .4
    draws = []
    for uu in (0.05, 0.2, 0.45, 0.7, 0.95):
        r = _one_step(zt, zd, [0], [0.0, uu], top_p=0.4)
        draws.append(int(r["out_tokens"][0, 1]))
        np.testing.assert_allclose(r["pos_stats"][0, 1, 0], np.log(3 * np.e), rtol=1e-14)
    assert set(draws) == {0, 1, 2}


@pytest.mark.parametrize("seed", range(5))
def test_against_an_independent_nucleus(seed):
    rng = np.random.default_rng(100 + seed)
    B, K, V = 12, 3, 300
    # a coarse grid of logit values gives many ties
    zt = (np.round(rng.normal(0, 2, (B, K + 1, V)) * 4) / 4).astype(np.float32)
    zd = (np.round((zt[:, :K] + rng.normal(0, 1, (B, K, V))) * 4) / 4).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    s = np.exp(rng.uniform(np.log(0.5), np.log(2.0), B)).astype(np.float32)
    top_p = float(rng.uniform(0.3, 0.97))
    r = oracle.verify(zt, zd, x, None, mode=oracle.GREEDY, inv_temp=s, top_p=top_p, est_params=np.ones(K + 1))
    for b in range(B):
        for j in range(K + 1):
            mask, lse, m = _ref_nucleus(zt[b, j], float(s[b]), top_p)
            if m < 1e-12:
                continue
            np.testing.assert_allclose(r["pos_stats"][b, j, 0], lse, rtol=1e-13)
            pz = special.softmax(float(s[b]) * zt[b, j].astype(np.float64)[mask])
            h = -(pz * np.log(pz)).sum() / np.log(V)
            np.testing.assert_allclose(r["pos_stats"][b, j, 1], h, rtol=1e-11, atol=1e-14)
            if j < K:
                md, lsed, md_m = _ref_nucleus(zd[b, j], float(s[b]), top_p)
                if md_m < 1e-12:
                    continue
                sb = float(s[b])
                lp = sb * float(zt[b, j, x[b, j]]) - lse if mask[x[b, j]] else -np.inf
                lq = sb * float(zd[b, j, x[b, j]]) - lsed if md[x[b, j]] else -np.inf
                want = lp - lq
                got = r["pos_stats"][b, j, 2]
                if np.isnan(want):
                    assert np.isnan(got)
                elif np.isinf(want):
                    assert got == want
                else:
                    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_token_outside_the_target_nucleus_is_rejected():
    rng = np.random.default_rng(7)
    V = 64
    row = rng.normal(0, 3, V).astype(np.float32)
    mask, _, _ = _ref_nucleus(row, 1.0, 0.5)
    out = int(np.flatnonzero(~mask)[0])
    zt = np.stack([row, row])
    zd = np.zeros((1, V), np.float32)         # uniform draft: every token in its nucleus
    for uu in (0.0, 0.3, 0.999):
        r = _one_step(zt, zd, [out], [uu, 0.5], top_p=0.5)
        assert r["accepted_len"][0] == 0
        assert mask[r["out_tokens"][0, 0]]    # the correction comes from the nucleus
        assert r["pos_stats"][0, 0, 2] == -np.inf


def test_tiny_top_p_is_greedy():
    rng = np.random.default_rng(9)
    B, K, V = 64, 4, 50
    zt = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    zd = (zt[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
    x = zd.argmax(-1).astype(np.int32)        # the only draft in the draft's nucleus
    u = rng.random((B, K + 1)).astype(np.float32)
    s = oracle.verify(zt, zd, x, u, top_p=1e-9)
    g = oracle.verify(zt, zd, x, None, mode=oracle.GREEDY)
    np.testing.assert_array_equal(s["accepted_len"], g["accepted_len"])
    np.testing.assert_array_equal(s["out_tokens"], g["out_tokens"])


def test_knife_edge_boundary_is_flagged():
    pr = np.array([0.5, 0.3, 0.2])
    row = np.log(pr).astype(np.float32)
    pf = special.softmax(row.astype(np.float64))
    zt = np.stack([row, row])
    # top_p just above the first token's mass: the second token (mass .3,
    # far above the benign size) may be dropped by a slightly different sum
    r = _one_step(zt, row[None], [0], [0.0, 0.5], top_p=float(pf[0] * (1 + 1e-7)))
    assert r["margin_acc"][0] < 1e-5
    # top_p just below the first token's mass: the second may be added
    r = _one_step(zt, row[None], [0], [0.0, 0.5], top_p=float(pf[0] * (1 - 1e-7)))
    assert r["margin_acc"][0] < 1e-5
    # nothing above the argmax: dropping it is impossible, nothing is in doubt
    r = _one_step(zt, row[None], [0], [0.0, 0.5], top_p=1e-9)
    assert r["margin_acc"][0] > 1e-3


def test_benign_boundary_is_not_flagged_but_a_draft_in_it_is():
    # a long tail of tiny tied tokens: the group (all 3996 of them, 2.5e-8 of
    # the mass) is below the benign size, so a boundary in doubt there is not
    # flagged ...
    V = 4000
    row = np.full(V, -25.0, np.float32)
    row[:4] = [0.0, -0.5, -1.0, -1.5]
    pf = special.softmax(row.astype(np.float64))
    top_p = float(pf[:4].sum() + 0.5 * pf[4])           # inside the tied tail group
    zt = np.stack([row, row])
    r = _one_step(zt, row[None], [0], [0.0, 0.5], top_p=top_p)
    assert r["margin_acc"][0] > 1e-3
    # ... a group of 4 tokens of mass 1.5e-4 each is not benign
    row2 = row.copy()
    row2[4:8] = -8.0
    pf2 = special.softmax(row2.astype(np.float64))
    tp2 = float(pf2[:4].sum() * (1 + 1e-8))              # the group at -8 is the boundary, in doubt
    r = _one_step(np.stack([row2, row2]), row2[None], [0], [0.0, 0.5], top_p=tp2)
    assert r["margin_acc"][0] < 1e-5
    # ... and a draft token in a group in doubt flags the sequence
    r = _one_step(np.stack([row2, row2]), row2[None], [5], [0.0, 0.5], top_p=tp2)
    assert r["margin_acc"][0] == 0.0


def test_lossless_under_top_p():
    rng = np.random.default_rng(5)
    V, K, B, reps, tp = 6, 2, 20000, 10, 0.8
    pt = np.log(np.array([[0.3, 0.25, 0.2, 0.12, 0.08, 0.05], [0.1, 0.4, 0.2, 0.1, 0.1, 0.1],
                          [1 / 6] * 6]))
    pd = np.log(np.array([[0.2, 0.3, 0.1, 0.25, 0.1, 0.05], [0.3, 0.2, 0.2, 0.1, 0.1, 0.1]]))
    zt = np.broadcast_to(pt.astype(np.float32), (B, K + 1, V)).copy()
    zd = np.broadcast_to(pd.astype(np.float32), (B, K, V)).copy()
    qn = []
    for i in range(K):
        m, _, _ = _ref_nucleus(zd[0, i], 1.0, tp)
        qq = special.softmax(zd[0, i].astype(np.float64)) * m
        qn.append(qq / qq.sum())
    qn = np.array(qn)
    counts = np.zeros(V)
    for _ in range(reps):
        x = (qn.cumsum(-1)[None] > rng.random((B, K, 1))).argmax(-1).astype(np.int32)
        u = rng.random((B, K + 1)).astype(np.float32)
        r = oracle.verify(zt, zd, x, u, top_p=tp)
        counts += np.bincount(r["out_tokens"][:, 0], minlength=V)
    m0, _, _ = _ref_nucleus(zt[0, 0], 1.0, tp)
    p0 = special.softmax(zt[0, 0].astype(np.float64)) * m0
    p0 /= p0.sum()
    nz = p0 > 0
    assert counts[~nz].sum() == 0
    _, pval = stats.chisquare(counts[nz], p0[nz] * counts.sum())
    assert pval > 1e-3, (counts / counts.sum(), p0, pval)
