"""The parity checker itself (tests/helpers.py compare()), on the CPU.

The "GPU" results here are stand-ins built from the oracle: its own outputs,
and its outputs along other decision paths (imposed decisions, a nucleus
boundary moved one tie group), with planted mistakes. The checker must
accept a result that differs from the oracle's only at decisions within the
flag margin ("Speculative Decoding: ...", "Математика верификации": accept
iff u < min(1, p/q); "Training-Free Loosely Speculative Decoding", 2.A.1:
h >= theta), and reject everything else: a decision flipped outside the
margin, a wrong final token, an unwritten (poisoned) output, a float out of
tolerance, a nucleus boundary moved where it is not in doubt. CPU only.
"""
import numpy as np
import pytest
import torch
from scipy import special

import oracle
from helpers import POISON_I32, compare, oracle_run


def _as_gpu(r, keys=("out_tokens", "accepted_len", "pos_stats", "feature", "conf")):
    out = {}
    for k in keys:
        v = r[k]
        out[k] = torch.from_numpy(np.array(v, np.float32 if v.dtype == np.float64 else v.dtype))
    return out


def _stochastic_inputs(seed=0, B=40, K=4, V=50):
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    zd = (zt[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    u = rng.random((B, K + 1), dtype=np.float32)
    return zt, zd, x, u


def _knife_edge(zt, zd, x, u, b, i):
    """Put u[b, i] within 1e-7 of min(1, p/q) at position i, and accept every
    earlier position of sequence b, so that the scan reaches i."""
    p = special.softmax(zt[b, i].astype(np.float64))
    q = special.softmax(zd[b, i].astype(np.float64))
    acc = min(1.0, p[x[b, i]] / q[x[b, i]])
    if acc >= 1.0:                     # make the ratio fall below 1: draft token = argmax q
        x[b, i] = int(np.argmax(q - p))
        acc = min(1.0, p[x[b, i]] / q[x[b, i]])
    u[b, :i] = 0.0
    u[b, i] = np.float32(acc)
    return acc


def _inp(zt, zd, x, u):
    return dict(zt=torch.from_numpy(zt), zd=torch.from_numpy(zd), x=torch.from_numpy(x), u=torch.from_numpy(u))


def test_the_oracle_itself_passes():
    zt, zd, x, u = _stochastic_inputs()
    r = oracle_run(_inp(zt, zd, x, u), oracle.STOCHASTIC, est=np.r_[1.0, np.zeros(4)])
    s = compare(_as_gpu(r), r, "f32", check_feature=True, check_conf=True)
    assert s["differ"] == 0


def test_a_decision_in_doubt_taken_the_other_way_passes():
    zt, zd, x, u = _stochastic_inputs(1)
    b, i = 7, 2
    _knife_edge(zt, zd, x, u, b, i)
    r = oracle_run(_inp(zt, zd, x, u), oracle.STOCHASTIC)
    assert r["margin_pos"][b, i] < 1e-5
    nat = r["natural_pos"][b, i]
    f = np.full_like(x, -1)
    f[b, :i] = 1
    f[b, i] = 1 - nat
    other = oracle.verify(zt, zd, x, u, force=f)
    assert other["accepted_len"][b] != r["accepted_len"][b]
    s = compare(_as_gpu(other, ("out_tokens", "accepted_len", "pos_stats")), r, "f32")
    assert s["differ"] == 1 and s["differ_path"] == 1


def test_a_decision_flipped_outside_the_margin_fails():
    zt, zd, x, u = _stochastic_inputs(2)
    r = oracle_run(_inp(zt, zd, x, u), oracle.STOCHASTIC)
    b = int(np.flatnonzero((r["margin_pos"][:, 0] > 0.05) & (r["natural_pos"][:, 0] == 1))[0])
    f = np.full_like(x, -1)
    f[b, 0] = 0
    other = oracle.verify(zt, zd, x, u, force=f)
    with pytest.raises(AssertionError, match="decided against the rule"):
        compare(_as_gpu(other, ("out_tokens", "accepted_len", "pos_stats")), r, "f32")


def test_a_wrong_final_token_fails():
    zt, zd, x, u = _stochastic_inputs(3)
    r = oracle_run(_inp(zt, zd, x, u), oracle.STOCHASTIC)
    g = _as_gpu(r, ("out_tokens", "accepted_len", "pos_stats"))
    b = int(np.flatnonzero(r["margin_cdf"] > 0.01)[0])
    n = int(r["accepted_len"][b])
    g["out_tokens"][b, n] = (g["out_tokens"][b, n] + 1) % zt.shape[2]
    with pytest.raises(AssertionError, match="final token"):
        compare(g, r, "f32")


@pytest.mark.parametrize("what", ["token", "length", "stat"])
def test_an_unwritten_output_fails(what):
    zt, zd, x, u = _stochastic_inputs(4)
    r = oracle_run(_inp(zt, zd, x, u), oracle.STOCHASTIC)
    g = _as_gpu(r, ("out_tokens", "accepted_len", "pos_stats"))
    if what == "token":
        g["out_tokens"][5, -1] = POISON_I32
    elif what == "length":
        g["accepted_len"][5] = POISON_I32
    else:
        g["pos_stats"][5, 1, 1] = torch.tensor(POISON_I32, dtype=torch.int32).view(torch.float32)
    with pytest.raises(AssertionError):
        compare(g, r, "f32")


def test_a_float_out_of_tolerance_fails():
    zt, zd, x, u = _stochastic_inputs(5)
    r = oracle_run(_inp(zt, zd, x, u), oracle.STOCHASTIC, est=np.r_[1.0, np.zeros(4)])
    g = _as_gpu(r)
    g["conf"][3, 1] *= 1.001          # 1e-3 relative against an fp32 tolerance of 1e-5
    with pytest.raises(AssertionError, match="floats"):
        compare(g, r, "f32", check_conf=True)
    # within the bf16 tolerance it passes
    compare(g, r, "bf16", check_conf=True)


def test_too_many_differing_sequences_fail():
    zt, zd, x, u = _stochastic_inputs(6, B=20)
    f = np.full_like(x, -1)
    for b in range(6):
        _knife_edge(zt, zd, x, u, b, 1)
    r = oracle_run(_inp(zt, zd, x, u), oracle.STOCHASTIC)
    for b in range(6):
        f[b, 0] = 1
        f[b, 1] = 1 - r["natural_pos"][b, 1]
    other = oracle.verify(zt, zd, x, u, force=f)
    g = _as_gpu(other, ("out_tokens", "accepted_len", "pos_stats"))
    with pytest.raises(AssertionError, match="differ from the oracle"):
        compare(g, r, "f32")
    assert compare(g, r, "f32", max_diff=6)["differ"] == 6


def test_fly_gate_in_doubt_taken_the_other_way_passes():
    V, K = 2, 3
    zt = np.zeros((3, K + 1, V), np.float32)       # uniform rows: h = 1 exactly
    x = np.array([[1, 0, 0]] * 3, np.int32)        # a deviation at 0, matches after
    inp = dict(zt=torch.from_numpy(zt), zd=None, x=torch.from_numpy(x), u=None)
    r = oracle_run(inp, oracle.FLY, fly_theta=1.0, fly_window=2, with_draft=False)
    assert (r["accepted_len"] == 3).all() and (r["margin_pos"][:, 0] == 0).all()
    f = np.full_like(x, -1)
    f[1, 0] = 0                                     # "GPU" closed the gate at the tie
    other = oracle.verify(zt, None, x, None, mode=oracle.FLY, fly_theta=1.0, fly_window=2, force=f)
    s = compare(_as_gpu(other, ("out_tokens", "accepted_len", "pos_stats")), r, "f32")
    assert s["differ"] == 1
    # far from the tie the same flip fails
    r2 = oracle_run(inp, oracle.FLY, fly_theta=0.5, fly_window=2, with_draft=False)
    other2 = oracle.verify(zt, None, x, None, mode=oracle.FLY, fly_theta=0.5, fly_window=2, force=f)
    with pytest.raises(AssertionError):
        compare(_as_gpu(other2, ("out_tokens", "accepted_len", "pos_stats")), r2, "f32")


def test_nucleus_boundary_moved_where_in_doubt_passes_elsewhere_fails():
    # p = (.5, .3, .15, .05) rows; top_p at the upper mass of the first two
    # groups puts every row's boundary in doubt downwards (the next group may
    # be added); upwards it is not in doubt
    row = np.log(np.array([0.5, 0.3, 0.15, 0.05])).astype(np.float32)
    pf = special.softmax(row.astype(np.float64))
    B, K = 3, 1
    zt = np.broadcast_to(row, (B, K + 1, 4)).copy()
    zd = np.broadcast_to(row, (B, K, 4)).copy()
    x = np.zeros((B, K), np.int32)
    u = np.full((B, K + 1), 0.3, np.float32)
    inp = _inp(zt, zd, x, u)
    top_p = pf[0] + pf[1]
    r = oracle_run(inp, oracle.STOCHASTIC, top_p=top_p, est=np.r_[1.0, 0.0])
    assert (r["nuc_doubt"] == 2).all()
    ns = np.zeros((B, 2 * K + 1), np.int32)
    ns[1, 0] = 1                                    # target row 0 of sequence 1 one group down
    other = oracle.verify(zt, zd, x, u, top_p=top_p, nuc_shift=ns, est_params=np.r_[1.0, 0.0])
    g = _as_gpu(other)
    s = compare(g, r, "f32", check_feature=True, check_conf=True)
    assert s["differ"] == 1
    ns[1, 0] = -1                                   # one group up: not in doubt
    other = oracle.verify(zt, zd, x, u, top_p=top_p, nuc_shift=ns, est_params=np.r_[1.0, 0.0])
    with pytest.raises(AssertionError, match="nucleus boundary"):
        compare(_as_gpu(other), r, "f32", check_feature=True, check_conf=True)
