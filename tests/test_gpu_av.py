"""GPU parity of adaptive-verification pruning (spec_av_budget), pruned
(ragged) verification and the pruned label rule, against the fp64 oracle.

"Verificación Adaptativa sin una cabeza de confianza": AV verifies a subset of
the drafts; survival is the running product of the confidences, ranked over
the batch; the budget maximises expected emitted tokens per measured cost.

Tolerances: none for the budget. Survival is an fp32 running product on both
sides, the top-k sums are exact fixed-point integers, and the ratio's steps
are correctly rounded fp32 operations, so survival, the objective, the budget
and the draft lengths are compared bit for bit. Ragged verification uses the parity contract of the
unpruned pass (tests/helpers.py); the pruned labels are exact counts and the
estimator/IRLS tolerances of their own tests.
"""
import numpy as np
import pytest

import oracle
import workloads
from helpers import compare, oracle_run
import helpers as hv

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _sv():
    import speculative_decoding_token_verify_gb300 as sv
    sv.build()
    return sv


def _costs(rng, N, B):
    dc = (0.05 * np.arange(N + 1) / max(B, 1)).astype(np.float32)
    vc = (1.0 + rng.uniform(0.1, 0.5) / max(B, 1) * np.arange(N + 1)).astype(np.float32)
    return dc, vc


def _budget_case(sv, conf, dc, vc):
    t = lambda a: torch.tensor(a, device=DEV)
    g = sv.av_budget(t(conf), t(dc), t(vc), want_survival=True, want_objective=True)
    torch.cuda.synchronize()
    r = oracle.av_budget(conf, dc, vc)
    np.testing.assert_array_equal(g["survival"].cpu().numpy(), r["survival"])
    # every step of the decision is exact or correctly rounded on both sides
    np.testing.assert_array_equal(g["objective"].cpu().numpy(), r["objective"])
    assert int(g["budget"].item()) == r["budget"]
    np.testing.assert_array_equal(g["draft_len"].cpu().numpy(), r["draft_len"])
    return g, r


@pytest.mark.parametrize("B,K", [(1, 1), (3, 5), (256, 8), (64, 31), (2048, 8), (512, 31)])
def test_av_budget_matches_oracle(B, K):
    sv = _sv()
    rng = np.random.default_rng(B * 100 + K)
    conf = rng.beta(4, 2, (B, K)).astype(np.float32)
    dc, vc = _costs(rng, B * K, B)
    g, r = _budget_case(sv, conf, dc, vc)
    assert 0 < r["budget"] < B * K or B * K == 1


def test_av_budget_ties_zeros_and_bad_costs():
    sv = _sv()
    rng = np.random.default_rng(9)
    B, K = 40, 6
    conf = rng.choice(np.array([0.0, 0.5, 1.0], np.float32), (B, K))
    conf[3, 2] = np.nan
    dc, vc = _costs(rng, B * K, B)
    vc[5:20] = 0.0
    vc[30] = -1.0
    _budget_case(sv, conf, dc, vc)
    # nothing eligible: budget 0
    z = np.zeros(B * K + 1, np.float32)
    g, r = _budget_case(sv, conf, z, z)
    assert r["budget"] == 0 and int(g["budget"].item()) == 0


def test_av_budget_cuts_through_a_cross_sequence_tie():
    """Budgets that end inside a group of equal survival values spread over
    sequences: ties rank by ascending flat index on both sides."""
    sv = _sv()
    g, _ = _budget_case(sv, np.array([[0.5], [0.5]], np.float32), np.zeros(3, np.float32),
                        np.array([1, 1, 2], np.float32))
    assert g["draft_len"].cpu().tolist() == [1, 0]
    g, _ = _budget_case(sv, np.full((3, 2), 0.5, np.float32), np.zeros(7, np.float32),
                        np.array([1, 1, 1, 1, 1, 4, 4], np.float32))
    assert g["draft_len"].cpu().tolist() == [2, 1, 1]


@pytest.mark.parametrize("mode", ["stochastic", "greedy", "fly"])
def test_ragged_verify_matches_oracle(mode):
    sv = _sv()
    w = workloads.LLAMA3_VOCAB
    w = type(w)(**{**w.__dict__, "B": 24})
    inp = workloads.make_inputs(w, 4321, DEV)
    rng = np.random.default_rng(3)
    dl = rng.integers(0, w.K + 1, w.B).astype(np.int32)
    dl[:3] = [0, w.K, 1]
    est = torch.tensor(np.r_[1.0, np.zeros(w.K)], dtype=torch.float32, device=DEV)
    kw = dict(fly_theta=0.3, fly_window=2) if mode == "fly" else {}
    g = hv.verify(inp["zt"], inp["zd"], inp["x"], inp["u"] if mode == "stochastic" else None, mode=mode,
                  est_params=est, want_pos_stats=True, want_feature=True, want_conf=True,
                  draft_len=torch.tensor(dl, device=DEV), **kw)
    torch.cuda.synchronize()
    om = {"stochastic": oracle.STOCHASTIC, "greedy": oracle.GREEDY, "fly": oracle.FLY}[mode]
    r = oracle_run(inp, om, est=np.r_[1.0, np.zeros(w.K)], draft_len=dl, **kw)
    compare(g, r, w.dtype, check_feature=True, check_conf=True)
    assert sv.device_status(g["_workspace"]) == 0


def test_full_draft_length_equals_the_unpruned_launch():
    sv = _sv()
    w = workloads.ESTIMATOR
    w = type(w)(**{**w.__dict__, "B": 32})
    inp = workloads.make_inputs(w, 77, DEV)
    a = hv.verify(inp["zt"], inp["zd"], inp["x"], inp["u"], want_pos_stats=True, want_feature=True)
    b = hv.verify(inp["zt"], inp["zd"], inp["x"], inp["u"], want_pos_stats=True, want_feature=True,
                  draft_len=torch.full((w.B,), w.K, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    for k in ("out_tokens", "accepted_len", "pos_stats", "feature"):
        assert torch.equal(a[k], b[k]) or (k in ("pos_stats", "feature") and torch.allclose(
            a[k], b[k], rtol=0, atol=0, equal_nan=True)), k


def test_pruned_labels_match_oracle():
    sv = _sv()
    rng = np.random.default_rng(12)
    B, K = 300, 8
    f = rng.normal(0, 2, (B, K)).astype(np.float32)
    dl = rng.integers(0, K + 1, B).astype(np.int32)
    n = np.array([rng.integers(0, d + 1) for d in dl], np.int32)
    th = np.r_[0.7, rng.normal(0, 0.5, K)].astype(np.float32)
    t = lambda a: torch.tensor(a, device=DEV)
    p = t(th)
    grad, cnt = sv.estimator_update(t(f), t(n), p, 0.0, want_grad=True, draft_len=t(dl))
    st = sv.IrlsState(K, DEV)
    sv.irls_accumulate(t(f), t(n), t(th), st, draft_len=t(dl))
    torch.cuda.synchronize()
    _, g_ref, c_ref = oracle.estimator_update(f.astype(np.float64), n, th.astype(np.float64), 0.0, draft_len=dl)
    np.testing.assert_array_equal(cnt.cpu().numpy(), c_ref)
    np.testing.assert_allclose(grad.cpu().numpy(), g_ref, rtol=1e-4, atol=1e-5)
    ref = oracle.irls_zero(K)
    oracle.irls_accumulate(f.astype(np.float64), n, th.astype(np.float64), ref, draft_len=dl)
    nn = st.parts()[4].cpu().numpy()
    np.testing.assert_array_equal(nn, ref[2].astype(np.float64))
    np.testing.assert_allclose(st.parts()[0].cpu().numpy(), ref[0], rtol=1e-4, atol=1e-4)


def test_av_step_end_to_end():
    """One AV decoding step, run twice from the same seeded logits: on the GPU
    (spec_confidence, spec_av_budget, spec_verify_ragged) and in the oracle
    (confidence, budget, pruned verify). The two pipelines share only the
    inputs; the draft lengths must agree, then the verification outputs."""
    sv = _sv()
    w = workloads.ESTIMATOR
    w = type(w)(**{**w.__dict__, "B": 48})
    inp = workloads.make_inputs(w, 2024, DEV)
    est_h = np.r_[0.5, np.linspace(1.0, -0.5, w.K)]
    est = torch.tensor(est_h, dtype=torch.float32, device=DEV)
    N = w.B * w.K
    dc, vc = _costs(np.random.default_rng(1), N, w.B)
    # GPU pipeline
    _, conf = hv.confidence(inp["zd"], est)
    bud = sv.av_budget(conf, torch.tensor(dc, device=DEV), torch.tensor(vc, device=DEV))
    g = hv.verify(inp["zt"], inp["zd"], inp["x"], inp["u"], est_params=est, want_pos_stats=True,
                  want_feature=True, want_conf=True, draft_len=bud["draft_len"])
    torch.cuda.synchronize()
    # oracle pipeline
    _, conf_r, _ = oracle.confidence(workloads.to_numpy_logits(inp["zd"]), est_h.astype(np.float32).astype(np.float64))
    rb = oracle.av_budget(conf_r.astype(np.float32), dc, vc)
    np.testing.assert_array_equal(bud["draft_len"].cpu().numpy(), rb["draft_len"])
    assert 0 < rb["budget"] < N
    r = oracle_run(inp, oracle.STOCHASTIC, est=est_h.astype(np.float32).astype(np.float64),
                   draft_len=rb["draft_len"])
    compare(g, r, w.dtype, check_feature=True, check_conf=True)
