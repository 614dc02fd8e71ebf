"""GPU parity of the IRLS refit (spec_irls_*) against the fp64 oracle.

"Verificación Adaptativa sin una cabeza de confianza", "Ajuste de los
Coeficientes". Inputs are seeded numpy draws; the oracle sees the same fp32
features and parameters (widened to fp64).

Tolerances. The GPU forms each label's sigmoid terms in fp32 (a few ulp each)
and sums them in fp64, so a round's sums carry a relative error of about
1e-6 of the sum of their terms' magnitudes: the test allows 1e-5 (the fp32
figure of the parity contract) of that magnitude. The refit's solve is fp64
on both sides: given the same round (uploaded from the host) the applied
steps agree to 1e-11; after a GPU-accumulated round they agree to the round's
error times the condition of H (2e-4 here). fp32 parameters agree to one fp32
rounding beyond that.
"""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _sv():
    import speculative_decoding_token_verify_gb300 as sv
    sv.build()
    return sv


def _step_data(rng, B, K, spread=2.0):
    f = rng.normal(0.0, spread, (B, K)).astype(np.float32)
    n = rng.integers(0, K + 1, B).astype(np.int32)
    return f, n


def _params(rng, K):
    return np.r_[0.8, rng.normal(0.0, 0.5, K)].astype(np.float32)


def _magnitudes(f, n, th, K):
    """Per coefficient, the sum of |term| magnitudes of g and H (tolerance scale only)."""
    B = f.shape[0]
    mg, mH = np.zeros(K + 1), np.zeros((K + 1, K + 1))
    for b in range(B):
        for i in range(min(int(n[b]), K - 1) + 1):
            x = np.zeros(K + 1)
            x[0], x[1 + i] = f[b, i], 1.0
            mg += np.abs(x)
            mH += 0.25 * np.abs(np.outer(x, x))
    return mg, mH


def _dense(parts, K):
    g, hww, hwb, hbb, n = (t.double().cpu().numpy() for t in parts)
    H = np.zeros((K + 1, K + 1))
    H[0, 0] = hww[0]
    H[0, 1:] = H[1:, 0] = hwb
    H[np.arange(1, K + 1), np.arange(1, K + 1)] = hbb
    return g, H, n


@pytest.mark.parametrize("B,K", [(256, 8), (37, 5), (1, 1), (64, 31), (1000, 3)])
def test_accumulate_matches_oracle(B, K):
    sv = _sv()
    rng = np.random.default_rng(100 + B + K)
    th = _params(rng, K)
    st = sv.IrlsState(K, DEV)
    ref = oracle.irls_zero(K)
    p_dev = torch.tensor(th, device=DEV)
    mg, mH = np.zeros(K + 1), np.zeros((K + 1, K + 1))
    for _ in range(3):
        f, n = _step_data(rng, B, K)
        sv.irls_accumulate(torch.tensor(f, device=DEV), torch.tensor(n, device=DEV), p_dev, st)
        oracle.irls_accumulate(f.astype(np.float64), n, th.astype(np.float64), ref)
        a, b = _magnitudes(f.astype(np.float64), n, th, K)
        mg, mH = mg + a, mH + b
    torch.cuda.synchronize()
    g, H, cnt = _dense(st.parts(), K)
    assert (np.abs(g - ref[0]) <= 1e-5 * mg + 1e-12).all(), np.max(np.abs(g - ref[0]) / (mg + 1e-30))
    assert (np.abs(H - ref[1]) <= 1e-5 * mH + 1e-12).all(), np.max(np.abs(H - ref[1]) / (mH + 1e-30))
    np.testing.assert_array_equal(cnt, ref[2].astype(np.float64))


@pytest.mark.parametrize("damping", [0.0, 16.0, 1e6])
def test_round_then_refit_matches_oracle(damping):
    sv = _sv()
    K, B = 8, 256
    rng = np.random.default_rng(7)
    th = _params(rng, K)
    st = sv.IrlsState(K, DEV)
    ref = oracle.irls_zero(K)
    p_dev = torch.tensor(th, device=DEV)
    for _ in range(4):
        f, n = _step_data(rng, B, K)
        sv.irls_accumulate(torch.tensor(f, device=DEV), torch.tensor(n, device=DEV), p_dev, st)
        oracle.irls_accumulate(f.astype(np.float64), n, th.astype(np.float64), ref)
    step = sv.irls_refit(st, p_dev, damping, want_step=True)
    torch.cuda.synchronize()
    p_ref, step_ref = oracle.irls_refit(ref, th.astype(np.float64), damping)
    np.testing.assert_allclose(step.cpu().numpy(), step_ref, rtol=2e-4, atol=1e-7)
    got = p_dev.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(got, p_ref, rtol=1e-5, atol=1e-6)
    assert float(st.tensor.abs().max()) == 0.0          # the refit starts the next round


def _upload_round(sv, K, g, H, n):
    st = sv.IrlsState(K, DEV)
    t = np.concatenate([g, [H[0, 0]], H[0, 1:], np.diag(H)[1:], n.astype(np.float64)])
    st.tensor.copy_(torch.tensor(t, dtype=torch.float64))
    return st


def _arrow_round(rng, K, labelled=None, slope_free=False):
    """A consistent round built on the host: H = sum of w x x^T over labels."""
    n = rng.integers(1, 50, K + 1).astype(np.int64)
    if labelled is not None:
        n[1:][~labelled] = 0
    n[0] = n[1:].sum()
    D = rng.uniform(0.5, 5.0, K) * (n[1:] > 0)
    c = rng.normal(0.0, 1.0, K) * (n[1:] > 0)
    if slope_free:
        c[:] = 0.0
        hww = 0.0
    else:
        hww = float(np.sum(c * c / np.where(D > 0, D, 1.0))) + rng.uniform(0.5, 3.0)
    H = np.zeros((K + 1, K + 1))
    H[0, 0] = hww
    H[0, 1:] = H[1:, 0] = c
    H[np.arange(1, K + 1), np.arange(1, K + 1)] = D
    g = rng.normal(0.0, 2.0, K + 1)
    g[1:][n[1:] == 0] = 0.0
    return g, H, n


@pytest.mark.parametrize("case", ["full", "holes", "slope_held"])
@pytest.mark.parametrize("damping", [0.0, 3.0])
def test_refit_solve_on_a_given_round(case, damping):
    sv = _sv()
    K = 9
    rng = np.random.default_rng({"full": 1, "holes": 2, "slope_held": 3}[case])
    labelled = None
    if case == "holes":
        labelled = np.array([True, True, False, True, False, False, True, True, False])
    g, H, n = _arrow_round(rng, K, labelled, slope_free=(case == "slope_held"))
    th = _params(rng, K)
    st = _upload_round(sv, K, g, H, n)
    p_dev = torch.tensor(th, device=DEV)
    step = sv.irls_refit(st, p_dev, damping, want_step=True).cpu().numpy()
    p_ref, step_ref = oracle.irls_refit((g.copy(), H.copy(), n.copy()), th.astype(np.float64), damping)
    np.testing.assert_allclose(step, step_ref, rtol=1e-11, atol=1e-13)
    if case == "slope_held":
        assert step[0] == 0.0
    if case == "holes":
        assert (step[1:][~labelled] == 0.0).all()
    np.testing.assert_allclose(p_dev.cpu().numpy().astype(np.float64), p_ref, rtol=2e-7, atol=1e-7)


def test_iterated_rounds_follow_the_oracle_to_the_fit():
    sv = _sv()
    K, B = 4, 400
    rng = np.random.default_rng(11)
    f, n = _step_data(rng, B, K, spread=1.5)
    th_ref = np.zeros(K + 1)
    p_dev = torch.zeros(K + 1, dtype=torch.float32, device=DEV)
    st = sv.IrlsState(K, DEV)
    fd, nd = torch.tensor(f, device=DEV), torch.tensor(n, device=DEV)
    for _ in range(12):
        sv.irls_accumulate(fd, nd, p_dev, st)
        sv.irls_refit(st, p_dev, 0.0)
        th_ref, _ = oracle.irls_refit(oracle.irls_accumulate(f.astype(np.float64), n, th_ref, oracle.irls_zero(K)),
                                      th_ref, 0.0)
    torch.cuda.synchronize()
    np.testing.assert_allclose(p_dev.cpu().numpy().astype(np.float64), th_ref, rtol=1e-4, atol=1e-5)


def test_empty_round_changes_nothing_and_runs_are_bitwise_repeatable():
    sv = _sv()
    K = 6
    rng = np.random.default_rng(5)
    th = _params(rng, K)
    p_dev = torch.tensor(th, device=DEV)
    st = sv.IrlsState(K, DEV)
    empty_f = torch.empty((0, K), dtype=torch.float32, device=DEV)
    empty_n = torch.empty((0,), dtype=torch.int32, device=DEV)
    sv.irls_accumulate(empty_f, empty_n, p_dev, st)
    step = sv.irls_refit(st, p_dev, 1.0, want_step=True)
    torch.cuda.synchronize()
    assert float(step.abs().max()) == 0.0
    np.testing.assert_array_equal(p_dev.cpu().numpy(), th)
    f, n = _step_data(rng, 512, K)
    fd, nd = torch.tensor(f, device=DEV), torch.tensor(n, device=DEV)
    states = []
    for _ in range(3):
        s2 = sv.IrlsState(K, DEV)
        for _ in range(2):
            sv.irls_accumulate(fd, nd, p_dev, s2)
        states.append(s2.tensor.clone())
    torch.cuda.synchronize()
    assert torch.equal(states[0], states[1]) and torch.equal(states[0], states[2])
