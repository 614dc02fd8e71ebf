"""Pins of the oracle's IRLS refit of the acceptance estimator.

"Verificación Adaptativa sin una cabeza de confianza", section "Ajuste de los
Coeficientes": over a round of decoding steps the gradient and Hessian of the
log-loss are accumulated at fixed coefficients; the refit solves the Newton
system and damps each coefficient's step by n / (n + c). Each test ties the
oracle to something other than its own code: central finite differences, a
library linear solve, the maximum-likelihood fit of scipy's minimiser on a
log-loss written here with scipy's special functions, hand-derived cases and
the additivity of a round. CPU only.
"""
import numpy as np
import pytest
from scipy import optimize, special

import oracle


def _data(seed, B=24, K=4, spread=2.0):
    rng = np.random.default_rng(seed)
    f = rng.normal(0.0, spread, (B, K))
    n = rng.integers(0, K + 1, B).astype(np.int32)
    th = np.r_[0.7, rng.normal(0.0, 0.6, K)]
    return f, n, th


def _labels(f, n):
    """(x rows, y) of the eligible labels, as the pages define them."""
    B, K = f.shape
    X, Y = [], []
    for b in range(B):
        for i in range(min(int(n[b]), K - 1) + 1):
            x = np.zeros(K + 1)
            x[0] = f[b, i]
            x[1 + i] = 1.0
            X.append(x)
            Y.append(1.0 if i < n[b] else 0.0)
    return np.array(X), np.array(Y)


def _sum_loss(th, X, Y):
    z = X @ th
    return float(-(Y * special.log_expit(z) + (1 - Y) * special.log_expit(-z)).sum())


def _round(f, n, th):
    K = f.shape[1]
    st = oracle.irls_zero(K)
    oracle.irls_accumulate(f, n, th, st)
    return st


def test_gradient_and_hessian_by_finite_differences():
    f, n, th = _data(1)
    X, Y = _labels(f, n)
    g, H, cnt = _round(f, n, th)
    h = 1e-5
    K1 = th.size
    g_fd = np.empty(K1)
    H_fd = np.empty((K1, K1))
    for k in range(K1):
        e = np.zeros(K1)
        e[k] = h
        g_fd[k] = (_sum_loss(th + e, X, Y) - _sum_loss(th - e, X, Y)) / (2 * h)
        # the Hessian column from the gradient of a different function: the
        # oracle's mean-gradient step (lr = 0), times the label count
        gp = oracle.estimator_update(f, n, th + e, 0.0)[1] * cnt[0]
        gm = oracle.estimator_update(f, n, th - e, 0.0)[1] * cnt[0]
        H_fd[:, k] = (gp - gm) / (2 * h)
    np.testing.assert_allclose(g, g_fd, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(H, H_fd, rtol=1e-6, atol=1e-6)
    np.testing.assert_array_equal(H, H.T)
    assert cnt[0] == len(Y) and cnt[1:].sum() == len(Y)


def test_undamped_step_is_the_newton_solve():
    f, n, th = _data(2, B=64)
    g, H, cnt = st = _round(f, n, th)
    assert (cnt > 0).all()
    p, step = oracle.irls_refit(st, th, 0.0)
    np.testing.assert_allclose(step, np.linalg.solve(H, g), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(p, th - step, rtol=0, atol=1e-15)


def test_iterated_refits_reach_the_maximum_likelihood_fit():
    f, n, _ = _data(3, B=200, K=3, spread=1.5)
    X, Y = _labels(f, n)
    th = np.zeros(4)
    for _ in range(30):
        th, _step = oracle.irls_refit(_round(f, n, th), th, 0.0)
    res = optimize.minimize(_sum_loss, np.zeros(4), args=(X, Y), method="BFGS",
                            jac=lambda t, X, Y: X.T @ (special.expit(X @ t) - Y),
                            options={"gtol": 1e-10, "maxiter": 1000})
    np.testing.assert_allclose(th, res.x, rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("c", [0.5, 7.0, 300.0])
def test_damping_scales_each_step_by_its_evidence(c):
    f, n, th = _data(4, B=40)
    st = _round(f, n, th)
    cnt = st[2]
    _, step0 = oracle.irls_refit(st, th, 0.0)
    p, step = oracle.irls_refit(st, th, c)
    np.testing.assert_allclose(step, step0 * cnt / (cnt + c), rtol=1e-13, atol=0)
    np.testing.assert_allclose(p, th - step, rtol=0, atol=1e-15)
    p_inf, _ = oracle.irls_refit(st, th, 1e15)
    np.testing.assert_allclose(p_inf, th, rtol=0, atol=1e-9)


def test_hand_cases():
    # one accepted label at f = 0, theta = 0: s = 1/2, e = -1/2, w = 1/4;
    # g = (0, -1/2), H = [[0, 0], [0, 1/4]]: the slope is not determined and
    # is held; the intercept moves by -(-1/2)/(1/4) = +2
    st = oracle.irls_zero(1)
    oracle.irls_accumulate(np.zeros((1, 1)), np.array([1]), np.zeros(2), st)
    np.testing.assert_allclose(st[0], [0.0, -0.5])
    np.testing.assert_allclose(st[1], [[0.0, 0.0], [0.0, 0.25]])
    np.testing.assert_array_equal(st[2], [1, 1])
    p, step = oracle.irls_refit(st, np.zeros(2), 0.0)
    np.testing.assert_allclose(p, [0.0, 2.0])
    p, _ = oracle.irls_refit(st, np.zeros(2), 1.0)                # damped by 1 / (1 + 1)
    np.testing.assert_allclose(p, [0.0, 1.0])
    # an accepted label at f = +1 and a rejected one at f = -1, theta = 0:
    # g = (-1, 0), H = [[1/2, 0], [0, 1/2]], so theta becomes (2, 0)
    st = oracle.irls_zero(1)
    oracle.irls_accumulate(np.array([[1.0], [-1.0]]), np.array([1, 0]), np.zeros(2), st)
    np.testing.assert_allclose(st[0], [-1.0, 0.0])
    np.testing.assert_allclose(st[1], [[0.5, 0.0], [0.0, 0.5]])
    p, _ = oracle.irls_refit(st, np.zeros(2), 0.0)
    np.testing.assert_allclose(p, [2.0, 0.0])


def test_unlabelled_coefficients_keep_their_value():
    # every draft rejected at position 0: only beta_1 (and the slope) have labels
    f, _, th = _data(5, B=30, K=3)
    n = np.zeros(30, np.int32)
    st = _round(f, n, th)
    np.testing.assert_array_equal(st[2], [30, 30, 0, 0])
    p, step = oracle.irls_refit(st, th, 0.0)
    assert step[2] == 0.0 and step[3] == 0.0 and p[2] == th[2] and p[3] == th[3]
    # an empty round changes nothing
    p, step = oracle.irls_refit(oracle.irls_zero(3), th, 0.0)
    np.testing.assert_array_equal(p, th)
    np.testing.assert_array_equal(step, 0.0)


def test_a_round_adds_its_steps():
    f, n, th = _data(6, B=50)
    st = oracle.irls_zero(4)
    oracle.irls_accumulate(f[:20], n[:20], th, st)
    oracle.irls_accumulate(f[20:], n[20:], th, st)
    whole = _round(f, n, th)
    for a, b in zip(st, whole):
        np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)
