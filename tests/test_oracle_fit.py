"""Pins of the oracle's AV refit (CPU only).

The refit is the IRLS / Newton step of the AV article, section "Fitting the
coefficients": labels on drafts up to and including the first rejection,
gradient g and Hessian H of the summed log-loss, H * delta = g with H of
size (K+1)x(K+1), shared slope, damping n / (n + constant), accumulation over
a round of N decode steps.  Pinned here against finite differences, numpy's
dense solver, scipy's optimiser and recovery of known parameters.
"""
import numpy as np
import pytest
from scipy.optimize import minimize
from scipy.special import expit

import oracle


def _dataset(B, K, seed, omega=0.5, beta0=0.55, slope_beta=-0.25, kept=None):
    """Features and accept lengths drawn from a known per-position logistic
    model (slope 0.5, intercepts falling with depth from 0.55)."""
    rng = np.random.default_rng(seed)
    beta = beta0 + slope_beta * np.arange(K)
    x = rng.normal(1.0, 2.0, (B, K))
    acc = rng.random((B, K)) < expit(omega * x + beta)
    a = np.where(acc.all(1), K, np.argmin(acc, axis=1)).astype(np.int32)
    if kept is not None:
        a = np.minimum(a, kept)
    return x, a, np.concatenate([[omega], beta])


def _labels(x, a, kept, K):
    rows = []
    for b in range(x.shape[0]):
        k = K if kept is None else kept[b]
        for i in range(min(a[b] + 1, k)):
            rows.append((i, x[b, i], 1.0 if i < a[b] else 0.0))
    return rows


def _loss(theta, rows):
    s = 0.0
    for i, x, y in rows:
        z = theta[0] * x + theta[1 + i]
        s += np.logaddexp(0, z) - y * z  # -[y log sig(z) + (1-y) log(1-sig(z))]
    return s


def test_label_eligibility_counts():
    K = 5
    x, a, _ = _dataset(300, K, seed=1)
    kept = np.random.default_rng(2).integers(0, K + 1, 300).astype(np.int32)
    a = np.minimum(a, kept)
    acc = oracle.av_accumulate(np.zeros(K + 1), x, a, kept)
    want = np.zeros(K)
    for i, _, _ in _labels(x, a, kept, K):
        want[i] += 1
    assert np.array_equal(acc["n"], want)
    # a fully accepted canvas carries K positive labels and no negative one
    acc1 = oracle.av_accumulate(np.zeros(K + 1), np.zeros((1, K)), np.array([K]))
    assert acc1["n"].sum() == K


def test_gradient_and_hessian_by_finite_differences():
    K = 4
    x, a, _ = _dataset(200, K, seed=3)
    theta = np.array([0.3, 0.2, 0.1, -0.1, -0.4])
    acc = oracle.av_accumulate(theta, x, a)
    rows = _labels(x, a, None, K)
    h = 1e-6
    for j in range(K + 1):
        e = np.zeros(K + 1)
        e[j] = h
        fd = (_loss(theta + e, rows) - _loss(theta - e, rows)) / (2 * h)
        assert abs(fd - acc["g"][j]) < 1e-5 * max(1.0, abs(fd))
        g_plus = oracle.av_accumulate(theta + e, x, a)["g"]
        g_minus = oracle.av_accumulate(theta - e, x, a)["g"]
        fdH = (g_plus - g_minus) / (2 * h)
        assert np.abs(fdH - acc["H"][j]).max() < 1e-5 * max(1.0, np.abs(fdH).max())


def test_newton_delta_equals_dense_solve():
    K = 6
    x, a, _ = _dataset(400, K, seed=4)
    theta = np.zeros(K + 1)
    acc = oracle.av_accumulate(theta, x, a)
    assert np.all(acc["n"] > 0)
    H, g = acc["H"], acc["g"]
    ridge = 1e-9 * np.trace(H) / (K + 1)
    want = np.linalg.solve(H + ridge * np.eye(K + 1), g)
    new, delta, st = oracle.av_solve_update(theta, acc, damping_c=10.0)
    assert st == 0
    assert np.abs(delta - want).max() < 1e-10 * np.abs(want).max()
    ntot = acc["n"].sum()
    assert abs(new[0] - (theta[0] - ntot / (ntot + 10) * want[0])) < 1e-12
    for i in range(K):
        n = acc["n"][i]
        assert abs(new[1 + i] - (theta[1 + i] - n / (n + 10) * want[1 + i])) < 1e-12


def test_positions_without_labels_keep_their_intercept():
    K = 5
    x, a, _ = _dataset(100, K, seed=5)
    kept = np.full(100, 3, np.int32)
    a = np.minimum(a, kept)
    theta = np.array([0.5, 0.4, 0.3, 0.2, 0.7, -0.9])
    acc = oracle.av_accumulate(theta, x, a, kept)
    assert acc["n"][3] == 0 and acc["n"][4] == 0
    new, delta, st = oracle.av_solve_update(theta, acc)
    assert st == 0
    assert new[4] == theta[4] and new[5] == theta[5]
    assert delta[4] == 0 and delta[5] == 0
    # the reduced system is the dense solve over (omega, beta_0..beta_2)
    idx = [0, 1, 2, 3]
    Hr = acc["H"][np.ix_(idx, idx)]
    ridge = 1e-9 * np.trace(acc["H"]) / (K + 1)
    want = np.linalg.solve(Hr + ridge * np.eye(4), acc["g"][idx])
    assert np.abs(delta[idx] - want).max() < 1e-10 * np.abs(want).max()


def test_no_labels_no_update():
    K = 3
    theta = np.array([0.5, 0.1, 0.2, 0.3])
    acc = oracle.av_accumulate(theta, np.zeros((4, K)), np.zeros(4, np.int32), np.zeros(4, np.int32))
    new, _, st = oracle.av_solve_update(theta, acc)
    assert st == 1 and np.array_equal(new, theta)


def test_undamped_iterations_converge_to_mle():
    K = 4
    x, a, _ = _dataset(3000, K, seed=6)
    rows = _labels(x, a, None, K)
    mle = minimize(_loss, np.zeros(K + 1), args=(rows,), method="BFGS", options=dict(gtol=1e-9)).x
    theta = np.zeros(K + 1)
    for _ in range(12):
        acc = oracle.av_accumulate(theta, x, a)
        theta, _, st = oracle.av_solve_update(theta, acc, damping_c=0.0)
        assert st == 0
    assert np.abs(theta - mle).max() < 1e-5


def test_recovers_known_parameters():
    K = 5
    x, a, truth = _dataset(40000, K, seed=7)
    theta = np.zeros(K + 1)
    for _ in range(10):
        acc = oracle.av_accumulate(theta, x, a)
        theta, _, _ = oracle.av_solve_update(theta, acc, damping_c=0.0)
    acc = oracle.av_accumulate(theta, x, a)
    se = np.sqrt(np.diag(np.linalg.inv(acc["H"])))
    assert np.all(np.abs(theta - truth) < 4 * se), (theta, truth, se)
    assert 0.45 < theta[0] < 0.55


def test_round_accumulation_equals_pooled_data():
    K = 4
    fit = oracle.AVFit(np.zeros(K + 1), round_len=3, damping_c=10.0)
    xs, as_ = [], []
    for s in range(3):
        x, a, _ = _dataset(150, K, seed=20 + s)
        xs.append(x)
        as_.append(a)
        st = fit.step(x, a)
        assert (st is None) == (s < 2)
    pooled = oracle.av_accumulate(np.zeros(K + 1), np.concatenate(xs), np.concatenate(as_))
    want, _, _ = oracle.av_solve_update(np.zeros(K + 1), pooled, 10.0)
    assert np.abs(fit.theta - want).max() < 1e-12


@pytest.mark.parametrize("c", [0.0, 10.0, 1e6])
def test_damping_scales_the_step(c):
    K = 3
    x, a, _ = _dataset(500, K, seed=8)
    theta = np.array([0.2, 0.0, 0.0, 0.0])
    acc = oracle.av_accumulate(theta, x, a)
    new, delta, _ = oracle.av_solve_update(theta, acc, c)
    n = np.concatenate([[acc["n"].sum()], acc["n"]])
    assert np.allclose(theta - new, n / (n + c) * delta, rtol=0, atol=1e-13)
