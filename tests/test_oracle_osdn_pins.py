"""Pins of the OSDN write-key oracle (oracle.osdn), CPU only: the page's
worked loss-ratio example, the reduction to the plain recurrence at
eta = 0, the scan against its affine form A_t d + b_t, the projection
bounds, the emission order (the write key uses d before its update), the
APF retention, and the scalar recursion of one-hot keys."""
import os

import numpy as np

import oracle
from oracle import osdn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "osdn_loss_ratio.txt")


def rows(seed, B=1, T=6, H=2, nh=2, Dk=5, Dv=3):
    rng = np.random.default_rng(seed)
    k = rng.normal(size=(B, T, H, nh, Dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    return dict(q=rng.normal(size=(B, T, H, Dk)), k=k, v=rng.normal(size=(B, T, H, nh, Dv)),
                beta=rng.uniform(0.1, 0.9, size=(B, T, H, nh)), g=rng.uniform(0.6, 1.0, size=(B, T, H)),
                h0=rng.normal(size=(B, H, Dk, Dv)))


def test_worked_loss_ratio():
    data = np.loadtxt(GOLDEN)
    for d1, d2, b, q_ref in data:
        k = np.array([1.0, 0.0])
        v = np.array([1.0])
        kw = np.array([d1, d2]) * k
        args = dict(q=np.zeros((1, 1, 1, 2)), k=k.reshape(1, 1, 1, 1, 2), v=v.reshape(1, 1, 1, 1, 1),
                    beta=np.full((1, 1, 1, 1), b))
        _, hf = oracle.forward(**args, kw=kw.reshape(1, 1, 1, 1, 2), threads=1)
        before = 0.5 * float(np.sum((np.zeros(1) - v) ** 2))
        after = 0.5 * float(np.sum((hf[0, 0].T @ k - v) ** 2))
        np.testing.assert_allclose(after / before, q_ref, rtol=1e-14)


def test_eta_zero_is_plain_recurrence():
    x = rows(1)
    o, hf, kw, d = osdn.forward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], eta=0.0, threads=1)
    np.testing.assert_array_equal(kw, x["k"])
    np.testing.assert_array_equal(d, 1.0)
    o2, hf2 = oracle.forward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], threads=1)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(hf, hf2)


def test_scan_affine_form():
    """Without the projection the update is d' = A d + b with
    A = r I - (eta beta^2 / nbar) s s^T and b = (eta beta / nbar) s."""
    x = rows(2, T=5, H=1, nh=3, Dk=4)
    rng = np.random.default_rng(3)
    r = rng.uniform(0.5, 1.0, size=(1, 5, 1))
    eta = 0.2
    kw, d = osdn.dscan(x["k"], x["beta"], r, eta=eta, d_lo=-np.inf, d_hi=np.inf)
    dd = np.ones(4)
    for t in range(5):
        for j in range(3):
            kk, b = x["k"][0, t, 0, j], x["beta"][0, t, 0, j]
            np.testing.assert_allclose(kw[0, t, 0, j], dd * kk, rtol=1e-14)
            s = kk * kk
            nbar = max(s.sum(), osdn.EPS)
            rr = r[0, t, 0] if j == 0 else 1.0
            A = rr * np.eye(4) - (eta * b * b / nbar) * np.outer(s, s)
            dd = A @ dd + (eta * b / nbar) * s
    np.testing.assert_allclose(d[0, 0], dd, rtol=1e-12)


def test_projection_bounds_and_first_row():
    x = rows(4, T=20, H=2, nh=2)
    kw, d = osdn.dscan(x["k"], x["beta"], eta=50.0)
    assert np.all(d >= 0.5) and np.all(d <= 2.0)
    assert np.any(d == 0.5) or np.any(d == 2.0)
    np.testing.assert_array_equal(kw[:, 0, :, 0], x["k"][:, 0, :, 0])   # d_1 = 1 on the first row


def test_apf_retention_pulls_down_to_the_bound():
    x = rows(5, T=3, H=1, nh=1)
    _, d = osdn.dscan(x["k"], x["beta"], r=np.zeros((1, 3, 1)), eta=0.0)
    np.testing.assert_array_equal(d, 0.5)


def test_one_hot_keys_scalar_recursion():
    T, Dk, eta = 40, 3, 0.05
    rng = np.random.default_rng(6)
    idx = rng.integers(0, Dk, size=T)
    k = np.zeros((1, T, 1, 1, Dk))
    k[0, np.arange(T), 0, 0, idx] = 1.0
    beta = rng.uniform(0.2, 0.9, size=(1, T, 1, 1))
    _, d = osdn.dscan(k, beta, eta=eta)
    ref = np.ones(Dk)
    for t in range(T):
        i, b = idx[t], beta[0, t, 0, 0]
        ref[i] = min(max(ref[i] + eta * b * (1 - b * ref[i]), 0.5), 2.0)
    np.testing.assert_allclose(d[0, 0], ref, rtol=1e-14)
