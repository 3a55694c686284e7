"""Pins of the fp64 backward oracle (oracle.backward), CPU only.

The backward is pinned to things other than itself: central finite
differences of L = <d_o, o> + <dh_final, h_final> evaluated with the forward
oracle (itself pinned in test_oracle_pins.py) over every entry of every
gradient on small inputs; the closed form of a single token with one
sub-step; the beta = 0 invariant (no write, so no gradient to k and v). A
numpy copy of the backward with plausible mistakes planted in it must fail
at least one pin, and the copy without a mistake must pass all of them and
agree with the C oracle.
"""
import numpy as np
import pytest

import oracle

SHAPE = dict(B=1, T=3, H=1, nh=2, Dk=3, Dv=2)


def case(seed, B, T, H, nh, Dk, Dv, gated=True, with_h0=True):
    rng = np.random.default_rng(seed)
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    x = {
        "q": rng.normal(size=(B, T, H, Dk)),
        "k": unit(rng.normal(size=(B, T, H, nh, Dk))),
        "v": rng.normal(size=(B, T, H, nh, Dv)),
        "beta": rng.uniform(0.2, 1.8, size=(B, T, H, nh)),
        "g": rng.uniform(0.5, 1.0, size=(B, T, H)) if gated else None,
        "h0": rng.normal(size=(B, H, Dk, Dv)) if with_h0 else None,
    }
    cot = {"d_o": rng.normal(size=(B, T, H, Dv)), "dh_final": rng.normal(size=(B, H, Dk, Dv))}
    return x, cot


def loss(x, cot):
    o, hf = oracle.forward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], threads=1)
    return float(np.sum(o * cot["d_o"]) + np.sum(hf * cot["dh_final"]))


def c_backward(x, cot):
    return oracle.backward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], cot["d_o"], cot["dh_final"],
                           threads=1)


GRADS = {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "g": "dg", "h0": "dh0"}


def pin_finite_differences(bwd, seed=31, gated=True, with_h0=True, nh=2):
    """Every entry of every gradient against central differences (fp64,
    step 1e-6: truncation ~1e-12, rounding ~1e-10)."""
    x, cot = case(seed, **{**SHAPE, "nh": nh}, gated=gated, with_h0=with_h0)
    grads = bwd(x, cot)
    eps = 1e-6
    for name, gname in GRADS.items():
        if x[name] is None:
            continue
        fd = np.zeros_like(x[name])
        for idx in np.ndindex(*x[name].shape):
            xp = {kk: (None if vv is None else vv.copy()) for kk, vv in x.items()}
            xm = {kk: (None if vv is None else vv.copy()) for kk, vv in x.items()}
            xp[name][idx] += eps
            xm[name][idx] -= eps
            fd[idx] = (loss(xp, cot) - loss(xm, cot)) / (2 * eps)
        np.testing.assert_allclose(grads[gname], fd, rtol=1e-6, atol=1e-7, err_msg=gname)


def pin_single_step_closed_form(bwd, seed=32):
    """T = 1, n_h = 1, no gate, H0 = 0: o = beta (k.q) v and h_final =
    beta k v^T, so dq = beta (v.do) k + beta dH v, etc. (derived by hand)."""
    rng = np.random.default_rng(seed)
    Dk, Dv = 4, 3
    q, k, v = rng.normal(size=Dk), rng.normal(size=Dk), rng.normal(size=Dv)
    b = 0.7
    do, dH = rng.normal(size=Dv), rng.normal(size=(Dk, Dv))
    x = {"q": q[None, None, None], "k": k[None, None, None, None], "v": v[None, None, None, None],
         "beta": np.array(b).reshape(1, 1, 1, 1), "g": None, "h0": None}
    cot = {"d_o": do[None, None, None], "dh_final": dH[None, None]}
    gr = bwd(x, cot)
    kq, vdo = k @ q, v @ do
    np.testing.assert_allclose(gr["dq"].ravel(), b * vdo * k, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gr["dv"].ravel(), b * kq * do + b * dH.T @ k, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gr["dk"].ravel(), b * vdo * q + b * dH @ v, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gr["dbeta"].ravel(), [kq * vdo + k @ dH @ v], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gr["dh0"].ravel(), (dH - b * np.outer(k, k @ dH) + np.outer(q, do)
                                                   - b * np.outer(k, (k @ q) * do)).ravel(),
                               rtol=1e-12, atol=1e-12)


def pin_zero_beta(bwd, seed=33):
    """beta = 0 everywhere: nothing is written, o_t = (prod g) H0^T q_t, so
    dk = dv = 0 while dbeta, dq, dg and dh0 are not."""
    x, cot = case(seed, B=1, T=4, H=2, nh=3, Dk=5, Dv=4)
    x["beta"][:] = 0.0
    gr = bwd(x, cot)
    assert np.all(gr["dk"] == 0) and np.all(gr["dv"] == 0)
    assert np.abs(gr["dbeta"]).max() > 0 and np.abs(gr["dq"]).max() > 0 and np.abs(gr["dg"]).max() > 0


PINS = [pin_finite_differences, pin_single_step_closed_form, pin_zero_beta,
        lambda bwd: pin_finite_differences(bwd, seed=34, gated=False, with_h0=False, nh=3),
        lambda bwd: pin_finite_differences(bwd, seed=35, gated=True, with_h0=False, nh=1)]


@pytest.mark.parametrize("i", range(len(PINS)))
def test_backward_pin(i):
    PINS[i](c_backward)


# --------------------------------------------------------------------------
# numpy copy of the backward with planted mistakes
# --------------------------------------------------------------------------

MUTANTS = ["dk_state_term_dropped", "dbeta_uses_v", "dstate_not_projected", "dg_after_scaling",
           "dq_from_gated_state", "dh0_not_gated", "dv_without_beta", "substeps_forward_order"]


def numpy_backward(kind):
    def bwd(x, cot):
        q, k, v, beta, g, h0 = (x[n] for n in ("q", "k", "v", "beta", "g", "h0"))
        B, T, H, nh, Dk = k.shape
        Dv = v.shape[-1]
        out = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v),
               "dbeta": np.zeros_like(beta), "dg": None if g is None else np.zeros_like(g),
               "dh0": np.zeros((B, H, Dk, Dv))}
        for b in range(B):
            for h in range(H):
                S = np.zeros((Dk, Dv)) if h0 is None else h0[b, h].copy()
                starts = []
                for t in range(T):
                    starts.append(S.copy())
                    if g is not None:
                        S = g[b, t, h] * S
                    for j in range(nh):
                        S = S + beta[b, t, h, j] * np.outer(k[b, t, h, j], v[b, t, h, j] - S.T @ k[b, t, h, j])
                dS = cot["dh_final"][b, h].copy()
                for t in range(T - 1, -1, -1):
                    gt = 1.0 if g is None else g[b, t, h]
                    subs, errs = [gt * starts[t]], []
                    for j in range(nh):
                        e = v[b, t, h, j] - subs[-1].T @ k[b, t, h, j]
                        errs.append(e)
                        subs.append(subs[-1] + beta[b, t, h, j] * np.outer(k[b, t, h, j], e))
                    do = cot["d_o"][b, t, h]
                    out["dq"][b, t, h] = (subs[0] if kind == "dq_from_gated_state" else subs[nh]) @ do
                    dS = dS + np.outer(q[b, t, h], do)
                    order = range(nh) if kind == "substeps_forward_order" else range(nh - 1, -1, -1)
                    for j in order:
                        kk, bt, e = k[b, t, h, j], beta[b, t, h, j], errs[j]
                        du = dS.T @ kk
                        out["dv"][b, t, h, j] = du if kind == "dv_without_beta" else bt * du
                        out["dbeta"][b, t, h, j] = du @ (v[b, t, h, j] if kind == "dbeta_uses_v" else e)
                        dk = dS @ (bt * e)
                        if kind != "dk_state_term_dropped":
                            dk = dk - bt * subs[j] @ du
                        out["dk"][b, t, h, j] = dk
                        if kind != "dstate_not_projected":
                            dS = dS - bt * np.outer(kk, du)
                    if g is not None:
                        if kind == "dg_after_scaling":
                            dS = gt * dS
                            out["dg"][b, t, h] = np.sum(dS * starts[t])
                        else:
                            out["dg"][b, t, h] = np.sum(dS * starts[t])
                            if kind != "dh0_not_gated":
                                dS = gt * dS
                out["dh0"][b, h] = dS
        return out
    return bwd


@pytest.mark.parametrize("kind", MUTANTS)
def test_backward_mutant_is_caught(kind):
    bwd = numpy_backward(kind)
    caught = []
    for i, pin in enumerate(PINS):
        try:
            pin(bwd)
        except AssertionError:
            caught.append(i)
    assert caught, f"mutant {kind} passed every pin"


def test_unmutated_numpy_copy_passes_and_matches_c():
    bwd = numpy_backward("none")
    for pin in PINS:
        pin(bwd)
    x, cot = case(36, B=2, T=5, H=2, nh=3, Dk=6, Dv=5)
    a, c = bwd(x, cot), c_backward(x, cot)
    for name in a:
        np.testing.assert_allclose(a[name], c[name], rtol=1e-11, atol=1e-12, err_msg=name)
