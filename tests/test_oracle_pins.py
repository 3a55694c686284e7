"""Pins for the fp64 oracle: what the DeltaProduct paper and plain mathematics fix.

Every check is a function of a forward callable with the oracle's signature,
so the same checks run against (a) the C recurrence, (b) the numpy product
form, (c) the numpy chunked UT/WY form, and (d) deliberately broken copies of
the recurrence ("mutants", defined below on the CPU), each of which must fail
at least one pin. CPU only.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import chunkwise, product_form

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def one_head(fwd, k, v, beta, q=None, g=None, h0=None):
    """Run a single (batch, head) sequence. k [T,nh,Dk], v [T,nh,Dv], beta [T,nh]."""
    k = np.asarray(k, float)
    v = np.asarray(v, float)
    beta = np.asarray(beta, float)
    T, nh, Dk = k.shape
    Dv = v.shape[-1]
    if q is None:
        q = np.zeros((T, Dk))
    q = np.asarray(q, float)
    o, hf = fwd(q[None, :, None], k[None, :, None], v[None, :, None], beta[None, :, None],
                None if g is None else np.asarray(g, float)[None, :, None],
                None if h0 is None else np.asarray(h0, float)[None, None])
    return o[0, :, 0], hf[0, 0]


def transition(fwd, keys, betas, gate=None):
    """A_i of one token: run from H0 = I with zero values."""
    keys = np.asarray(keys, float)
    nh, Dk = keys.shape
    _, A = one_head(fwd, keys[None], np.zeros((1, nh, Dk)), np.asarray(betas, float)[None],
                    g=None if gate is None else [gate], h0=np.eye(Dk))
    return A


def unit(x):
    x = np.asarray(x, float)
    return x / np.linalg.norm(x)


def read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows[key] = np.array([float(x) for x in vals])
    return rows


# --------------------------------------------------------------------------
# pins, each a function of a forward callable
# --------------------------------------------------------------------------

def pin_mod3(fwd):
    """Sec.4 worked example: two beta=2 reflections give a 120-degree rotation."""
    gd = read_golden("mod3_rotation.txt")
    keys = np.stack([gd["k1"], gd["k2"]])
    A = transition(fwd, keys, gd["beta"])
    np.testing.assert_allclose(A, gd["F2F1"].reshape(2, 2), atol=1e-12)
    # one token at a time, carrying the 2x1 state (D_v = 1, B_i = 0)
    h = gd["state0"].reshape(2, 1)
    for step in range(1, 4):
        _, h = one_head(fwd, keys[None], np.zeros((1, 2, 1)), gd["beta"][None], h0=h)
        np.testing.assert_allclose(h[:, 0], gd[f"state{step}"], atol=1e-12)
    # the same three tokens in one call
    _, h3 = one_head(fwd, np.repeat(keys[None], 3, 0), np.zeros((3, 2, 1)),
                     np.repeat(gd["beta"][None], 3, 0), h0=gd["state0"].reshape(2, 1))
    np.testing.assert_allclose(h3[:, 0], gd["state3"], atol=1e-12)


def pin_nh2_closed_form(fwd, seed=1):
    """Sec.4: A_i for n_h = 2 incl. the beta1 beta2 (k2.k1) k2 k1^T cross term,
    and B_i = F2 C1 + C2."""
    rng = np.random.default_rng(seed)
    for _ in range(5):
        Dk, Dv = 5, 3
        k1, k2 = unit(rng.normal(size=Dk)), unit(rng.normal(size=Dk))
        b1, b2 = rng.uniform(0, 2, size=2)
        A = transition(fwd, [k1, k2], [b1, b2])
        I = np.eye(Dk)
        A_ref = (I - b1 * np.outer(k1, k1) - b2 * np.outer(k2, k2)
                 + b1 * b2 * (k2 @ k1) * np.outer(k2, k1))
        np.testing.assert_allclose(A, A_ref, atol=1e-12)
        v1, v2 = rng.normal(size=Dv), rng.normal(size=Dv)
        _, Bm = one_head(fwd, np.stack([k1, k2])[None], np.stack([v1, v2])[None],
                         np.array([[b1, b2]]))
        B_ref = (I - b2 * np.outer(k2, k2)) @ (b1 * np.outer(k1, v1)) + b2 * np.outer(k2, v2)
        np.testing.assert_allclose(Bm, B_ref, atol=1e-12)


def pin_identical_keys(fwd, seed=2):
    """App.A: identical keys collapse to one factor with beta_eff = 1 - prod(1 - beta_j);
    and two beta=2 reflections on the same key give the identity."""
    rng = np.random.default_rng(seed)
    Dk = 6
    k = unit(rng.normal(size=Dk))
    for nh in (2, 3, 4):
        betas = rng.uniform(0, 2, size=nh)
        A = transition(fwd, np.repeat(k[None], nh, 0), betas)
        beff = 1.0 - np.prod(1.0 - betas)
        np.testing.assert_allclose(A, np.eye(Dk) - beff * np.outer(k, k), atol=1e-12)
    A = transition(fwd, np.stack([k, k]), [2.0, 2.0])
    np.testing.assert_allclose(A, np.eye(Dk), atol=1e-12)


def pin_orthogonal_keys(fwd, seed=3):
    """App.A: mutually orthogonal keys give A = I - sum_j beta_j k_j k_j^T (symmetric)."""
    rng = np.random.default_rng(seed)
    Dk = 6
    Qm, _ = np.linalg.qr(rng.normal(size=(Dk, Dk)))
    keys = Qm[:, :3].T
    betas = rng.uniform(0, 2, size=3)
    A = transition(fwd, keys, betas)
    ref = np.eye(Dk) - sum(b * np.outer(kk, kk) for b, kk in zip(betas, keys))
    np.testing.assert_allclose(A, ref, atol=1e-12)
    np.testing.assert_allclose(A, A.T, atol=1e-12)


def pin_exact_recall(fwd, seed=4):
    """Sec.2 after Eq.(2): with a unit key and beta = 1 the state maps that key to v."""
    rng = np.random.default_rng(seed)
    T, nh, Dk, Dv = 6, 3, 8, 5
    k = np.stack([[unit(rng.normal(size=Dk)) for _ in range(nh)] for _ in range(T)])
    v = rng.normal(size=(T, nh, Dv))
    beta = rng.uniform(0, 2, size=(T, nh))
    beta[:, -1] = 1.0
    q = k[:, -1, :]                          # read with the last key of each token
    o, _ = one_head(fwd, k, v, beta, q=q, h0=rng.normal(size=(Dk, Dv)))
    np.testing.assert_allclose(o, v[:, -1, :], atol=1e-12)


def pin_rank(fwd, seed=5):
    """Sec.4: rank(A_i - I) <= n_h; gated: rank(A_i - g_i I) <= n_h."""
    rng = np.random.default_rng(seed)
    Dk = 8
    for nh in (1, 2, 3, 4):
        keys = [unit(rng.normal(size=Dk)) for _ in range(nh)]
        betas = rng.uniform(0.1, 2, size=nh)
        A = transition(fwd, keys, betas)
        s = np.linalg.svd(A - np.eye(Dk), compute_uv=False)
        assert np.sum(s > 1e-10) == nh
        gate = rng.uniform(0.2, 0.9)
        Ag = transition(fwd, keys, betas, gate=gate)
        s = np.linalg.svd(Ag - gate * np.eye(Dk), compute_uv=False)
        assert np.sum(s > 1e-10) <= nh
        np.testing.assert_allclose(Ag, gate * A, atol=1e-12)


def pin_stability(fwd, seed=6):
    """Sec.4 / App.B.6: ||A_t ... A_1||_2 <= 1 for unit keys and beta in [0,2]."""
    rng = np.random.default_rng(seed)
    for trial in range(20):
        Dk = int(rng.integers(2, 9))
        nh = int(rng.integers(1, 5))
        T = int(rng.integers(1, 65))
        k = rng.normal(size=(T, nh, Dk))
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        beta = rng.uniform(0, 2, size=(T, nh))
        if trial % 4 == 0:
            beta[:] = 2.0                    # pure reflections: norm exactly 1
        _, P = one_head(fwd, k, np.zeros((T, nh, Dk)), beta, h0=np.eye(Dk))
        assert np.linalg.norm(P, 2) <= 1.0 + 1e-12
        if trial % 4 == 0:
            np.testing.assert_allclose(P.T @ P, np.eye(Dk), atol=1e-10)   # orthogonal


def pin_rotation_condition(fwd, seed=7):
    """App.A: in span(k1,k2), tau = 2 - b1 - b2 + b1 b2 c^2 and delta = (1-b1)(1-b2)
    are the trace and determinant, and tau^2 - 4 delta < 0 iff eigenvalues are complex."""
    rng = np.random.default_rng(seed)
    seen = {True: 0, False: 0}
    for _ in range(200):
        th = rng.uniform(0, np.pi)
        k1, k2 = np.array([1.0, 0.0]), np.array([np.cos(th), np.sin(th)])
        b1, b2 = rng.uniform(0, 2, size=2)
        A = transition(fwd, [k1, k2], [b1, b2])
        c = k1 @ k2
        tau = 2 - b1 - b2 + b1 * b2 * c * c
        delta = (1 - b1) * (1 - b2)
        assert abs(np.trace(A) - tau) < 1e-12 and abs(np.linalg.det(A) - delta) < 1e-12
        disc = tau * tau - 4 * delta
        if abs(disc) < 1e-9:
            continue
        ev = np.linalg.eigvals(A)
        cplx = bool(np.max(np.abs(ev.imag)) > 1e-12)
        assert cplx == (disc < 0)
        seen[cplx] += 1
    assert seen[True] > 5 and seen[False] > 5


def pin_permutation(fwd, seed=8):
    """Thm.1 construction (App.B.2): transposition reflections k = (e_a - e_b)/sqrt(2),
    beta = 2, B_i = 0 act on H0 = (1..n)^T as the permutation they compose."""
    rng = np.random.default_rng(seed)
    n = 5
    for _ in range(10):
        swaps = [tuple(rng.choice(n, size=2, replace=False)) for _ in range(n - 1)]
        keys = []
        for a, b in swaps:
            kk = np.zeros(n)
            kk[a], kk[b] = 1 / math.sqrt(2), -1 / math.sqrt(2)
            keys.append(kk)
        h0 = np.arange(1, n + 1, dtype=float).reshape(n, 1)
        _, h = one_head(fwd, np.array(keys)[None], np.zeros((1, n - 1, 1)),
                        np.full((1, n - 1), 2.0), h0=h0)
        ref = list(range(1, n + 1))
        for a, b in swaps:                   # brute force: apply swaps in order
            ref[a], ref[b] = ref[b], ref[a]
        np.testing.assert_allclose(h[:, 0], ref, atol=1e-12)


def pin_reset(fwd, seed=9):
    """Sec.4.1 / App.B.3: g_t = 0 wipes the old state; the run from t on equals a
    fresh run with H0 = 0."""
    rng = np.random.default_rng(seed)
    T, nh, Dk, Dv, t0 = 12, 2, 6, 4, 5
    k = rng.normal(size=(T, nh, Dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.normal(size=(T, nh, Dv))
    beta = rng.uniform(0, 2, size=(T, nh))
    q = rng.normal(size=(T, Dk))
    g = rng.uniform(0.5, 1, size=T)
    g[t0] = 0.0
    o, hf = one_head(fwd, k, v, beta, q=q, g=g, h0=rng.normal(size=(Dk, Dv)))
    o2, hf2 = one_head(fwd, k[t0:], v[t0:], beta[t0:], q=q[t0:], g=g[t0:])
    np.testing.assert_allclose(o[t0:], o2, atol=1e-12)
    np.testing.assert_allclose(hf, hf2, atol=1e-12)


def pin_forgetting(fwd, seed=10):
    """Sec.5.3: beta = 1 projections on an orthonormal basis with v = 0 clear any
    state within ceil(D_k / n_h) tokens."""
    rng = np.random.default_rng(seed)
    Dk, Dv, nh = 7, 3, 3
    T = math.ceil(Dk / nh)
    Qm, _ = np.linalg.qr(rng.normal(size=(Dk, Dk)))
    keys = np.zeros((T, nh, Dk))
    for idx in range(T * nh):
        if idx < Dk:
            keys[idx // nh, idx % nh] = Qm[:, idx]
    beta = np.ones((T, nh))
    beta[keys.sum(-1) == 0] = 0.0          # padding steps do nothing
    _, h = one_head(fwd, keys, np.zeros((T, nh, Dv)), beta, h0=rng.normal(size=(Dk, Dv)))
    np.testing.assert_allclose(h, 0.0, atol=1e-12)


def pin_beta_zero(fwd, seed=11):
    """beta = 0 makes every factor the identity: o_t = (prod g) H0^T q_t."""
    rng = np.random.default_rng(seed)
    T, nh, Dk, Dv = 9, 2, 5, 4
    k = rng.normal(size=(T, nh, Dk))
    v = rng.normal(size=(T, nh, Dv))
    q = rng.normal(size=(T, Dk))
    g = rng.uniform(0.3, 1, size=T)
    h0 = rng.normal(size=(Dk, Dv))
    o, hf = one_head(fwd, k, v, np.zeros((T, nh)), q=q, g=g, h0=h0)
    cg = np.cumprod(g)
    np.testing.assert_allclose(o, cg[:, None] * (q @ h0), atol=1e-12)
    np.testing.assert_allclose(hf, cg[-1] * h0, atol=1e-12)


def pin_extended_sequence(fwd, seed=12):
    """Sec.5.1: DeltaProduct_{n_h} equals DeltaNet (n_h = 1) on the interleaved
    T*n_h sequence with the gate expanded to (g_1,1,..,1,g_2,..) and only the last
    output of each token kept."""
    rng = np.random.default_rng(seed)
    T, nh, Dk, Dv = 7, 3, 6, 4
    k = rng.normal(size=(T, nh, Dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.normal(size=(T, nh, Dv))
    beta = rng.uniform(0, 2, size=(T, nh))
    q = rng.normal(size=(T, Dk))
    g = rng.uniform(0.3, 1, size=T)
    h0 = rng.normal(size=(Dk, Dv))
    o, hf = one_head(fwd, k, v, beta, q=q, g=g, h0=h0)
    ge = np.ones(T * nh)
    ge[0::nh] = g
    qe = np.repeat(q, nh, axis=0)
    oe, hfe = one_head(fwd, k.reshape(T * nh, 1, Dk), v.reshape(T * nh, 1, Dv),
                       beta.reshape(T * nh, 1), q=qe, g=ge, h0=h0)
    np.testing.assert_allclose(o, oe[nh - 1::nh], atol=1e-12)
    np.testing.assert_allclose(hf, hfe, atol=1e-12)


def pin_linearity(fwd, seed=13):
    """For fixed keys, betas and gates the map (H0, V) -> (o, H_T) is linear."""
    rng = np.random.default_rng(seed)
    T, nh, Dk, Dv = 8, 2, 5, 3
    k = rng.normal(size=(T, nh, Dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    beta = rng.uniform(0, 2, size=(T, nh))
    q = rng.normal(size=(T, Dk))
    g = rng.uniform(0.3, 1, size=T)
    v1, v2 = rng.normal(size=(2, T, nh, Dv))
    h1, h2 = rng.normal(size=(2, Dk, Dv))
    a, b = 0.7, -1.3
    o1, f1 = one_head(fwd, k, v1, beta, q=q, g=g, h0=h1)
    o2, f2 = one_head(fwd, k, v2, beta, q=q, g=g, h0=h2)
    o3, f3 = one_head(fwd, k, a * v1 + b * v2, beta, q=q, g=g, h0=a * h1 + b * h2)
    np.testing.assert_allclose(o3, a * o1 + b * o2, atol=1e-12)
    np.testing.assert_allclose(f3, a * f1 + b * f2, atol=1e-12)


PINS = [pin_mod3, pin_nh2_closed_form, pin_identical_keys, pin_orthogonal_keys,
        pin_exact_recall, pin_rank, pin_stability, pin_rotation_condition,
        pin_permutation, pin_reset, pin_forgetting, pin_beta_zero,
        pin_extended_sequence, pin_linearity]


# --------------------------------------------------------------------------
# the forward callables under test
# --------------------------------------------------------------------------

def c_oracle(q, k, v, beta, g=None, h0=None):
    return oracle.forward(q, k, v, beta, g, h0, threads=2)


def chunked(chunk, token_aligned=False):
    def fwd(q, k, v, beta, g=None, h0=None):
        return chunkwise.forward(q, k, v, beta, g, h0, chunk=chunk, token_aligned=token_aligned)
    fwd.__name__ = f"chunkwise_c{chunk}_{'tok' if token_aligned else 'ext'}"
    return fwd


IMPLS = {
    "c_recurrence": c_oracle,
    "numpy_product_form": product_form.forward,
    "chunkwise_c4_ext": chunked(4),
    "chunkwise_c5_tok": chunked(5, token_aligned=True),
    "chunkwise_c64_ext": chunked(64),
}


@pytest.mark.parametrize("impl", list(IMPLS))
@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin, impl):
    pin(IMPLS[impl])


# --------------------------------------------------------------------------
# mutants: plausible mistakes planted in a CPU copy of the recurrence; every
# one must be caught by at least one pin
# --------------------------------------------------------------------------

MUTANTS = ["substep_order_reversed", "error_sign_flipped", "no_error_correction",
           "gate_after_updates", "gate_every_substep", "readout_before_updates",
           "beta_squared", "initial_state_dropped", "readout_after_first_substep"]


def mutant(kind):
    def fwd(q, k, v, beta, g=None, h0=None):
        q, k, v, beta = (np.asarray(x, float) for x in (q, k, v, beta))
        B, T, H, nh, Dk = k.shape
        Dv = v.shape[-1]
        o = np.zeros((B, T, H, Dv))
        hf = np.zeros((B, H, Dk, Dv))
        for b in range(B):
            for h in range(H):
                S = np.zeros((Dk, Dv))
                if h0 is not None and kind != "initial_state_dropped":
                    S = np.array(h0[b, h], float)
                for t in range(T):
                    gt = None if g is None else float(g[b, t, h])
                    if kind == "readout_before_updates":
                        o[b, t, h] = S.T @ q[b, t, h]
                    if gt is not None and kind not in ("gate_after_updates", "gate_every_substep"):
                        S = gt * S
                    order = range(nh - 1, -1, -1) if kind == "substep_order_reversed" else range(nh)
                    for n, j in enumerate(order):
                        if gt is not None and kind == "gate_every_substep":
                            S = gt * S
                        kk, vv, bb = k[b, t, h, j], v[b, t, h, j], beta[b, t, h, j]
                        if kind == "beta_squared":
                            bb = bb * bb
                        if kind == "error_sign_flipped":
                            e = vv + S.T @ kk
                        elif kind == "no_error_correction":
                            e = vv
                        else:
                            e = vv - S.T @ kk
                        S = S + bb * np.outer(kk, e)
                        if kind == "readout_after_first_substep" and n == 0:
                            o[b, t, h] = S.T @ q[b, t, h]
                    if gt is not None and kind == "gate_after_updates":
                        S = gt * S
                    if kind not in ("readout_before_updates", "readout_after_first_substep"):
                        o[b, t, h] = S.T @ q[b, t, h]
                hf[b, h] = S
        return o, hf
    return fwd


@pytest.mark.parametrize("kind", MUTANTS)
def test_mutant_is_caught(kind):
    fwd = mutant(kind)
    caught = []
    for pin in PINS:
        try:
            pin(fwd)
        except (AssertionError, ValueError, np.linalg.LinAlgError):
            caught.append(pin.__name__)
    assert caught, f"mutant {kind} passed every pin"


def test_unmutated_copy_passes():
    """The mutant harness itself is sound: with no mutation it passes every pin."""
    fwd = mutant("none")
    for pin in PINS:
        pin(fwd)


# --------------------------------------------------------------------------
# cross-checks of the three restatements on random inputs
# --------------------------------------------------------------------------

def random_case(rng, B, T, H, nh, Dk, Dv, gated, with_h0, zero_gates=0):
    q = rng.normal(size=(B, T, H, Dk))
    k = rng.normal(size=(B, T, H, nh, Dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.normal(size=(B, T, H, nh, Dv))
    beta = rng.uniform(0, 2, size=(B, T, H, nh))
    g = rng.uniform(0.6, 1.0, size=(B, T, H)) if gated else None
    if gated and zero_gates:
        idx = rng.choice(T, size=zero_gates, replace=False)
        g[:, idx, :] = 0.0
    h0 = rng.normal(size=(B, H, Dk, Dv)) if with_h0 else None
    return q, k, v, beta, g, h0


@pytest.mark.parametrize("nh", [1, 2, 3, 4])
@pytest.mark.parametrize("gated", [False, True])
def test_product_form_matches_recurrence(nh, gated):
    rng = np.random.default_rng(100 + nh)
    case = random_case(rng, 2, 11, 2, nh, 6, 5, gated, True, zero_gates=1 if gated else 0)
    o1, f1 = oracle.forward(*case)
    o2, f2 = product_form.forward(*case)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(f1, f2, atol=1e-12)


@pytest.mark.parametrize("nh", [1, 2, 3, 4])
@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("chunk,tok", [(16, False), (16, True), (64, True), (7, False)])
def test_chunkwise_matches_recurrence(nh, gated, chunk, tok):
    rng = np.random.default_rng(200 + nh)
    case = random_case(rng, 1, 45, 2, nh, 16, 8, gated, gated, zero_gates=2 if gated else 0)
    o1, f1 = oracle.forward(*case)
    o2, f2 = chunkwise.forward(*case, chunk=chunk, token_aligned=tok)
    scale = max(1.0, np.abs(o1).max())
    np.testing.assert_allclose(o1, o2, atol=1e-10 * scale)
    np.testing.assert_allclose(f1, f2, atol=1e-10 * max(1.0, np.abs(f1).max()))


def test_decode_step_equals_forward():
    rng = np.random.default_rng(300)
    q, k, v, beta, g, h0 = random_case(rng, 2, 5, 3, 3, 8, 4, True, True)
    o, hf = oracle.forward(q, k, v, beta, g, h0)
    state = h0
    for t in range(5):
        ot, state = oracle.decode_step(q[:, t], k[:, t], v[:, t], beta[:, t], g[:, t], state)
        np.testing.assert_allclose(ot, o[:, t], atol=1e-12)
    np.testing.assert_allclose(state, hf, atol=1e-12)


def test_empty_sequence_returns_initial_state():
    rng = np.random.default_rng(301)
    q, k, v, beta, g, h0 = random_case(rng, 1, 0, 2, 2, 4, 4, False, True)
    o, hf = oracle.forward(q, k, v, beta, g, h0)
    assert o.shape == (1, 0, 2, 4)
    np.testing.assert_array_equal(hf, h0)


def test_state_carry_equals_single_call():
    """Splitting the sequence and carrying the state is exact (associativity, Sec.2 Eq.(1))."""
    rng = np.random.default_rng(302)
    q, k, v, beta, g, h0 = random_case(rng, 1, 40, 2, 3, 8, 6, True, True)
    o, hf = oracle.forward(q, k, v, beta, g, h0)
    state, outs = h0, []
    for s in range(0, 40, 10):
        sl = slice(s, s + 10)
        os_, state = oracle.forward(q[:, sl], k[:, sl], v[:, sl], beta[:, sl], g[:, sl], state)
        outs.append(os_)
    np.testing.assert_allclose(np.concatenate(outs, 1), o, atol=1e-12)
    np.testing.assert_allclose(state, hf, atol=1e-12)
