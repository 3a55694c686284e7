"""Pins of the prologue oracle (oracle.prologue), CPU only: each map against
a library routine or a closed form, and the composition with the recurrence
against the recurrence run on the mapped inputs."""
import numpy as np
import pytest
import torch

import oracle
from oracle import prologue as P


def test_silu_matches_library():
    x = np.linspace(-12, 12, 1001)
    ref = torch.nn.functional.silu(torch.from_numpy(x)).numpy()
    np.testing.assert_allclose(P.silu(x), ref, rtol=1e-14, atol=1e-15)


def test_sigmoid_closed_forms():
    assert P.sigmoid(0.0) == 0.5
    np.testing.assert_allclose(P.sigmoid(np.log(3.0)), 0.75, rtol=1e-15)
    x = np.linspace(-30, 30, 61)
    np.testing.assert_allclose(P.sigmoid(x) + P.sigmoid(-x), 1.0, rtol=1e-15)


def test_key_map_unit_norm_and_direction():
    rng = np.random.default_rng(0)
    k = rng.normal(size=(7, 3, 16))
    q, kk, b, g = P.apply(P.KEY_SILU_L2, k[:, 0], k, np.zeros((7, 3)))
    np.testing.assert_allclose(np.linalg.norm(kk, axis=-1), 1.0, rtol=1e-14)
    s = P.silu(k)
    # parallel to SiLU(k) with a positive factor
    np.testing.assert_allclose(kk * np.linalg.norm(s, axis=-1, keepdims=True), s, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(q, k[:, 0])          # queries untouched without QUERY_L2
    z, _, _, _ = P.apply(P.QUERY_L2, np.zeros((2, 4)), k, np.zeros((7, 3)))
    assert np.all(z == 0)                               # a zero row stays zero


@pytest.mark.parametrize("flag,lo,hi", [(P.BETA_SIGMOID, 0.0, 1.0), (P.BETA_2SIGMOID, 0.0, 2.0)])
def test_beta_maps_ranges(flag, lo, hi):
    x = np.linspace(-20, 20, 401)
    _, _, b, _ = P.apply(flag, np.zeros(2), np.zeros(2), x)
    assert np.all(b > lo) and np.all(b < hi)
    np.testing.assert_allclose(b[200], (lo + hi) / 2, rtol=1e-15)


def test_prologue_then_recurrence():
    rng = np.random.default_rng(1)
    B, T, H, nh, D = 1, 5, 2, 2, 6
    q, k = rng.normal(size=(B, T, H, D)), rng.normal(size=(B, T, H, nh, D))
    v, b, g = rng.normal(size=(B, T, H, nh, D)), rng.normal(size=(B, T, H, nh)), rng.normal(size=(B, T, H))
    flags = P.KEY_SILU_L2 | P.QUERY_L2 | P.BETA_2SIGMOID | P.GATE_SIGMOID
    o, hf = P.forward(flags, q, k, v, b, g, threads=1)
    qn = q / np.linalg.norm(q, axis=-1, keepdims=True)
    sk = k / (1 + np.exp(-k))
    kn = sk / np.linalg.norm(sk, axis=-1, keepdims=True)
    o2, hf2 = oracle.forward(qn, kn, v, 2 / (1 + np.exp(-b)), 1 / (1 + np.exp(-g)), None, threads=1)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(hf, hf2, rtol=1e-12, atol=1e-12)


def test_bf16_operand_rounding():
    """round_bf16 is round-to-nearest-even onto bfloat16's grid: exact on
    representable values, half-way cases to the even neighbour."""
    one_ulp = 2.0 ** -7                        # bf16 spacing in [1, 2)
    xs = np.array([1.0, 1.0 + one_ulp, 1.0 + one_ulp / 2, 1.0 + 1.5 * one_ulp, 1.0 + 0.3 * one_ulp])
    np.testing.assert_array_equal(P.round_bf16(xs), [1.0, 1.0 + one_ulp, 1.0, 1.0 + 2 * one_ulp, 1.0])
