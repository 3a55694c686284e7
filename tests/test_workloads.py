"""Seeded synthetic inputs: shapes, dtypes, ranges and determinism (CPU)."""
import torch

from deltaproduct_householder_product_gb300 import workloads as W


def test_shapes_and_ranges_small():
    for base in W.ALL:
        w = base.scaled(B=1, T=40, H=2)
        x = W.make_inputs(w)
        assert x["q"].shape == (1, 40, 2, w.Dk)
        assert x["k"].shape == (1, 40, 2, w.nh, w.Dk)
        assert x["v"].shape == (1, 40, 2, w.nh, w.Dv)
        assert x["beta"].shape == (1, 40, 2, w.nh)
        assert x["q"].dtype == w.torch_dtype
        n = torch.linalg.vector_norm(x["k"].double(), dim=-1)
        assert torch.allclose(n, torch.ones_like(n), atol=1e-2)   # bf16-rounded unit keys
        b = x["beta"].double()
        assert b.min() >= 0 and b.max() <= w.beta_max
        if w.gated:
            assert x["g"].shape == (1, 40, 2) and x["g"].min() >= 0 and x["g"].max() <= 1
        else:
            assert x["g"] is None
        assert (x["h0"] is None) == (w.h0_std == 0)
        if x["h0"] is not None:
            assert x["h0"].dtype == torch.float32


def test_deterministic():
    w = W.GATED.scaled(B=1, T=16, H=2)
    a, b = W.make_inputs(w), W.make_inputs(w)
    for key in a:
        assert torch.equal(a[key], b[key])


def test_near_duplicates():
    w = W.NEARDUP.scaled(B=1, T=100, H=2)
    k = W.make_inputs(w)["k"].double()
    cos = (k[..., 0, :] * k[..., 1, :]).sum(-1)        # [B,T,H]
    per_head = (cos > 0.99).sum(dim=1)                 # tokens per (b,h)
    assert (per_head >= 20).all()                      # round(0.2*T) forced, plus chance
    assert cos.max() < 1.0 + 1e-2


def test_algorithmic_counts():
    # q + k + v + beta + o per token-head at n_h = 2, D = 128, bf16, plus the final state
    w = W.BASE
    per = (128 + 2 * 128 + 2 * 128 + 2 + 128) * 2
    assert W.algorithmic_bytes(w) == per * w.B * w.T * w.H + w.B * w.H * 128 * 128 * 4
    assert W.algorithmic_flops(w) == 10 * 128 * 128 * w.B * w.T * w.H
