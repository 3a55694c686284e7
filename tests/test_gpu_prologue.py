"""GPU parity of the fused input prologue (dims.prologue: SiLU + L2 keys, L2
queries, sigmoid / 2 sigmoid betas, sigmoid gates applied by the kernels as
they load their inputs) against the fp64 oracle (oracle.prologue.forward on
the same raw inputs), through the C ABI; the standalone dp_prologue against
oracle.prologue.apply; the modes of the chunk path bit-identical to one
another with the prologue; the decode step and packed sequences with it.

Tolerance: the bf16 rule of the forward (max|err| <= 2e-2 RMS(ref) on
outputs and final states), against the oracle that rounds the mapped keys
and queries to bf16 as the library states for bf16 inputs (the kernel
rounds its fp32 map, the oracle its fp64 map: they differ by at most one
bf16 step on a few elements). dp_prologue's outputs are
compared element-wise with the fp64 maps within one bf16 rounding of the
fp32 result: |err| <= 2^-8 |ref| + 1e-6.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import prologue as OP
from deltaproduct_householder_product_gb300 import workloads as W
from tests.parity import assert_parity, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dp():
    from deltaproduct_householder_product_gb300 import build
    build.build()
    import deltaproduct_householder_product_gb300 as dp
    assert torch.cuda.is_available()
    return dp


def raw_case(w):
    x = W.make_raw_inputs(w)
    return x, {k: (None if v is None else v.cuda()) for k, v in x.items()}, W.prologue_flags(w)


def record_bytes(flags):
    """Bytes per chunk record: 18688, plus the mapped K and Q rows (12288)
    with a key or query prologue."""
    return 18688 + (12288 if flags & 3 else 0)


def run(dp, xc, flags, path, out_dtype=torch.float32):
    """path: "coop" (fast workspace: one cooperative launch), "split" (the
    records only: prep kernel + state-pass kernel), "fused" (minimum
    workspace), "recurrent"."""
    B, T, H, nh, Dk = xc["k"].shape
    ws_lo = dp.workspace_size(B, T, H, Dk, Dk, nh)
    ct = min(16, 32 // nh)
    size = {"fused": ws_lo, "recurrent": ws_lo, "coop": dp.workspace_size(B, T, H, Dk, Dk, nh, fast=True),
            "split": ws_lo + ((B * H * (-(-T // ct)) * record_bytes(flags) + 255) // 256) * 256}[path]
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    o, hf = dp.forward(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], xc["h0"], workspace=ws,
                       impl="recurrent" if path == "recurrent" else "chunk_tc", out_dtype=out_dtype,
                       prologue=flags)
    dp.check_status(ws)
    return o, hf


CASES = [("base", W.BASE.scaled(B=2, H=2, T=150)), ("gated", W.GATED.scaled(B=1, H=3, T=97)),
         ("long-nh3", W.LONG.scaled(B=1, H=2, T=64))]


@pytest.mark.parametrize("path", ["coop", "split", "fused", "recurrent"])
@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_fused_prologue_parity(dp, name, w, path):
    x, xc, flags = raw_case(w)
    o, hf = run(dp, xc, flags, path)
    ro, rh = OP.forward(flags, x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], operand_dtype="bf16")
    assert_parity(o, ro, "bf16", f"{name} {path} o")
    assert_parity(hf, rh, "bf16", f"{name} {path} h_final")


def test_prologue_modes_bitwise(dp):
    x, xc, flags = raw_case(W.GATED.scaled(B=2, H=2, T=80, nh=2))
    f = run(dp, xc, flags, "fused")
    for path in ("coop", "split"):
        a = run(dp, xc, flags, path)
        assert torch.equal(a[0], f[0]) and torch.equal(a[1], f[1]), path


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_standalone_prologue_matches_maps(dp, name, w):
    x, xc, flags = raw_case(w)
    q, k, b, g = dp.prologue(xc["q"], xc["k"], xc["beta"], xc["g"], flags=flags)
    rq, rk, rb, rg = OP.apply(flags, x["q"].double().numpy(), x["k"].double().numpy(),
                              x["beta"].double().numpy(), None if x["g"] is None else x["g"].double().numpy())
    for got, ref, what in ((q, rq, "q"), (k, rk, "k"), (b, rb, "beta"), (g, rg, "g")):
        if ref is None:
            continue
        d = np.abs(to_np(got) - ref)
        assert np.all(d <= 2.0 ** -8 * np.abs(ref) + 1e-6), (what, float(d.max()))


def test_unfused_equals_fused_up_to_rounding(dp):
    w = W.BASE.scaled(B=2, H=2, T=130)
    x, xc, flags = raw_case(w)
    o_f, h_f = run(dp, xc, flags, "coop")
    q, k, b, g = dp.prologue(xc["q"], xc["k"], xc["beta"], xc["g"], flags=flags)
    o_u, h_u = dp.forward(q, k, xc["v"], b, g, xc["h0"], impl="chunk_tc", out_dtype=torch.float32)
    assert_parity(o_u, to_np(o_f), "bf16", "unfused vs fused o")
    assert_parity(h_u, to_np(h_f), "bf16", "unfused vs fused h_final")


def test_decode_step_with_prologue(dp):
    w = W.GATED.scaled(B=2, H=2, T=6, nh=3)
    x, xc, flags = raw_case(w)
    state = xc["h0"].clone()
    outs = []
    for t in range(w.T):
        outs.append(dp.decode_step(xc["q"][:, t].contiguous(), xc["k"][:, t].contiguous(),
                                   xc["v"][:, t].contiguous(), xc["beta"][:, t].contiguous(),
                                   xc["g"][:, t].contiguous(), state, out_dtype=torch.float32, prologue=flags))
    ro, rh = OP.forward(flags, x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], operand_dtype="bf16")
    assert_parity(torch.stack(outs, 1), ro, "bf16", "decode o")
    assert_parity(state, rh, "bf16", "decode state")


@pytest.mark.parametrize("path", ["coop", "recurrent"])
def test_packed_sequences_with_prologue(dp, path):
    w = W.GATED.scaled(B=1, H=2, T=90, nh=2, h0_std=0.0)
    x, xc, flags = raw_case(w)
    lengths = [17, 0, 40, 33]
    cu = torch.tensor([0, 17, 17, 57, 90], dtype=torch.int32, device="cuda")
    pk = lambda t: None if t is None else t[0].contiguous()
    impl = "recurrent" if path == "recurrent" else "chunk_tc"
    o, hf = dp.forward_varlen(pk(xc["q"]), pk(xc["k"]), pk(xc["v"]), pk(xc["beta"]), pk(xc["g"]), None,
                              cu_seqlens=cu, max_seqlen=40, impl=impl, out_dtype=torch.float32, prologue=flags)
    a = 0
    for s, n in enumerate(lengths):
        sl = lambda t: None if t is None else t[:, a:a + n]
        ro, rh = OP.forward(flags, sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["beta"]), sl(x["g"]), None,
                            operand_dtype="bf16")
        if n:
            assert_parity(o[a:a + n], ro[0], "bf16", f"seq {s} o")
        assert_parity(hf[s], rh[0], "bf16", f"seq {s} h_final")
        a += n


def test_forward_path_with_prologue(dp):
    """The records-only workspace (with the mapped K/Q rows) selects the
    two-launch split mode, the fast size the cooperative one."""
    x, xc, flags = raw_case(W.BASE.scaled(B=2, H=3, T=100))
    B, T, H, nh, Dk = xc["k"].shape
    lo = dp.workspace_size(B, T, H, Dk, Dk, nh)
    rec = lo + ((B * H * (-(-T // 16)) * record_bytes(flags) + 255) // 256) * 256
    assert dp.forward_path(B, T, H, Dk, Dk, nh, rec, prologue=flags) == "chunk_split"
    assert dp.forward_path(B, T, H, Dk, Dk, nh, rec - 256, prologue=flags) == "chunk_fused"
    fast = dp.workspace_size(B, T, H, Dk, Dk, nh, fast=True, prologue=flags)
    assert dp.forward_path(B, T, H, Dk, Dk, nh, fast, prologue=flags) == "chunk_coop"
