"""GPU parity of the recurrent (token-by-token) kernel, decode step and state I/O
against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from deltaproduct_householder_product_gb300 import workloads as W
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dp():
    from deltaproduct_householder_product_gb300 import build
    build.build()
    import deltaproduct_householder_product_gb300 as dp
    assert torch.cuda.is_available()
    return dp


def cuda(x):
    return {k: (None if v is None else v.cuda()) for k, v in x.items()}


def gpu_forward(dp, x, impl="recurrent", h0=True):
    xc = cuda(x)
    o, hf = dp.forward(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"],
                       xc["h0"] if h0 else None, impl=impl)
    torch.cuda.synchronize()
    return o, hf


def oracle_forward(x, h0=True):
    return oracle.forward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"] if h0 else None)


def test_tiny_fp32(dp):
    """The fp32 reference workload: B1 H2 T64 n_h2 D32, max abs error <= 1e-4."""
    x = W.make_inputs(W.TINY)
    o, hf = gpu_forward(dp, x)
    ro, rh = oracle_forward(x)
    assert_parity(o, ro, "f32", "o")
    assert_parity(hf, rh, "f32", "h_final")


@pytest.mark.parametrize("base", [W.BASE, W.NEARDUP, W.GATED, W.LONG], ids=lambda w: w.name)
def test_scaled_bf16(dp, base):
    w = base.scaled(B=2, H=3, T=150)
    x = W.make_inputs(w)
    o, hf = gpu_forward(dp, x)
    ro, rh = oracle_forward(x)
    assert_parity(o, ro, "bf16", "o")
    assert_parity(hf, rh, "bf16", "h_final")


@pytest.mark.parametrize("Dk,Dv,nh,dtype", [(64, 128, 1, "f32"), (128, 32, 4, "f32"),
                                            (32, 64, 3, "bf16"), (64, 64, 2, "bf16")])
def test_other_head_dims(dp, Dk, Dv, nh, dtype):
    w = W.GATED.scaled(B=1, H=2, T=37, Dk=Dk, Dv=Dv, nh=nh, dtype=dtype)
    x = W.make_inputs(w)
    o, hf = gpu_forward(dp, x)
    ro, rh = oracle_forward(x)
    assert_parity(o, ro, dtype, "o")
    assert_parity(hf, rh, dtype, "h_final")


def test_empty_sequence_copies_state(dp):
    w = W.GATED.scaled(B=2, H=2, T=0)
    x = W.make_inputs(w)
    o, hf = gpu_forward(dp, x)
    assert o.shape == (2, 0, 2, 128)
    assert torch.equal(hf.cpu(), x["h0"])
    x2 = dict(x)
    o, hf = gpu_forward(dp, x2, h0=False)
    assert torch.count_nonzero(hf) == 0


def test_h0_aliases_h_final(dp):
    w = W.GATED.scaled(B=1, H=2, T=40)
    x = W.make_inputs(w)
    xc = cuda(x)
    state = xc["h0"].clone()
    dp.forward(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], state, h_final=state,
               impl="recurrent")
    ro, rh = oracle_forward(x)
    assert_parity(state, rh, "bf16", "in-place state")


def test_decode_continues_forward(dp):
    """Prefill with dp_forward, then decode steps; compare every step to the oracle."""
    w = W.LONG.scaled(H=4, T=64)
    x = W.make_inputs(w)
    _, hf = gpu_forward(dp, x)
    _, rstate = oracle_forward(x)
    steps = 16
    d = W.make_decode_inputs(w, steps)
    dc = cuda(d)
    state = hf.clone()
    for s in range(steps):
        o = dp.decode_step(dc["q"][s], dc["k"][s], dc["v"][s], dc["beta"][s], None, state)
        ro, rstate = oracle.decode_step(d["q"][s], d["k"][s], d["v"][s], d["beta"][s], None, rstate)
        assert_parity(o, ro, "bf16", f"decode o step {s}")
    assert_parity(state, rstate, "bf16", "decode state")


def test_decode_gated_equals_forward_T1(dp):
    w = W.GATED.scaled(B=2, H=3, T=1)
    x = W.make_inputs(w)
    xc = cuda(x)
    o_f, hf = dp.forward(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], xc["h0"], impl="recurrent")
    state = xc["h0"].clone()
    o_d = dp.decode_step(xc["q"][:, 0], xc["k"][:, 0], xc["v"][:, 0], xc["beta"][:, 0],
                         xc["g"][:, 0], state)
    torch.cuda.synchronize()
    assert torch.equal(o_d, o_f[:, 0])
    assert torch.equal(state, hf)


@pytest.mark.parametrize("ext_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("transposed", [False, True])
def test_state_io(dp, ext_dtype, transposed):
    B, H, Dk, Dv = 2, 3, 64, 128
    src = torch.randn(B, H, Dk, Dv, generator=torch.Generator().manual_seed(1))
    ext = (src.transpose(-1, -2) if transposed else src).contiguous().to(ext_dtype).cuda()
    state = torch.full((B, H, Dk, Dv), 7.0, device="cuda")
    dp.state_io(dp.STATE_IMPORT, state, ext, transposed)
    ref = (src.to(ext_dtype).float())
    torch.cuda.synchronize()
    assert torch.equal(state.cpu(), ref)
    back = torch.zeros_like(ext)
    dp.state_io(dp.STATE_EXPORT, state, back, transposed)
    torch.cuda.synchronize()
    assert torch.equal(back, ext)
    dp.state_io(dp.STATE_ZERO, state)
    torch.cuda.synchronize()
    assert torch.count_nonzero(state) == 0


def test_status_clean_and_host_errors(dp):
    w = W.BASE.scaled(B=1, H=1, T=8)
    x = cuda(W.make_inputs(w))
    ws = torch.zeros(dp.workspace_size(1, 8, 1, 128, 128, 2), dtype=torch.uint8, device="cuda")
    dp.forward(x["q"], x["k"], x["v"], x["beta"], impl="recurrent", workspace=ws)
    dp.check_status(ws)
    with pytest.raises(dp.DPError) as e:                     # host tensor -> invalid argument
        dp._lib.lib()  # loaded
        import ctypes
        dims = dp._lib.make_dims(1, 8, 1, 128, 128, 2, torch.bfloat16)
        qh = x["q"].cpu()
        rc = dp._lib.lib().dp_forward(dims, ctypes.c_void_p(qh.data_ptr()), dp._lib._ptr(x["k"]),
                                      dp._lib._ptr(x["v"]), dp._lib._ptr(x["beta"]), None, None,
                                      dp._lib._ptr(x["q"]), None, dp._lib._ptr(ws), ws.numel(),
                                      dp._lib._stream(None))
        dp._lib._check(rc, "dp_forward")
    assert e.value.code in (1, 3)
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(dp.DPError) as e:
        dp.forward(x["q"], x["k"], x["v"], x["beta"], impl="recurrent", workspace=small)
    assert e.value.code == 4
