"""GPU parity of the OSDN write-key variant through the C ABI: phase 1
(dp_osdn_write_keys) against oracle.osdn.dscan, phase 2
(dp_forward_write_keys, recurrent kernel and tensor-core chunk path in
both split modes) against the C oracle fed the same write keys, both
phases against oracle.osdn.forward, the eta = 0 reduction to the plain
recurrence (bit for bit), with and without APF retention, and sampled heads
of the bench-sized workload.

Tolerances: the scan runs in fp32 (the oracle in fp64); the write keys are
rounded to the input dtype, so |kw - ref| <= 2^-8 |ref| + 1e-5 (one bf16
step plus the fp32 drift of d over the rows), and d_final within 1e-4
relative. The forward follows the bf16 rule (max|err| <= 2e-2 RMS(ref))."""
import numpy as np
import pytest
import torch

import oracle
from oracle import osdn as OS
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


def inputs(w, apf_seed=None, d0=False):
    x = W.make_inputs(w)
    xc = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    r = rc = d = dc = None
    if apf_seed is not None:
        gen = torch.Generator().manual_seed(apf_seed)
        r = torch.sigmoid(torch.randn(w.B, w.T, w.H, generator=gen) + 2.0).to(w.torch_dtype)
        rc = r.cuda()
    if d0:
        gen = torch.Generator().manual_seed(7)
        d = 0.5 + 1.5 * torch.rand(w.B, w.H, w.Dk, generator=gen)
        dc = d.cuda()
    return x, xc, r, rc, d, dc


def check_scan(kw, dfin, ref_kw, ref_d):
    d = np.abs(to_np(kw) - ref_kw)
    assert np.all(d <= 2.0 ** -8 * np.abs(ref_kw) + 1e-5), float(d.max())
    np.testing.assert_allclose(to_np(dfin), ref_d, rtol=1e-4, atol=1e-5)


CASES = [("base", W.BASE.scaled(B=2, H=2, T=120), None, False, 0.003),
         ("gated-apf-d0", W.GATED.scaled(B=1, H=3, T=90), 11, True, 0.003),
         ("long-nh3-eta", W.LONG.scaled(B=1, H=2, T=200), None, False, 0.05),
         ("tiny-f32-apf", W.TINY.scaled(T=50), 12, False, 0.2)]


@pytest.mark.parametrize("name,w,apf,d0,eta", CASES, ids=[c[0] for c in CASES])
def test_osdn_parity(dp, name, w, apf, d0, eta):
    x, xc, r, rc, d, dc = inputs(w, apf, d0)
    kw, dfin = dp.osdn_write_keys(xc["k"], xc["beta"], rc, dc, eta=eta)
    ref_kw, ref_d = OS.dscan(x["k"], x["beta"], r, d, eta=eta)
    check_scan(kw, dfin, ref_kw, ref_d)
    o, hf = dp.forward_write_keys(xc["q"], xc["k"], kw, xc["v"], xc["beta"], xc["g"], xc["h0"], impl="recurrent",
                                  out_dtype=torch.float32)
    # phase 2 alone: the oracle on the kernel's own write keys
    ro, rh = oracle.forward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], kw=kw.cpu())
    kind = "f32" if w.dtype == "f32" else "bf16"
    assert_parity(o, ro, kind, f"{name} o (phase 2)")
    assert_parity(hf, rh, kind, f"{name} h_final (phase 2)")
    # both phases against the fp64 scan and recurrence
    ro2, rh2, _, _ = OS.forward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], r, d, eta=eta)
    assert_parity(o, ro2, "bf16", f"{name} o")
    assert_parity(hf, rh2, "bf16", f"{name} h_final")


def test_eta_zero_is_plain_forward(dp):
    w = W.GATED.scaled(B=2, H=2, T=70, nh=3)
    x, xc, *_ = inputs(w)
    kw, dfin = dp.osdn_write_keys(xc["k"], xc["beta"], eta=0.0)
    assert torch.equal(kw, xc["k"]) and torch.all(dfin == 1)
    o1, h1 = dp.forward_write_keys(xc["q"], xc["k"], kw, xc["v"], xc["beta"], xc["g"], xc["h0"], impl="recurrent",
                                   out_dtype=torch.float32)
    o2, h2 = dp.forward(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], xc["h0"], impl="recurrent",
                        out_dtype=torch.float32)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_scan_carries_across_calls(dp):
    """Two calls on halves, the second from the first's d_final, equal one call."""
    w = W.BASE.scaled(B=1, H=2, T=64)
    x, xc, *_ = inputs(w)
    kw, d = dp.osdn_write_keys(xc["k"], xc["beta"], eta=0.05)
    h = lambda t, a, b: t[:, a:b].contiguous()
    kw1, d1 = dp.osdn_write_keys(h(xc["k"], 0, 32), h(xc["beta"], 0, 32), eta=0.05)
    kw2, d2 = dp.osdn_write_keys(h(xc["k"], 32, 64), h(xc["beta"], 32, 64), None, d1, eta=0.05)
    assert torch.equal(torch.cat([kw1, kw2], 1), kw) and torch.equal(d2, d)


def test_osdn_full_size_sampled_heads(dp):
    """Bench workload (B4 H8 T2048 n_h 2): phase 1 and 2 on the whole batch,
    the first and last heads against the oracle run on those heads."""
    w = W.BASE
    x, xc, *_ = inputs(w)
    kw, dfin = dp.osdn_write_keys(xc["k"], xc["beta"])
    o, hf = dp.forward_write_keys(xc["q"], xc["k"], kw, xc["v"], xc["beta"], None, None, out_dtype=torch.float32)
    # (AUTO: the tensor-core chunk path with the fast workspace)
    for b, hh in ((0, 0), (w.B - 1, w.H - 1)):
        sl = lambda t: t[b:b + 1, :, hh:hh + 1]
        rk, rd = OS.dscan(sl(x["k"]), sl(x["beta"]))
        check_scan(sl(kw), dfin[b:b + 1, hh:hh + 1], rk, rd)
        ro, rh = oracle.forward(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["beta"]), None, None, kw=rk)
        assert_parity(sl(o), ro, "bf16", f"head ({b},{hh}) o")
        assert_parity(hf[b:b + 1, hh:hh + 1], rh, "bf16", f"head ({b},{hh}) h_final")


def chunk_ws(dp, w, mode):
    """Workspace selecting a split mode of the chunk path: "coop" (the fast
    size) or "split" (the records only: prep kernel + state-pass kernel)."""
    B, T, H, nh, D = w.B, w.T, w.H, w.nh, w.Dk
    lo = dp.workspace_size(B, T, H, D, D, nh)
    if mode == "coop":
        n = dp.workspace_size(B, T, H, D, D, nh, fast=True)
    else:
        ct = min(16, 32 // nh)
        n = lo + ((B * H * (-(-T // ct)) * 18688 + 255) // 256) * 256
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


CHUNK_CASES = [("base", W.BASE.scaled(B=2, H=2, T=150), 0.003), ("gated-h0", W.GATED.scaled(B=1, H=3, T=90), 0.2),
               ("neardup-nh3", W.NEARDUP.scaled(B=1, H=2, T=77), 0.5)]


@pytest.mark.parametrize("mode", ["coop", "split"])
@pytest.mark.parametrize("name,w,eta", CHUNK_CASES, ids=[c[0] for c in CHUNK_CASES])
def test_chunk_path_write_keys(dp, name, w, eta, mode):
    """The tensor-core path with write keys (asymmetric Gram K K~^T, readout
    Q K~^T, state update along K~) against the oracle on the same write keys."""
    x, xc, *_ = inputs(w)
    kw, _ = dp.osdn_write_keys(xc["k"], xc["beta"], eta=eta)
    ws = chunk_ws(dp, w, mode)
    o, hf = dp.forward_write_keys(xc["q"], xc["k"], kw, xc["v"], xc["beta"], xc["g"], xc["h0"], impl="chunk_tc",
                                  workspace=ws, out_dtype=torch.float32)
    dp.check_status(ws)
    ro, rh = oracle.forward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], kw=kw.cpu())
    assert_parity(o, ro, "bf16", f"{name} {mode} o")
    assert_parity(hf, rh, "bf16", f"{name} {mode} h_final")


@pytest.mark.parametrize("mode", ["coop", "split"])
def test_chunk_write_keys_equal_keys_is_plain_chunk_forward(dp, mode):
    """kw = k: the write-key chunk path computes what the plain chunk path
    computes (the plain path's prep solves the UT transform with another
    summation order, so the two agree up to rounding: each meets the bf16
    rule against the oracle, and against each other)."""
    w = W.GATED.scaled(B=2, H=2, T=100, nh=2)
    x, xc, *_ = inputs(w)
    ws = chunk_ws(dp, w, mode)
    o1, h1 = dp.forward_write_keys(xc["q"], xc["k"], xc["k"], xc["v"], xc["beta"], xc["g"], xc["h0"],
                                   impl="chunk_tc", workspace=ws, out_dtype=torch.float32)
    ws2 = chunk_ws(dp, w, mode)
    o2, h2 = dp.forward(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], xc["h0"], impl="chunk_tc", workspace=ws2,
                        out_dtype=torch.float32)
    ro, rh = oracle.forward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"])
    for o, h in ((o1, h1), (o2, h2)):
        assert_parity(o, ro, "bf16", f"{mode} o")
        assert_parity(h, rh, "bf16", f"{mode} h_final")
    assert_parity(o1, o2.cpu().double().numpy(), "bf16", "write-key path vs plain path")


def test_write_keys_fall_back_to_recurrent_without_records(dp):
    """With the minimum workspace the write keys run on the recurrent kernel;
    CHUNK_TC is then refused."""
    w = W.BASE.scaled(B=1, H=2, T=40)
    x, xc, *_ = inputs(w)
    kw, _ = dp.osdn_write_keys(xc["k"], xc["beta"], eta=0.1)
    lo = torch.zeros(dp.workspace_size(1, 40, 2, 128, 128, 2), dtype=torch.uint8, device="cuda")
    o, _ = dp.forward_write_keys(xc["q"], xc["k"], kw, xc["v"], xc["beta"], workspace=lo, out_dtype=torch.float32)
    o2, _ = dp.forward_write_keys(xc["q"], xc["k"], kw, xc["v"], xc["beta"], impl="recurrent",
                                  out_dtype=torch.float32)
    assert torch.equal(o, o2)
    with pytest.raises(dp.DPError):
        dp.forward_write_keys(xc["q"], xc["k"], kw, xc["v"], xc["beta"], impl="chunk_tc", workspace=lo)
