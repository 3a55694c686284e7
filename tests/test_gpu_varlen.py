"""GPU parity of packed variable-length sequences (dp_forward_varlen) against
the fp64 oracle run on each sequence, through the C ABI: every chunk-path
mode and the recurrent kernel, lengths that are empty, single tokens, chunk
multiples and ragged; bit-exact agreement with the dense call when every
sequence has the same length; offsets that break the contract are reported
by the device without any access outside the sequences."""
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


def packed_inputs(base, lengths, nh, seed):
    """Seeded dense inputs for one long sequence per head, cut into the
    packed layout: tokens of all sequences back to back (B axis dropped)."""
    T = int(sum(lengths))
    w = base.scaled(B=1, H=3, T=max(T, 1), nh=nh, seed=seed)
    x = W.make_inputs(w)
    out = {k: (None if x[k] is None else x[k][0, :T].contiguous()) for k in ("q", "k", "v", "beta", "g")}
    gen = torch.Generator().manual_seed(seed + 100)
    N = len(lengths)
    out["h0"] = (0.02 * torch.randn(N, w.H, w.Dk, w.Dv, generator=gen)) if base.h0_std > 0 else None
    out["cu"] = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    return w, out


def oracle_varlen(x, lengths):
    cu = x["cu"].tolist()
    os_, hs = [], []
    for s in range(len(lengths)):
        a, e = cu[s], cu[s + 1]
        sl = lambda t: None if t is None else t[a:e].unsqueeze(0)
        h0 = None if x["h0"] is None else x["h0"][s:s + 1]
        o, h = oracle.forward(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["beta"]), sl(x["g"]), h0)
        os_.append(np.asarray(o)[0])
        hs.append(np.asarray(h)[0])
    return np.concatenate(os_, 0), np.stack(hs, 0)


def run_varlen(dp, x, impl="auto", path="split", max_seqlen=None):
    xc = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    T, H, nh, Dk = xc["k"].shape
    N = xc["cu"].numel() - 1
    if max_seqlen is None:
        max_seqlen = int((x["cu"][1:] - x["cu"][:-1]).max().item())
    lo = dp.workspace_size(N, T, H, Dk, Dk, nh, impl=impl)
    hi = dp.workspace_size(N, T, H, Dk, Dk, nh, impl=impl, fast=True)
    dims_size = {"split": hi, "fused": lo}[path]
    ws = torch.zeros(dims_size, dtype=torch.uint8, device="cuda")
    o, hf = dp.forward_varlen(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], xc["h0"], cu_seqlens=xc["cu"],
                              max_seqlen=max_seqlen, impl=impl, workspace=ws, out_dtype=torch.float32)
    dp.check_status(ws)
    return o, hf


LENGTHS = [[0, 1, 15, 16, 17, 100, 33], [200, 3, 64, 0, 47], [1], [31, 32, 5]]


@pytest.mark.parametrize("impl,path", [("chunk_tc", "split"), ("chunk_tc", "fused"), ("recurrent", "fused")])
@pytest.mark.parametrize("base,nh,lengths", [(W.BASE, 2, LENGTHS[0]), (W.GATED, 4, LENGTHS[1]),
                                             (W.NEARDUP, 3, LENGTHS[3]), (W.LONG, 1, LENGTHS[1]),
                                             (W.GATED, 2, LENGTHS[2])],
                         ids=lambda v: getattr(v, "name", str(v)))
def test_varlen_parity(dp, base, nh, lengths, impl, path):
    w, x = packed_inputs(base, lengths, nh, seed=21)
    o, hf = run_varlen(dp, x, impl=impl, path=path)
    ro, rh = oracle_varlen(x, lengths)
    assert_parity(o, ro, "bf16", "o")
    assert_parity(hf, rh, "bf16", "h_final")


@pytest.mark.parametrize("path", ["split", "fused"])
def test_equal_lengths_match_dense_bitwise(dp, path):
    """Packing B sequences of one length T runs the same chunk grid on the
    same values as the dense [B, T] call."""
    B, T, nh = 3, 70, 2
    w = W.GATED.scaled(B=B, H=3, T=T, nh=nh)
    x = W.make_inputs(w)
    xc = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    lo = dp.workspace_size(B, T, 3, 128, 128, nh)
    size = dp.workspace_size(B, T, 3, 128, 128, nh, fast=True) if path == "split" else lo
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    o_d, h_d = dp.forward(xc["q"], xc["k"], xc["v"], xc["beta"], xc["g"], xc["h0"], workspace=ws,
                          out_dtype=torch.float32)
    pk = lambda t: None if t is None else t.reshape(B * T, *t.shape[2:]).contiguous()
    cu = torch.arange(0, B * T + 1, T, dtype=torch.int32, device="cuda")
    ws2 = torch.zeros(size, dtype=torch.uint8, device="cuda")
    o_v, h_v = dp.forward_varlen(pk(xc["q"]), pk(xc["k"]), pk(xc["v"]), pk(xc["beta"]), pk(xc["g"]), xc["h0"],
                                 cu_seqlens=cu, max_seqlen=T, workspace=ws2, out_dtype=torch.float32)
    dp.check_status(ws2)
    assert torch.equal(o_v.reshape(B, T, *o_v.shape[1:]), o_d)
    assert torch.equal(h_v, h_d)


@pytest.mark.parametrize("impl", ["chunk_tc", "recurrent"])
def test_bad_offsets_are_reported(dp, impl):
    """Offsets out of order, or a sequence longer than max_seqlen: the device
    skips those sequences and reports DP_ERR_DEVICE; the valid ones still run."""
    w, x = packed_inputs(W.BASE, [40, 40, 40], 2, seed=5)
    xc = {k: (None if v is None else v.cuda()) for k, v in x.items()}
    T = 120
    for cu_list, max_len in (([0, 50, 30, 120], 90), ([0, 40, 80, 120], 20)):
        cu = torch.tensor(cu_list, dtype=torch.int32, device="cuda")
        ws = torch.zeros(dp.workspace_size(3, T, 3, 128, 128, 2, impl=impl, fast=True), dtype=torch.uint8,
                         device="cuda")
        dp.forward_varlen(xc["q"], xc["k"], xc["v"], xc["beta"], None, None, cu_seqlens=cu, max_seqlen=max_len,
                          impl=impl, workspace=ws, out_dtype=torch.float32)
        with pytest.raises(dp.DPError) as e:
            dp.check_status(ws)
        assert e.value.code == 7
