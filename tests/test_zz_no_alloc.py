"""dp_forward_noalloc: the forward entry point for callers that cannot allocate
device memory (their HBM belongs to a framework allocator or a fixed budget),
which keeps its scratch in a fixed array inside libdp.so. Called through the C
ABI and checked against dp_forward on the same inputs, on two calls in a row
(the second call reuses the scratch the first one left behind). This file is
collected last on purpose."""
import ctypes

import pytest
import torch

from deltaproduct_householder_product_gb300 import workloads as W
from tests.parity import err_stats

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from deltaproduct_householder_product_gb300 import build
    build.build()
    from deltaproduct_householder_product_gb300 import _lib
    assert torch.cuda.is_available()
    return _lib


@pytest.mark.parametrize("base", [W.GATED, W.NEARDUP], ids=lambda w: w.name)
def test_noalloc_matches_forward_on_two_calls(lib, base):
    import deltaproduct_householder_product_gb300 as dp
    w = base.scaled(B=2, H=4, T=300)
    x = {k: (None if v is None else v.cuda()) for k, v in W.make_inputs(w).items()}
    o_ref, h_ref = dp.forward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                              out_dtype=torch.float32)
    L = lib.lib()
    dims = lib.make_dims(w.B, w.T, w.H, w.Dk, w.Dv, w.nh, torch.bfloat16, "auto", torch.float32)
    for call in range(2):
        o = torch.full_like(o_ref, float("nan"))
        hf = torch.full_like(h_ref, float("nan"))
        rc = L.dp_forward_noalloc(ctypes.byref(dims), lib._ptr(x["q"]), lib._ptr(x["k"]),
                                  lib._ptr(x["v"]), lib._ptr(x["beta"]), lib._ptr(x["g"]),
                                  lib._ptr(x["h0"]), lib._ptr(o), lib._ptr(hf), lib._stream(None))
        assert rc == 0, f"call {call}: status {rc}"
        torch.cuda.synchronize()
        so, sh = err_stats(o, o_ref), err_stats(hf, h_ref)
        assert so["rel_max"] <= 2e-2 and sh["rel_max"] <= 2e-2, (call, so, sh)


def test_noalloc_rejects_bad_arguments(lib):
    L = lib.lib()
    bad = lib.make_dims(1, 64, 2, 100, 128, 2, torch.bfloat16)
    assert L.dp_forward_noalloc(ctypes.byref(bad), *([None] * 8), None) == 2
    assert L.dp_forward_noalloc(None, *([None] * 8), None) == 1
