"""dp_forward_noalloc: the forward entry point for callers that cannot allocate
device memory (their HBM belongs to a framework allocator or a fixed budget),
which keeps its scratch in a fixed array inside libdp.so. Called through the C
ABI and checked against dp_forward on the same inputs, on two calls in a row
(the second call reuses the scratch the first one left behind), and on tiny
shapes of different sizes, one after another, that keep their per-chunk
records and flags inside the array. This file is collected last on purpose."""
import ctypes

import pytest
import torch

import oracle
from deltaproduct_householder_product_gb300 import workloads as W
from tests.parity import assert_parity, err_stats

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 * 1024   # the array's size, as dp.h states it


@pytest.fixture(scope="module")
def lib():
    from deltaproduct_householder_product_gb300 import build
    build.build()
    from deltaproduct_householder_product_gb300 import _lib
    assert torch.cuda.is_available()
    return _lib


def call_noalloc(lib, w, x, o, hf):
    dims = lib.make_dims(w.B, w.T, w.H, w.Dk, w.Dv, w.nh, torch.bfloat16, "auto", torch.float32)
    return lib.lib().dp_forward_noalloc(ctypes.byref(dims), lib._ptr(x["q"]), lib._ptr(x["k"]),
                                        lib._ptr(x["v"]), lib._ptr(x["beta"]), lib._ptr(x["g"]),
                                        lib._ptr(x["h0"]), lib._ptr(o), lib._ptr(hf), lib._stream(None))


@pytest.mark.parametrize("base", [W.GATED, W.NEARDUP], ids=lambda w: w.name)
def test_noalloc_matches_forward_on_two_calls(lib, base):
    import deltaproduct_householder_product_gb300 as dp
    w = base.scaled(B=2, H=4, T=300)
    x = {k: (None if v is None else v.cuda()) for k, v in W.make_inputs(w).items()}
    o_ref, h_ref = dp.forward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                              out_dtype=torch.float32)
    for call in range(2):
        o = torch.full_like(o_ref, float("nan"))
        hf = torch.full_like(h_ref, float("nan"))
        rc = call_noalloc(lib, w, x, o, hf)
        assert rc == 0, f"call {call}: status {rc}"
        torch.cuda.synchronize()
        so, sh = err_stats(o, o_ref), err_stats(hf, h_ref)
        assert so["rel_max"] <= 2e-2 and sh["rel_max"] <= 2e-2, (call, so, sh)


# Problems of one to three chunks: their records and flags fit in the array,
# so they take the cooperative (or split) mode inside it. Alternating them
# puts each shape's flags on bytes another shape wrote.
TINY_SHAPES = [W.BASE.scaled(B=1, H=1, T=16, seed=31), W.GATED.scaled(B=1, H=3, T=8, nh=3, seed=32),
               W.NEARDUP.scaled(B=1, H=2, T=11, nh=2, seed=33)]


def test_noalloc_alternating_tiny_shapes(lib):
    """Each call of a sequence of tiny shapes (A, B, C, A, C, B, A) meets the
    bf16 rule against the oracle and equals dp_forward on a fresh workspace
    bit for bit (DeltaProduct paper, Sec.4: the result depends on the inputs
    only, not on what an earlier call left in the shared array)."""
    import deltaproduct_householder_product_gb300 as dp
    for w in TINY_SHAPES:
        assert dp.forward_path(w.B, w.T, w.H, w.Dk, w.Dv, w.nh, SCRATCH_BYTES,
                               out_dtype=torch.float32) in ("chunk_coop", "chunk_split"), w
    for i in (0, 1, 2, 0, 2, 1, 0):
        w = TINY_SHAPES[i]
        xh = W.make_inputs(w)
        x = {k: (None if v is None else v.cuda()) for k, v in xh.items()}
        o = torch.full((w.B, w.T, w.H, w.Dv), float("nan"), dtype=torch.float32, device="cuda")
        hf = torch.full((w.B, w.H, w.Dk, w.Dv), float("nan"), dtype=torch.float32, device="cuda")
        assert call_noalloc(lib, w, x, o, hf) == 0
        torch.cuda.synchronize()
        ro, rh = oracle.forward(xh["q"], xh["k"], xh["v"], xh["beta"], xh["g"], xh["h0"])
        assert_parity(o, ro, "bf16", f"o, shape {i}")
        assert_parity(hf, rh, "bf16", f"h_final, shape {i}")
        o_ref, h_ref = dp.forward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"],
                                  out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(hf, h_ref), i


def test_noalloc_rejects_bad_arguments(lib):
    L = lib.lib()
    bad = lib.make_dims(1, 64, 2, 100, 128, 2, torch.bfloat16)
    assert L.dp_forward_noalloc(ctypes.byref(bad), *([None] * 8), None) == 2
    assert L.dp_forward_noalloc(None, *([None] * 8), None) == 1
