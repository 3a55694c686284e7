"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the device. CPU only:
none of these calls reaches a kernel."""
import ctypes
import os
import re

import pytest

from deltaproduct_householder_product_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dp.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dp_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    from deltaproduct_householder_product_gb300 import build
    build.build()
    return _lib.lib()


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert "dp_forward" in names and "dp_decode_step" in names and "dp_state_io" in names
    for n in names:
        assert hasattr(L, n), f"libdp.so does not export {n}"


def test_abi_version_matches_header(L):
    m = re.search(r"#define DP_ABI_VERSION (\d+)", open(HEADER).read())
    assert L.dp_abi_version() == int(m.group(1))


def test_status_strings(L):
    for code in range(8):
        assert L.dp_status_string(code)
    assert L.dp_status_string(99) == b"unknown status"


def ws(L, **kw):
    d = dict(B=1, T=64, H=2, Dk=128, Dv=128, nh=2, dtype=_lib.DP_BF16, impl=0)
    d.update(kw)
    dims = _lib.Dims(**d)
    n = ctypes.c_size_t(0)
    rc = L.dp_forward_workspace_size(ctypes.byref(dims), ctypes.byref(n))
    return rc, n.value


def test_workspace_size_and_validation(L):
    rc, n = ws(L)
    assert rc == 0 and n >= 256 and n % 256 == 0
    assert ws(L, Dk=96)[0] == 2            # DP_ERR_UNSUPPORTED
    assert ws(L, Dv=256)[0] == 2
    assert ws(L, nh=0)[0] == 2
    assert ws(L, nh=5)[0] == 2
    assert ws(L, B=-1)[0] == 1             # DP_ERR_INVALID_ARG
    assert ws(L, dtype=7)[0] == 1
    assert ws(L, impl=9)[0] == 1
    assert ws(L, T=0)[0] == 0
    assert ws(L, Dk=32, Dv=32, dtype=_lib.DP_F32, impl=1)[0] == 0
    n_null = L.dp_forward_workspace_size(None, ctypes.byref(ctypes.c_size_t()))
    assert n_null == 1


def test_forward_rejects_before_launch(L):
    dims = _lib.Dims(1, 64, 2, 128, 128, 2, _lib.DP_BF16, 0)
    null = [None] * 9
    # NULL inputs -> invalid argument, nothing enqueued
    assert L.dp_forward(ctypes.byref(dims), *null, 0, None) == 1
    bad = _lib.Dims(1, 64, 2, 100, 128, 2, _lib.DP_BF16, 0)
    assert L.dp_forward(ctypes.byref(bad), *null, 0, None) == 2
    assert L.dp_forward(None, *null, 0, None) == 1
    # misaligned q pointer is reported as an alignment error before any CUDA call
    args = [ctypes.c_void_p(0x1001)] + [ctypes.c_void_p(0x1000)] * 8
    assert L.dp_forward(ctypes.byref(dims), *args, 1 << 20, None) == 3


def test_decode_and_state_io_reject(L):
    dims = _lib.Dims(1, 1, 2, 128, 128, 2, _lib.DP_BF16, 0)
    assert L.dp_decode_step(ctypes.byref(dims), *([None] * 7), None) == 1
    assert L.dp_state_io(5, 1, 1, 128, 128, None, None, 0, 0, None) == 1
    assert L.dp_state_io(0, 1, 1, 100, 128, None, None, 0, 0, None) == 2
    assert L.dp_state_io(0, 1, 1, 128, 128, None, None, 0, 0, None) == 1
    assert L.dp_state_io(0, 0, 1, 128, 128, None, None, 0, 0, None) == 0   # empty: no-op
    assert L.dp_check_status(None, None) == 1


def test_forward_path_validation(L):
    """dp_forward_path validates like dp_forward: NULL output, bad dims and a
    workspace below the minimum are rejected; a valid query names a path."""
    dims = _lib.make_dims(1, 16, 2, 64, 64, 2, _lib.DP_BF16, "recurrent")
    code = ctypes.c_int(-1)
    assert L.dp_forward_path(ctypes.byref(dims), 256, None) == 1
    assert L.dp_forward_path(ctypes.byref(dims), 255, ctypes.byref(code)) == 4
    bad = _lib.make_dims(1, 16, 2, 48, 64, 2, _lib.DP_BF16, "recurrent")
    assert L.dp_forward_path(ctypes.byref(bad), 256, ctypes.byref(code)) == 2
    assert L.dp_forward_path(ctypes.byref(dims), 256, ctypes.byref(code)) == 0
    assert _lib.PATHS[code.value] == "recurrent"


def test_varlen_validation(L):
    """dp_forward rejects a nonzero max_seqlen; dp_forward_varlen rejects a
    missing or host cu_seqlens and a max_seqlen beyond T, before any launch."""
    import ctypes as C
    dims = _lib.make_dims(2, 16, 2, 64, 64, 2, _lib.DP_BF16, "recurrent", max_seqlen=8)
    null = None
    args = [null] * 9 + [C.c_size_t(0), null]
    assert L.dp_forward(C.byref(dims), *args) == 1
    host_cu = (C.c_int * 3)(0, 8, 16)
    vargs = [C.cast(host_cu, C.c_void_p)] + [null] * 9 + [C.c_size_t(0), null]
    assert L.dp_forward_varlen(C.byref(dims), *vargs) == 1
    bad = _lib.make_dims(2, 16, 2, 64, 64, 2, _lib.DP_BF16, "recurrent", max_seqlen=17)
    assert L.dp_forward_varlen(C.byref(bad), *vargs) == 1


def test_backward_workspace_and_validation(L):
    """dp_backward_workspace_size: status block, one fp32 D_k x D_v
    checkpoint per (b,h) every segment of tokens and every sub-step's error;
    dp_backward rejects NULL inputs, an unknown impl and a short workspace
    before any launch."""
    import ctypes as C
    n = C.c_size_t(0)
    dims = _lib.make_dims(2, 100, 3, 128, 64, 2, _lib.DP_BF16, "auto", _lib.DP_F32)
    assert L.dp_backward_workspace_size(C.byref(dims), C.byref(n)) == 0
    r256 = lambda x: (x + 255) // 256 * 256
    seg = 12                                   # tokens per checkpoint at D_k = 128
    ck = 2 * 3 * ((100 + seg - 1) // seg) * 128 * 64 * 4
    errs = 2 * 100 * 3 * 2 * 64 * 4            # every sub-step's error, fp32
    assert n.value == 256 + r256(r256(ck) + errs)
    d32 = _lib.make_dims(1, 100, 1, 32, 32, 1, _lib.DP_F32)
    assert L.dp_backward_workspace_size(C.byref(d32), C.byref(n)) == 0
    assert n.value == 256 + r256(r256(((100 + 47) // 48) * 32 * 32 * 4) + 100 * 32 * 4)
    explicit = _lib.make_dims(2, 100, 3, 128, 64, 2, _lib.DP_BF16, "recurrent")
    m = C.c_size_t(0)
    assert L.dp_backward_workspace_size(C.byref(explicit), C.byref(m)) == 0
    assert m.value == 256 + r256(r256(ck) + errs)
    assert L.dp_backward_workspace_size(C.byref(_lib.make_dims(2, 100, 3, 128, 64, 2, _lib.DP_BF16, 7)),
                                        C.byref(m)) == 1
    # D_k = D_v = 128: the chunked form's records (ct = 16 tokens per chunk at
    # n_h = 2; per chunk W, U [32,128], T [32,32], P [16,32], K K^T [32,32],
    # K [32,128], Q [16,128], for gated problems the decayed keys [32,128],
    # the undecayed scores [16,32], the decays [32,32], three [32] vectors
    # (Gamma, Gamma_C / Gamma, log gates) and <dS1, S0> in 4 floats, the state
    # at its start and the gradient at its end [128,128], U' and dU'
    # [32,128], fp32)
    rec = lambda impl: _lib.make_dims(2, 100, 3, 128, 128, 2, _lib.DP_BF16, impl, _lib.DP_F32)
    ck128 = 2 * 3 * ((100 + seg - 1) // seg) * 128 * 128 * 4
    need_rec = 256 + r256(r256(ck128) + 2 * 100 * 3 * 2 * 128 * 4)
    chunks = 2 * 3 * ((100 + 15) // 16)
    per_chunk = (2 * 32 * 128 + 32 * 32 + 16 * 32 + 32 * 32 + 32 * 128 + 16 * 128 + 32 * 128 + 16 * 32 + 32 * 32
                 + 3 * 32 + 4 + 2 * 128 * 128 + 2 * 32 * 128) * 4
    need_chunk = 256 + r256(chunks * per_chunk)
    for impl, want in (("recurrent", need_rec), ("chunk_tc", need_chunk), ("auto", max(need_rec, need_chunk))):
        assert L.dp_backward_workspace_size(C.byref(rec(impl)), C.byref(m)) == 0 and m.value == want, impl
    # packed sequences: both forms, sized for max_seqlen per (sequence, head)
    vl = lambda impl: _lib.make_dims(2, 100, 3, 128, 128, 2, _lib.DP_BF16, impl, _lib.DP_F32, max_seqlen=60)
    rec_vl = 256 + r256(r256(2 * 3 * 5 * 128 * 128 * 4) + 2 * 60 * 3 * 2 * 128 * 4)
    chunk_vl = 256 + r256(2 * 3 * ((60 + 15) // 16) * per_chunk)
    for impl, want in (("recurrent", rec_vl), ("chunk_tc", chunk_vl), ("auto", max(rec_vl, chunk_vl))):
        assert L.dp_backward_workspace_size(C.byref(vl(impl)), C.byref(m)) == 0 and m.value == want, impl
    assert L.dp_backward_workspace_size(C.byref(dims), None) == 1
    null = [None] * 15
    assert L.dp_backward(C.byref(dims), *null, C.c_size_t(0), None) == 1
    bad = _lib.make_dims(2, 100, 3, 96, 64, 2, _lib.DP_BF16)
    assert L.dp_backward(C.byref(bad), *null, C.c_size_t(0), None) == 2
    empty = _lib.make_dims(0, 100, 3, 128, 64, 2, _lib.DP_BF16)
    assert L.dp_backward_workspace_size(C.byref(empty), C.byref(n)) == 0 and n.value == 256


def test_wait_fault_hook_validation(L):
    """dp_test_set_wait_fault takes 0 or 1 for its withhold switch (anything
    else is rejected without changing the setting) and (0, 0) restores
    normal operation. Host-only: no kernel runs."""
    assert L.dp_test_set_wait_fault(2, 0) == 1
    assert L.dp_test_set_wait_fault(-1, 5) == 1
    assert L.dp_test_set_wait_fault(0, 1000) == 0
    assert L.dp_test_set_wait_fault(0, 0) == 0
