"""GB300 DeltaProduct forward recurrence: Python face of libdp.so.

The recurrence (DeltaProduct paper, Sec.4 Eq.(2)-(3), gated variant): per
(batch, head) and token t, H <- g_t H, then n_h ordered steps
H <- H + beta k (v - H^T k)^T, then o_t = H^T q_t. All arithmetic runs in the
library's CUDA kernels; these functions only marshal arguments (see
``_lib.py``) and raise on any non-zero status.
"""
import torch

from . import _lib
from ._lib import DPError, STATE_EXPORT, STATE_IMPORT, STATE_ZERO  # noqa: F401

__all__ = ["forward", "forward_varlen", "forward_noalloc", "forward_path", "supports", "decode_step", "state_io", "check_status",
           "backward", "backward_varlen", "prologue", "prologue_flags", "osdn_write_keys", "forward_write_keys",
           "workspace_size", "set_wait_fault",
           "DPError", "abi_version"]


PROLOGUE = {"key_silu_l2": 1, "query_l2": 2, "beta_sigmoid": 4, "beta_2sigmoid": 8, "gate_sigmoid": 16}


def prologue_flags(prologue):
    """dp_prologue_flags from an int, or from names (iterable or '+'-joined
    string) among PROLOGUE's keys."""
    if prologue is None:
        return 0
    if isinstance(prologue, int):
        return prologue
    names = prologue.split("+") if isinstance(prologue, str) else list(prologue)
    return sum(PROLOGUE[n] for n in names if n)


def abi_version():
    return _lib.lib().dp_abi_version()


def workspace_size(B, T, H, Dk, Dv, nh, dtype=torch.bfloat16, impl="auto", out_dtype=None,
                   fast=False, prologue=0):
    """Device workspace bytes dp_forward needs for this problem; with ``fast``,
    the size with which it takes its fastest path (the chunk path's parallel
    prep kernel and per-chunk records). ``prologue`` as for ``forward``."""
    return _lib.workspace_size(_lib.make_dims(B, T, H, Dk, Dv, nh, dtype, impl, out_dtype,
                                              prologue=prologue_flags(prologue)), fast)


def forward_path(B, T, H, Dk, Dv, nh, workspace_bytes, dtype=torch.bfloat16, impl="auto", out_dtype=None,
                 prologue=0):
    """How ``forward`` runs this problem with a workspace of ``workspace_bytes``:
    "recurrent", "chunk_fused", "chunk_split" (two kernels) or "chunk_coop"
    (one cooperative launch)."""
    return _lib.forward_path(_lib.make_dims(B, T, H, Dk, Dv, nh, dtype, impl, out_dtype,
                                            prologue=prologue_flags(prologue)), workspace_bytes)


def supports(impl, B, T, H, Dk, Dv, nh, dtype=torch.bfloat16):
    """True when kernel family ``impl`` handles this problem."""
    try:
        _lib.workspace_size(_lib.make_dims(B, T, H, Dk, Dv, nh, dtype, impl))
        return True
    except DPError as e:
        if e.code == 2:
            return False
        raise


def forward(q, k, v, beta, g=None, h0=None, *, impl="auto", out=None, h_final=True,
            workspace=None, stream=None, out_dtype=None, prologue=0):
    """Run the recurrence over whole sequences.

    q [B,T,H,Dk], k [B,T,H,nh,Dk], v [B,T,H,nh,Dv], beta [B,T,H,nh], g [B,T,H]
    or None (ungated), all CUDA tensors of one dtype (float32 or bfloat16);
    h0 [B,H,Dk,Dv] float32 or None (zeros). ``out_dtype`` is the dtype of o
    (default: the input dtype; float32 is allowed with bfloat16 inputs, or
    taken from ``out``). ``h_final`` may be True (allocate),
    False/None (do not write) or a float32 [B,H,Dk,Dv] tensor (may be h0).
    ``prologue``: dp_prologue_flags (int or names, see ``prologue_flags``):
    the named inputs hold raw projections and the kernels map them on load.
    Returns (o, h_final_or_None).
    """
    B, T, H, nh, Dk = k.shape
    Dv = v.shape[-1]
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g)):
        _lib._need_cuda(name, t, dt)
    _lib._need_cuda("h0", h0, torch.float32)
    if q.shape != (B, T, H, Dk) or v.shape != (B, T, H, nh, Dv) or beta.shape != (B, T, H, nh):
        raise ValueError("inconsistent shapes for q, k, v, beta")
    if g is not None and g.shape != (B, T, H):
        raise ValueError("g must be [B,T,H]")
    if h0 is not None and h0.shape != (B, H, Dk, Dv):
        raise ValueError("h0 must be [B,H,Dk,Dv]")
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else dt
    dims = _lib.make_dims(B, T, H, Dk, Dv, nh, dt, impl, out_dtype, prologue=prologue_flags(prologue))
    if out is None:
        out = torch.empty((B, T, H, Dv), dtype=out_dtype, device=q.device)
    _lib._need_cuda("out", out, out_dtype)
    if h_final is True:
        h_final = torch.empty((B, H, Dk, Dv), dtype=torch.float32, device=q.device)
    elif h_final is False:
        h_final = None
    _lib._need_cuda("h_final", h_final, torch.float32)
    need = _lib.workspace_size(dims, fast=True)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    _lib._need_cuda("workspace", workspace)
    rc = _lib.lib().dp_forward(
        dims, _lib._ptr(q), _lib._ptr(k), _lib._ptr(v), _lib._ptr(beta), _lib._ptr(g),
        _lib._ptr(h0), _lib._ptr(out), _lib._ptr(h_final), _lib._ptr(workspace),
        workspace.numel() * workspace.element_size(), _lib._stream(stream))
    _lib._check(rc, "dp_forward")
    return out, h_final


def backward(q, k, v, beta, g=None, h0=None, *, d_o, dh_final=None, want_dh0=True, workspace=None,
             stream=None, impl="auto"):
    """Gradients of <d_o, o> + <dh_final, h_final> through ``forward``.

    Inputs as for ``forward``; d_o [B,T,H,Dv] (float32, or the input dtype);
    dh_final float32 [B,H,Dk,Dv] or None (zeros). Returns a dict of float32
    tensors dq, dk, dv, dbeta, dg (None when ungated) and dh0 (None unless
    ``want_dh0``), in the layouts of the corresponding inputs. ``impl``:
    "auto" (the chunked form for ungated problems with Dk = Dv = 128, else
    the recurrent form), "recurrent", or "chunk_tc" (the chunked form;
    unsupported where it does not apply).
    """
    B, T, H, nh, Dk = k.shape
    Dv = v.shape[-1]
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g)):
        _lib._need_cuda(name, t, dt)
    _lib._need_cuda("h0", h0, torch.float32)
    _lib._need_cuda("d_o", d_o)
    _lib._need_cuda("dh_final", dh_final, torch.float32)
    if q.shape != (B, T, H, Dk) or v.shape != (B, T, H, nh, Dv) or beta.shape != (B, T, H, nh):
        raise ValueError("inconsistent shapes for q, k, v, beta")
    if d_o.shape != (B, T, H, Dv):
        raise ValueError("d_o must be [B,T,H,Dv]")
    dims = _lib.make_dims(B, T, H, Dk, Dv, nh, dt, impl, d_o.dtype)
    f32 = dict(dtype=torch.float32, device=q.device)
    out = {"dq": torch.empty((B, T, H, Dk), **f32), "dk": torch.empty((B, T, H, nh, Dk), **f32),
           "dv": torch.empty((B, T, H, nh, Dv), **f32), "dbeta": torch.empty((B, T, H, nh), **f32),
           "dg": None if g is None else torch.empty((B, T, H), **f32),
           "dh0": torch.empty((B, H, Dk, Dv), **f32) if want_dh0 else None}
    need = _lib.backward_workspace_size(dims)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    _lib._need_cuda("workspace", workspace)
    rc = _lib.lib().dp_backward(
        dims, _lib._ptr(q), _lib._ptr(k), _lib._ptr(v), _lib._ptr(beta), _lib._ptr(g), _lib._ptr(h0),
        _lib._ptr(d_o), _lib._ptr(dh_final), _lib._ptr(out["dq"]), _lib._ptr(out["dk"]), _lib._ptr(out["dv"]),
        _lib._ptr(out["dbeta"]), _lib._ptr(out["dg"]), _lib._ptr(out["dh0"]), _lib._ptr(workspace),
        workspace.numel() * workspace.element_size(), _lib._stream(stream))
    _lib._check(rc, "dp_backward")
    return out


def backward_varlen(q, k, v, beta, g=None, h0=None, *, cu_seqlens, max_seqlen=None, d_o, dh_final=None,
                    want_dh0=True, workspace=None, stream=None, impl="auto"):
    """``backward`` over packed variable-length sequences (the layouts of
    ``forward_varlen``; dh_final and dh0 are [N,H,Dk,Dv]); ``impl`` as for
    ``backward``."""
    T, H, nh, Dk = k.shape
    Dv = v.shape[-1]
    N = cu_seqlens.numel() - 1
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g)):
        _lib._need_cuda(name, t, dt)
    _lib._need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    _lib._need_cuda("h0", h0, torch.float32)
    _lib._need_cuda("d_o", d_o)
    _lib._need_cuda("dh_final", dh_final, torch.float32)
    if max_seqlen is None:
        max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if N > 0 else 0
    dims = _lib.make_dims(N, T, H, Dk, Dv, nh, dt, impl, d_o.dtype, max(int(max_seqlen), 1 if T > 0 else 0))
    f32 = dict(dtype=torch.float32, device=q.device)
    out = {"dq": torch.empty((T, H, Dk), **f32), "dk": torch.empty((T, H, nh, Dk), **f32),
           "dv": torch.empty((T, H, nh, Dv), **f32), "dbeta": torch.empty((T, H, nh), **f32),
           "dg": None if g is None else torch.empty((T, H), **f32),
           "dh0": torch.empty((N, H, Dk, Dv), **f32) if want_dh0 else None}
    if workspace is None:
        workspace = torch.zeros(_lib.backward_workspace_size(dims), dtype=torch.uint8, device=q.device)
    rc = _lib.lib().dp_backward_varlen(
        dims, _lib._ptr(cu_seqlens), _lib._ptr(q), _lib._ptr(k), _lib._ptr(v), _lib._ptr(beta), _lib._ptr(g),
        _lib._ptr(h0), _lib._ptr(d_o), _lib._ptr(dh_final), _lib._ptr(out["dq"]), _lib._ptr(out["dk"]),
        _lib._ptr(out["dv"]), _lib._ptr(out["dbeta"]), _lib._ptr(out["dg"]), _lib._ptr(out["dh0"]),
        _lib._ptr(workspace), workspace.numel() * workspace.element_size(), _lib._stream(stream))
    _lib._check(rc, "dp_backward_varlen")
    return out, workspace


def forward_varlen(q, k, v, beta, g=None, h0=None, *, cu_seqlens, max_seqlen=None, impl="auto", out=None,
                   h_final=True, workspace=None, stream=None, out_dtype=None, prologue=0):
    """Run the recurrence over N variable-length sequences packed along T.

    q [T,H,Dk], k [T,H,nh,Dk], v [T,H,nh,Dv], beta [T,H,nh], g [T,H] or None;
    cu_seqlens int32 CUDA tensor [N+1] of token offsets (0, ..., T); h0
    [N,H,Dk,Dv] float32 or None. ``max_seqlen`` bounds the longest sequence
    (read from cu_seqlens when None, which synchronises). Returns (o [T,H,Dv],
    h_final [N,H,Dk,Dv] or None). Every sequence starts from its own h0.
    """
    T, H, nh, Dk = k.shape
    Dv = v.shape[-1]
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g)):
        _lib._need_cuda(name, t, dt)
    _lib._need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    N = cu_seqlens.numel() - 1
    if N < 0:
        raise ValueError("cu_seqlens needs at least one entry")
    _lib._need_cuda("h0", h0, torch.float32)
    if q.shape != (T, H, Dk) or v.shape != (T, H, nh, Dv) or beta.shape != (T, H, nh):
        raise ValueError("inconsistent shapes for q, k, v, beta")
    if g is not None and g.shape != (T, H):
        raise ValueError("g must be [T,H]")
    if h0 is not None and h0.shape != (N, H, Dk, Dv):
        raise ValueError("h0 must be [N,H,Dk,Dv]")
    if max_seqlen is None:
        max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if N > 0 else 0
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else dt
    dims = _lib.make_dims(N, T, H, Dk, Dv, nh, dt, impl, out_dtype, max_seqlen, prologue_flags(prologue))
    if out is None:
        out = torch.empty((T, H, Dv), dtype=out_dtype, device=q.device)
    _lib._need_cuda("out", out, out_dtype)
    if h_final is True:
        h_final = torch.empty((N, H, Dk, Dv), dtype=torch.float32, device=q.device)
    elif h_final is False:
        h_final = None
    _lib._need_cuda("h_final", h_final, torch.float32)
    if workspace is None:
        workspace = torch.zeros(_lib.workspace_size(dims, fast=True), dtype=torch.uint8, device=q.device)
    _lib._need_cuda("workspace", workspace)
    rc = _lib.lib().dp_forward_varlen(
        dims, _lib._ptr(cu_seqlens), _lib._ptr(q), _lib._ptr(k), _lib._ptr(v), _lib._ptr(beta), _lib._ptr(g),
        _lib._ptr(h0), _lib._ptr(out), _lib._ptr(h_final), _lib._ptr(workspace),
        workspace.numel() * workspace.element_size(), _lib._stream(stream))
    _lib._check(rc, "dp_forward_varlen")
    return out, h_final


def forward_noalloc(q, k, v, beta, g=None, h0=None, *, impl="auto", out, h_final=None,
                    stream=None):
    """dp_forward_noalloc: ``forward`` without a device workspace, for callers
    that cannot allocate device memory; the library's fixed scratch array is
    used instead. ``out`` (and ``h_final`` if wanted) must be given. Calls on
    one device whose kernels overlap on the GPU race on that shared scratch."""
    B, T, H, nh, Dk = k.shape
    Dv = v.shape[-1]
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g)):
        _lib._need_cuda(name, t, dt)
    _lib._need_cuda("h0", h0, torch.float32)
    _lib._need_cuda("out", out)
    _lib._need_cuda("h_final", h_final, torch.float32)
    dims = _lib.make_dims(B, T, H, Dk, Dv, nh, dt, impl, out.dtype)
    rc = _lib.lib().dp_forward_noalloc(
        dims, _lib._ptr(q), _lib._ptr(k), _lib._ptr(v), _lib._ptr(beta), _lib._ptr(g),
        _lib._ptr(h0), _lib._ptr(out), _lib._ptr(h_final), _lib._stream(stream))
    _lib._check(rc, "dp_forward_noalloc")
    return out, h_final


def decode_step(q, k, v, beta, g, state, *, out=None, stream=None, out_dtype=None, prologue=0):
    """One token on a carried fp32 state (updated in place).

    q [B,H,Dk], k [B,H,nh,Dk], v [B,H,nh,Dv], beta [B,H,nh], g [B,H] or None,
    state [B,H,Dk,Dv] float32. Returns o [B,H,Dv].
    """
    B, H, nh, Dk = k.shape
    Dv = v.shape[-1]
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g)):
        _lib._need_cuda(name, t, dt)
    _lib._need_cuda("state", state, torch.float32)
    if state.shape != (B, H, Dk, Dv):
        raise ValueError("state must be [B,H,Dk,Dv]")
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else dt
    if out is None:
        out = torch.empty((B, H, Dv), dtype=out_dtype, device=q.device)
    _lib._need_cuda("out", out, out_dtype)
    dims = _lib.make_dims(B, 1, H, Dk, Dv, nh, dt, "auto", out_dtype, prologue=prologue_flags(prologue))
    rc = _lib.lib().dp_decode_step(dims, _lib._ptr(q), _lib._ptr(k), _lib._ptr(v),
                                   _lib._ptr(beta), _lib._ptr(g), _lib._ptr(state),
                                   _lib._ptr(out), _lib._stream(stream))
    _lib._check(rc, "dp_decode_step")
    return out


def prologue(q, k, beta, g=None, *, flags, stream=None):
    """dp_prologue: the input maps on their own (the unfused form). Inputs as
    for ``forward`` (raw projections); returns (q, k, beta, g) with the
    flagged ones mapped (new tensors in the input dtype) and the others
    passed through."""
    f = prologue_flags(flags)
    B, T, H, nh, Dk = k.shape
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("beta", beta), ("g", g)):
        _lib._need_cuda(name, t, dt)
    dims = _lib.make_dims(B, T, H, Dk, Dk, nh, dt, "auto", dt, prologue=f)
    q_o = torch.empty_like(q) if f & 2 else q
    k_o = torch.empty_like(k) if f & 1 else k
    b_o = torch.empty_like(beta) if f & 12 else beta
    g_o = torch.empty_like(g) if (g is not None and f & 16) else g
    rc = _lib.lib().dp_prologue(dims, _lib._ptr(q), _lib._ptr(k), _lib._ptr(beta), _lib._ptr(g),
                                _lib._ptr(q_o) if f & 2 else None, _lib._ptr(k_o) if f & 1 else None,
                                _lib._ptr(b_o) if f & 12 else None,
                                _lib._ptr(g_o) if (g is not None and f & 16) else None, _lib._stream(stream))
    _lib._check(rc, "dp_prologue")
    return q_o, k_o, b_o, g_o


def osdn_write_keys(k, beta, r=None, d0=None, *, eta=0.003, d_lo=0.5, d_hi=2.0, eps=1e-6, stream=None):
    """dp_osdn_write_keys (OSDN phase 1): returns (kw, d_final) for keys k
    [B,T,H,nh,Dk], betas [B,T,H,nh], APF retention r [B,T,H] or None, and
    the initial preconditioner d0 [B,H,Dk] float32 or None (ones)."""
    B, T, H, nh, Dk = k.shape
    dt = k.dtype
    for name, t in (("k", k), ("beta", beta), ("r", r)):
        _lib._need_cuda(name, t, dt)
    _lib._need_cuda("d0", d0, torch.float32)
    dims = _lib.make_dims(B, T, H, Dk, Dk, nh, dt)
    kw = torch.empty_like(k)
    d_final = torch.empty((B, H, Dk), dtype=torch.float32, device=k.device)
    rc = _lib.lib().dp_osdn_write_keys(dims, _lib._ptr(k), _lib._ptr(beta), _lib._ptr(r), _lib._ptr(d0),
                                       eta, d_lo, d_hi, eps, _lib._ptr(kw), _lib._ptr(d_final),
                                       _lib._stream(stream))
    _lib._check(rc, "dp_osdn_write_keys")
    return kw, d_final


def forward_write_keys(q, k, kw, v, beta, g=None, h0=None, *, impl="auto", out=None, h_final=True,
                       workspace=None, stream=None, out_dtype=None, prologue=0):
    """dp_forward_write_keys (OSDN phase 2): ``forward`` with the state
    written along the write keys kw (layout of k)."""
    B, T, H, nh, Dk = k.shape
    Dv = v.shape[-1]
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("kw", kw), ("v", v), ("beta", beta), ("g", g)):
        _lib._need_cuda(name, t, dt)
    _lib._need_cuda("h0", h0, torch.float32)
    if kw.shape != k.shape:
        raise ValueError("kw must have the shape of k")
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else dt
    dims = _lib.make_dims(B, T, H, Dk, Dv, nh, dt, impl, out_dtype, prologue=prologue_flags(prologue))
    if out is None:
        out = torch.empty((B, T, H, Dv), dtype=out_dtype, device=q.device)
    if h_final is True:
        h_final = torch.empty((B, H, Dk, Dv), dtype=torch.float32, device=q.device)
    elif h_final is False:
        h_final = None
    if workspace is None:
        workspace = torch.zeros(_lib.workspace_size(dims, fast=True), dtype=torch.uint8, device=q.device)
    rc = _lib.lib().dp_forward_write_keys(
        dims, _lib._ptr(q), _lib._ptr(k), _lib._ptr(kw), _lib._ptr(v), _lib._ptr(beta), _lib._ptr(g),
        _lib._ptr(h0), _lib._ptr(out), _lib._ptr(h_final), _lib._ptr(workspace),
        workspace.numel() * workspace.element_size(), _lib._stream(stream))
    _lib._check(rc, "dp_forward_write_keys")
    return out, h_final


def state_io(op, state, ext=None, transposed=False, stream=None):
    """ZERO / IMPORT (ext -> state) / EXPORT (state -> ext) of a [B,H,Dk,Dv] state."""
    _lib._need_cuda("state", state, torch.float32)
    _lib._need_cuda("ext", ext)
    B, H, Dk, Dv = state.shape
    ext_dt = _lib.DP_F32 if ext is None else _lib._dtype_code(ext.dtype)
    rc = _lib.lib().dp_state_io(int(op), B, H, Dk, Dv, _lib._ptr(state), _lib._ptr(ext),
                                ext_dt, int(bool(transposed)), _lib._stream(stream))
    _lib._check(rc, "dp_state_io")
    return state if op != STATE_EXPORT else ext


def set_wait_fault(withhold_first_record=False, flag_wait_polls=0):
    """dp_test_set_wait_fault: fault injection for tests of the cooperative
    mode's bounded record wait (process-wide; ``set_wait_fault()`` restores
    normal operation)."""
    _lib._check(_lib.lib().dp_test_set_wait_fault(int(bool(withhold_first_record)), int(flag_wait_polls)),
                "dp_test_set_wait_fault")


def check_status(workspace, stream=None):
    """Synchronise and raise if the device recorded an error in ``workspace``."""
    _lib._need_cuda("workspace", workspace)
    _lib._check(_lib.lib().dp_check_status(_lib._ptr(workspace), _lib._stream(stream)),
                "dp_check_status")
