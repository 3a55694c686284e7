"""fp64 CPU oracle for the DeltaProduct forward recurrence.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the package smoke check
and by the bench's CPU-baseline leg, never by the product path. It shares no
code with the CUDA library and imports nothing from the package.

Three independent restatements live here:

* ``forward`` -- the plain sequential recurrence in C (``recurrence.c``):
  DeltaProduct paper, Sec.4 Eq.(2)-(3), gated variant and per-token
  pseudocode (Sec.4, Appendix B.1).
* ``backward`` -- reverse-mode gradients of that recurrence in C (the chain
  rule applied to each sub-step, readout and gate, in reverse token order).
* ``osdn`` -- the OSDN write-key variant: the phase-1 preconditioner scan
  (d-scan, optional APF retention) that emits the write keys k~ = d (.) k,
  then the recurrence above writing along k~.
* ``prologue`` -- the element-wise input maps of Sec.4 (SiLU and L2
  normalisation of keys, sigmoid / 2 sigmoid betas, sigmoid gates) applied
  to raw projections, in numpy fp64.
* ``product_form`` -- the per-token transition A_i = F_{n_h}...F_1 and write
  B_i = sum_j F_{n_h}...F_{j+1} C_j built by explicit matrix products
  (DeltaProduct paper, Sec.4, the expanded form of Eq.(3)).
* ``chunkwise`` -- the chunked UT/WY form (OSDN paper, App.A.2 / App.C, with
  the write key equal to the read key), extended to the per-token gate and
  the masked readout of the extended sequence (DeltaProduct paper, Sec.5.1).

Parity of every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` against the paper's worked example, closed forms,
invariants and brute force.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.oracle_forward.argtypes = [ctypes.c_int] * 6 + [dp] * 8 + [ctypes.c_int]
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_backward.argtypes = [ctypes.c_int] * 6 + [dp] * 14 + [ctypes.c_int]
        lib.oracle_forward_wk.argtypes = [ctypes.c_int] * 6 + [dp] * 9 + [ctypes.c_int]
        lib.oracle_forward_wk.restype = ctypes.c_int
        lib.oracle_backward.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def _as_f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor -> exact upcast on the CPU
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads():
    return max(1, os.cpu_count() or 1)


def forward(q, k, v, beta, g=None, h0=None, threads=None, kw=None):
    """Sequential fp64 recurrence. Returns (o [B,T,H,Dv], h_final [B,H,Dk,Dv]).

    ``kw`` [B,T,H,nh,Dk]: write keys (the OSDN variant writes the state along
    kw while the prediction error still reads with k); None = k.

    Shapes: q [B,T,H,Dk], k [B,T,H,nh,Dk], v [B,T,H,nh,Dv], beta [B,T,H,nh],
    g [B,T,H] or None, h0 [B,H,Dk,Dv] or None. Inputs of any float dtype
    (numpy or torch) are upcast exactly to fp64.
    """
    q, k, v, beta, g, h0, kw = (_as_f64(x) for x in (q, k, v, beta, g, h0, kw))
    B, T, H, nh, Dk = k.shape
    if kw is not None:
        assert kw.shape == k.shape, kw.shape
    Dv = v.shape[-1]
    assert q.shape == (B, T, H, Dk), q.shape
    assert v.shape == (B, T, H, nh, Dv), v.shape
    assert beta.shape == (B, T, H, nh), beta.shape
    if g is not None:
        assert g.shape == (B, T, H), g.shape
    if h0 is not None:
        assert h0.shape == (B, H, Dk, Dv), h0.shape
    o = np.zeros((B, T, H, Dv), dtype=np.float64)
    hf = np.zeros((B, H, Dk, Dv), dtype=np.float64)
    rc = _lib().oracle_forward_wk(B, T, H, Dk, Dv, nh, _ptr(q), _ptr(k), _ptr(kw), _ptr(v),
                                  _ptr(beta), _ptr(g), _ptr(h0), _ptr(o), _ptr(hf),
                                  int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_forward failed with code {rc}")
    return o, hf


def backward(q, k, v, beta, g=None, h0=None, d_o=None, dh_final=None, threads=None):
    """Gradients of L = <d_o, o> + <dh_final, h_final> through the recurrence
    (reverse mode, fp64). Returns dict dq, dk, dv, dbeta, dg (None when
    ungated), dh0, in the layouts of the corresponding inputs.

    d_o [B,T,H,Dv] (None = zeros), dh_final [B,H,Dk,Dv] or None (zeros).
    Memory: (T + 1) * Dk * Dv doubles per (batch, head) in flight.
    """
    q, k, v, beta, g, h0, d_o, dh_final = (_as_f64(x) for x in (q, k, v, beta, g, h0, d_o, dh_final))
    B, T, H, nh, Dk = k.shape
    Dv = v.shape[-1]
    assert q.shape == (B, T, H, Dk) and v.shape == (B, T, H, nh, Dv) and beta.shape == (B, T, H, nh)
    if d_o is None:
        d_o = np.zeros((B, T, H, Dv))
    assert d_o.shape == (B, T, H, Dv), d_o.shape
    if dh_final is not None:
        assert dh_final.shape == (B, H, Dk, Dv), dh_final.shape
    out = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v),
           "dbeta": np.zeros_like(beta), "dg": None if g is None else np.zeros_like(g),
           "dh0": np.zeros((B, H, Dk, Dv))}
    rc = _lib().oracle_backward(B, T, H, Dk, Dv, nh, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                                _ptr(h0), _ptr(d_o), _ptr(dh_final), _ptr(out["dq"]), _ptr(out["dk"]),
                                _ptr(out["dv"]), _ptr(out["dbeta"]), _ptr(out["dg"]), _ptr(out["dh0"]),
                                int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_backward failed with code {rc}")
    return out


def decode_step(q, k, v, beta, g, state, threads=None):
    """One token of the recurrence on a carried state.

    q [B,H,Dk], k [B,H,nh,Dk], v [B,H,nh,Dv], beta [B,H,nh], g [B,H] or None,
    state [B,H,Dk,Dv]. Returns (o [B,H,Dv], new_state). This is the same
    recurrence as ``forward`` with T = 1.
    """
    q, k, v, beta, g = (_as_f64(x) for x in (q, k, v, beta, g))
    o, hf = forward(q[:, None], k[:, None], v[:, None], beta[:, None],
                    None if g is None else g[:, None], state, threads)
    return o[:, 0], hf


from . import chunkwise, osdn, product_form, prologue  # noqa: E402,F401
