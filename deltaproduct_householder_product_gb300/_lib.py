"""ctypes binding of libdp.so: argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
checks tensor placement/dtype, takes data pointers and the current torch
stream, and turns a non-zero dp_status into an exception. There is no CPU or
PyTorch fallback: without the compiled library every call raises.
"""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdp.so")

DP_F32, DP_BF16 = 0, 1
IMPLS = {"auto": 0, "recurrent": 1, "chunk_tc": 2}
STATE_ZERO, STATE_IMPORT, STATE_EXPORT = 0, 1, 2
STATUS = {0: "DP_OK", 1: "DP_ERR_INVALID_ARG", 2: "DP_ERR_UNSUPPORTED", 3: "DP_ERR_ALIGNMENT",
          4: "DP_ERR_WORKSPACE", 5: "DP_ERR_CUDA", 6: "DP_ERR_TIMEOUT", 7: "DP_ERR_DEVICE"}


class DPError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({_strerror(code)})")


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("Dk", ctypes.c_int), ("Dv", ctypes.c_int), ("nh", ctypes.c_int),
                ("dtype", ctypes.c_int), ("impl", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("max_seqlen", ctypes.c_int), ("prologue", ctypes.c_int)]


_LIB = None
_vp = ctypes.c_void_p


def lib():
    """Load libdp.so (built by ``build.py``); raises if it is absent."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdp.so is not built ({LIB_PATH}); run "
                               "deltaproduct_householder_product_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        L.dp_abi_version.restype = ctypes.c_int
        L.dp_status_string.argtypes = [ctypes.c_int]
        L.dp_status_string.restype = ctypes.c_char_p
        L.dp_forward_workspace_size.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(ctypes.c_size_t)]
        L.dp_forward_workspace_size_fast.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(ctypes.c_size_t)]
        L.dp_forward_path.argtypes = [ctypes.POINTER(Dims), ctypes.c_size_t, ctypes.POINTER(ctypes.c_int)]
        L.dp_forward.argtypes = [ctypes.POINTER(Dims)] + [_vp] * 9 + [ctypes.c_size_t, _vp]
        L.dp_forward_varlen.argtypes = [ctypes.POINTER(Dims)] + [_vp] * 10 + [ctypes.c_size_t, _vp]
        L.dp_decode_step.argtypes = [ctypes.POINTER(Dims)] + [_vp] * 7 + [_vp]
        L.dp_state_io.argtypes = [ctypes.c_int] * 5 + [_vp, _vp, ctypes.c_int, ctypes.c_int, _vp]
        L.dp_check_status.argtypes = [_vp, _vp]
        L.dp_forward_noalloc.argtypes = [ctypes.POINTER(Dims)] + [_vp] * 9
        L.dp_backward_workspace_size.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(ctypes.c_size_t)]
        L.dp_backward.argtypes = [ctypes.POINTER(Dims)] + [_vp] * 15 + [ctypes.c_size_t, _vp]
        L.dp_prologue.argtypes = [ctypes.POINTER(Dims)] + [_vp] * 9
        L.dp_backward_varlen.argtypes = [ctypes.POINTER(Dims)] + [_vp] * 16 + [ctypes.c_size_t, _vp]
        L.dp_osdn_write_keys.argtypes = [ctypes.POINTER(Dims), _vp, _vp, _vp, _vp] + [ctypes.c_float] * 4 + \
            [_vp, _vp, _vp]
        L.dp_forward_write_keys.argtypes = [ctypes.POINTER(Dims)] + [_vp] * 10 + [ctypes.c_size_t, _vp]
        L.dp_test_set_wait_fault.argtypes = [ctypes.c_int, ctypes.c_uint]
        for name in ("dp_forward_workspace_size", "dp_forward_workspace_size_fast", "dp_forward_path",
                     "dp_forward", "dp_forward_varlen", "dp_decode_step",
                     "dp_state_io", "dp_check_status", "dp_forward_noalloc",
                     "dp_backward_workspace_size", "dp_backward", "dp_prologue",
                     "dp_osdn_write_keys", "dp_forward_write_keys", "dp_backward_varlen",
                     "dp_test_set_wait_fault"):
            getattr(L, name).restype = ctypes.c_int
        _LIB = L
    return _LIB


def _strerror(code):
    try:
        return lib().dp_status_string(code).decode()
    except Exception:
        return "?"


def _check(code, where):
    if code != 0:
        raise DPError(code, where)


def _dtype_code(t):
    if t == torch.float32:
        return DP_F32
    if t == torch.bfloat16:
        return DP_BF16
    raise TypeError(f"unsupported dtype {t}: use float32 or bfloat16")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(name, t, dtype=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")


PRO_KEY_SILU_L2, PRO_QUERY_L2, PRO_BETA_SIGMOID, PRO_BETA_2SIGMOID, PRO_GATE_SIGMOID = 1, 2, 4, 8, 16


def make_dims(B, T, H, Dk, Dv, nh, dtype, impl="auto", out_dtype=None, max_seqlen=0, prologue=0):
    dt = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    if out_dtype is None:
        od = dt
    else:
        od = out_dtype if isinstance(out_dtype, int) else _dtype_code(out_dtype)
    return Dims(B, T, H, Dk, Dv, nh, dt, IMPLS[impl] if isinstance(impl, str) else int(impl), od,
                max_seqlen, int(prologue))


PATHS = {0: "recurrent", 1: "chunk_fused", 2: "chunk_split", 3: "chunk_coop", 4: "chunk_seg"}
LAUNCHES = {"recurrent": 1, "chunk_fused": 1, "chunk_split": 2, "chunk_coop": 1, "chunk_seg": 4}


def forward_path(dims, workspace_bytes):
    """dp_forward_path: the path name dp_forward takes with this workspace."""
    code = ctypes.c_int(-1)
    _check(lib().dp_forward_path(ctypes.byref(dims), ctypes.c_size_t(workspace_bytes), ctypes.byref(code)),
           "dp_forward_path")
    return PATHS[code.value]


def backward_workspace_size(dims):
    """dp_backward_workspace_size."""
    n = ctypes.c_size_t(0)
    _check(lib().dp_backward_workspace_size(ctypes.byref(dims), ctypes.byref(n)), "dp_backward_workspace_size")
    return n.value


def workspace_size(dims, fast=False):
    """dp_forward_workspace_size, or dp_forward_workspace_size_fast if ``fast``."""
    n = ctypes.c_size_t(0)
    name = "dp_forward_workspace_size_fast" if fast else "dp_forward_workspace_size"
    _check(getattr(lib(), name)(ctypes.byref(dims), ctypes.byref(n)), name)
    return n.value
