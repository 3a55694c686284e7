"""Comparison helpers for GPU-vs-oracle parity.

Tolerances (the DeltaProduct forward contract): fp32 inputs -> max |err| <= 1e-4
on outputs and final states; bf16 inputs (fp32 accumulation) -> max |err| <=
2e-2 * RMS(reference), each tensor against its own RMS.
"""
import numpy as np
import torch

TOL_F32_ABS = 1e-4
TOL_BF16_REL = 2e-2


def to_np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def err_stats(got, ref):
    got, ref = to_np(got), to_np(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return dict(max_abs=0.0, rms_ref=0.0, rel_max=0.0, rel_rms=0.0)
    d = got - ref
    rms_ref = float(np.sqrt(np.mean(ref * ref)))
    max_abs = float(np.max(np.abs(d)))
    rms_err = float(np.sqrt(np.mean(d * d)))
    assert np.all(np.isfinite(got)), "non-finite values in GPU result"
    return dict(max_abs=max_abs, rms_ref=rms_ref,
                rel_max=max_abs / max(rms_ref, 1e-30), rel_rms=rms_err / max(rms_ref, 1e-30))


def assert_parity(got, ref, dtype, what=""):
    s = err_stats(got, ref)
    if dtype == torch.float32 or dtype == "f32":
        assert s["max_abs"] <= TOL_F32_ABS, f"{what}: {s}"
    else:
        assert s["rel_max"] <= TOL_BF16_REL, f"{what}: {s}"
    return s
