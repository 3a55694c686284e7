"""Seeded synthetic workloads for the DeltaProduct forward recurrence.

This module only draws random inputs; it holds none of the recurrence's
arithmetic. The same tensors feed the CUDA path and the fp64 oracle (which
upcasts them exactly), so both sides see identical values.

Recipe (DeltaProduct paper, Sec.4 input generation: keys are SiLU then
L2-normalised, beta is sigmoid or 2*sigmoid, the gate lies in [0,1]):
  q    = L2norm(N(0,1))              over D_k
  k    = L2norm(SiLU(N(0,1)))        over D_k, n_h keys per token
  v    ~ N(0,1)
  beta = beta_max * sigmoid(N(0,1))  beta_max in {1, 2}
  g    = sigmoid(N(3,1))             gated workloads only
  h0   ~ N(0, h0_std^2), fp32        when h0_std > 0, else no initial state
Near-duplicate keys: for round(frac*T) tokens per (batch, head), chosen by a
seeded permutation, k_{t,j} = L2norm(k_{t,0} + 0.005 z_j) for j >= 1
(cosine about 0.998 at D_k = 128).
Draw order: q, k, v, beta, g, h0, then the near-duplicate permutation and
noise. Values are drawn in fp32 with ``torch.Generator().manual_seed(seed)``
and then rounded to bf16 (round to nearest even) for bf16 workloads.
"""
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    nh: int
    Dk: int
    Dv: int
    dtype: str            # "f32" or "bf16": type of q, k, v, beta, g and o
    beta_max: float       # 1.0 -> beta in [0,1]; 2.0 -> beta in [0,2]
    gated: bool = False
    h0_std: float = 0.0
    near_dup_frac: float = 0.0
    seed: int = 0

    def scaled(self, **kw):
        """Same recipe at other sizes (parity cases the oracle finishes fast)."""
        return replace(self, **kw)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def tokens(self):
        return self.B * self.T


# The five workloads: sizes, distributions and seeds.
TINY = Workload("tiny-b1h2t64-nh2-d32-f32", 1, 64, 2, 2, 32, 32, "f32", 2.0, seed=0)
BASE = Workload("b4h8t2048-nh2-d128-bf16", 4, 2048, 8, 2, 128, 128, "bf16", 1.0, seed=2)
NEARDUP = Workload("b8h16t4096-nh3-d128-bf16-neardup", 8, 4096, 16, 3, 128, 128, "bf16", 2.0,
                   near_dup_frac=0.2, seed=3)
GATED = Workload("b4h16t8192-nh4-d128-bf16-gated-h0", 4, 8192, 16, 4, 128, 128, "bf16", 2.0,
                 gated=True, h0_std=0.02, seed=4)
LONG = Workload("b1h16t32768-nh3-d128-bf16-long", 1, 32768, 16, 3, 128, 128, "bf16", 2.0, seed=5)
LONG_DECODE_SEED = 15
LONG_CALLS = 8            # carried calls of T/8 tokens each

ALL = (TINY, BASE, NEARDUP, GATED, LONG)


def _l2norm(x):
    return x / torch.linalg.vector_norm(x, dim=-1, keepdim=True).clamp_min(1e-12)


def make_inputs(w: Workload):
    """Return dict(q, k, v, beta, g, h0) of CPU tensors (g/h0 may be None)."""
    gen = torch.Generator().manual_seed(w.seed)
    B, T, H, nh, Dk, Dv = w.B, w.T, w.H, w.nh, w.Dk, w.Dv
    q = _l2norm(torch.randn(B, T, H, Dk, generator=gen))
    k = _l2norm(torch.nn.functional.silu(torch.randn(B, T, H, nh, Dk, generator=gen)))
    v = torch.randn(B, T, H, nh, Dv, generator=gen)
    beta = w.beta_max * torch.sigmoid(torch.randn(B, T, H, nh, generator=gen))
    g = torch.sigmoid(torch.randn(B, T, H, generator=gen) + 3.0) if w.gated else None
    h0 = (w.h0_std * torch.randn(B, H, Dk, Dv, generator=gen)) if w.h0_std > 0 else None
    if w.near_dup_frac > 0 and nh > 1 and T > 0:
        count = int(round(w.near_dup_frac * T))
        for b in range(B):
            for h in range(H):
                toks = torch.randperm(T, generator=gen)[:count]
                z = torch.randn(count, nh - 1, Dk, generator=gen)
                base = k[b, toks, h, 0]                       # [count, Dk]
                k[b, toks, h, 1:] = _l2norm(base[:, None, :] + 0.005 * z)
    dt = w.torch_dtype
    out = dict(q=q.to(dt).contiguous(), k=k.to(dt).contiguous(), v=v.to(dt).contiguous(),
               beta=beta.to(dt).contiguous(),
               g=None if g is None else g.to(dt).contiguous(),
               h0=None if h0 is None else h0.float().contiguous())
    return out


# dp_prologue_flags values (include/dp.h)
PRO_KEY_SILU_L2, PRO_QUERY_L2, PRO_BETA_SIGMOID, PRO_BETA_2SIGMOID, PRO_GATE_SIGMOID = 1, 2, 4, 8, 16


def prologue_flags(w: Workload):
    """The prologue that maps ``make_raw_inputs(w)`` to the recipe's inputs."""
    f = PRO_KEY_SILU_L2 | PRO_QUERY_L2 | (PRO_BETA_SIGMOID if w.beta_max == 1.0 else PRO_BETA_2SIGMOID)
    assert w.beta_max in (1.0, 2.0), w.beta_max
    return f | (PRO_GATE_SIGMOID if w.gated else 0)


def make_raw_inputs(w: Workload):
    """The draws of ``make_inputs`` before their element-wise maps (raw
    projections: q, k, beta, g unmapped; v and h0 as in make_inputs), in the
    same order from the same seed. Near-duplicate keys are a property of
    mapped keys and are not produced here."""
    assert w.near_dup_frac == 0, "near-duplicate keys have no raw form"
    gen = torch.Generator().manual_seed(w.seed)
    B, T, H, nh, Dk, Dv = w.B, w.T, w.H, w.nh, w.Dk, w.Dv
    q = torch.randn(B, T, H, Dk, generator=gen)
    k = torch.randn(B, T, H, nh, Dk, generator=gen)
    v = torch.randn(B, T, H, nh, Dv, generator=gen)
    beta = torch.randn(B, T, H, nh, generator=gen)
    g = (torch.randn(B, T, H, generator=gen) + 3.0) if w.gated else None
    h0 = (w.h0_std * torch.randn(B, H, Dk, Dv, generator=gen)) if w.h0_std > 0 else None
    dt = w.torch_dtype
    return dict(q=q.to(dt).contiguous(), k=k.to(dt).contiguous(), v=v.to(dt).contiguous(),
                beta=beta.to(dt).contiguous(), g=None if g is None else g.to(dt).contiguous(),
                h0=None if h0 is None else h0.float().contiguous())


def make_decode_inputs(w: Workload, steps: int, seed: int = LONG_DECODE_SEED):
    """Fresh per-step inputs for ``steps`` decode calls: leading dim = step.

    Shapes: q [steps,B,H,Dk], k [steps,B,H,nh,Dk], v [steps,B,H,nh,Dv],
    beta [steps,B,H,nh], g [steps,B,H] or None; same distributions as
    ``make_inputs``.
    """
    gen = torch.Generator().manual_seed(seed)
    B, H, nh, Dk, Dv = w.B, w.H, w.nh, w.Dk, w.Dv
    q = _l2norm(torch.randn(steps, B, H, Dk, generator=gen))
    k = _l2norm(torch.nn.functional.silu(torch.randn(steps, B, H, nh, Dk, generator=gen)))
    v = torch.randn(steps, B, H, nh, Dv, generator=gen)
    beta = w.beta_max * torch.sigmoid(torch.randn(steps, B, H, nh, generator=gen))
    g = torch.sigmoid(torch.randn(steps, B, H, generator=gen) + 3.0) if w.gated else None
    dt = w.torch_dtype
    return dict(q=q.to(dt).contiguous(), k=k.to(dt).contiguous(), v=v.to(dt).contiguous(),
                beta=beta.to(dt).contiguous(),
                g=None if g is None else g.to(dt).contiguous())


def algorithmic_bytes(w: Workload, with_state_io=True, out_bytes=None):
    """HBM bytes one forward call must move: q, k, v, beta, g, o, state I/O.
    ``out_bytes`` is the size of one element of o (default: the input size)."""
    el = 4 if w.dtype == "f32" else 2
    ob = el if out_bytes is None else out_bytes
    per_tok_head = (w.Dk + w.nh * w.Dk + w.nh * w.Dv + w.nh) * el + w.Dv * ob
    if w.gated:
        per_tok_head += el
    total = per_tok_head * w.B * w.T * w.H
    if with_state_io:
        state = w.B * w.H * w.Dk * w.Dv * 4
        total += state                     # final state written
        if w.h0_std > 0:
            total += state                 # initial state read
    return total


def algorithmic_flops(w: Workload):
    """(4 n_h + 2) D_k D_v per token-head (+ D_k D_v for the gate)."""
    per = (4 * w.nh + 2) * w.Dk * w.Dv + (w.Dk * w.Dv if w.gated else 0)
    return per * w.B * w.T * w.H
