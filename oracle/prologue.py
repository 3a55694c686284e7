"""Input prologue of DeltaProduct: raw projections -> keys, betas, gates.

TEST INFRASTRUCTURE ONLY (see the package docstring). Pure numpy fp64, no
shared code with the CUDA library.

DeltaProduct paper, Sec.4 (the per-token inputs): the j-th key of token i is
psi(W_j x_i) divided by its Euclidean norm, with psi = SiLU; the j-th beta
is phi(U_j x_i) with phi = sigmoid (beta in (0, 1)) or 2 sigmoid (beta in
(0, 2), which admits reflections). The gated variant's forget gate is a
sigmoid of its own projection. Queries are L2-normalised like the keys
(without SiLU) when the model does so; that step is an option here.

The projections themselves (W_j x_i, ...) are outside the path: this module
takes their outputs ("raw" inputs) and applies the element-wise maps and the
normalisation. ``forward`` is the prologue followed by the recurrence oracle.
"""
import numpy as np

KEY_SILU_L2 = 1
QUERY_L2 = 2
BETA_SIGMOID = 4
BETA_2SIGMOID = 8
GATE_SIGMOID = 16


def sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-x))


def silu(x):
    """SiLU(x) = x * sigmoid(x)."""
    x = np.asarray(x, dtype=np.float64)
    return x * sigmoid(x)


def l2_normalise(x):
    """x / ||x||_2 along the last axis (a zero row stays zero)."""
    x = np.asarray(x, dtype=np.float64)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return np.where(n > 0, x / np.where(n > 0, n, 1.0), 0.0)


def apply(flags, q, k, beta, g=None):
    """Returns (q, k, beta, g) after the prologue selected by ``flags``."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    if flags & KEY_SILU_L2:
        k = l2_normalise(silu(k))
    if flags & QUERY_L2:
        q = l2_normalise(q)
    if flags & BETA_SIGMOID:
        beta = sigmoid(beta)
    elif flags & BETA_2SIGMOID:
        beta = 2.0 * sigmoid(beta)
    if g is not None:
        g = np.asarray(g, dtype=np.float64)
        if flags & GATE_SIGMOID:
            g = sigmoid(g)
    return q, k, beta, g


def round_bf16(x):
    """Round to the nearest bfloat16 (ties to even), returned as fp64."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.bfloat16).double().numpy()


def forward(flags, q, k, v, beta, g=None, h0=None, threads=None, operand_dtype=None):
    """The prologue, then the sequential recurrence (``oracle.forward``).

    ``operand_dtype="bf16"``: the mapped keys and queries are rounded to
    bfloat16 before the recurrence, as the library states for bf16 inputs
    (they are tensor-core operands); betas and gates stay exact."""
    from . import forward as recurrence
    q2, k2, b2, g2 = apply(flags, _f64(q), _f64(k), _f64(beta), None if g is None else _f64(g))
    if operand_dtype == "bf16":
        if flags & KEY_SILU_L2:
            k2 = round_bf16(k2)
        if flags & QUERY_L2:
            q2 = round_bf16(q2)
    elif operand_dtype is not None:
        raise ValueError(operand_dtype)
    return recurrence(q2, k2, v, b2, g2, h0, threads=threads)


def _f64(x):
    if hasattr(x, "detach"):
        return x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)
