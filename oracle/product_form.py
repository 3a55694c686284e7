"""Product form of one DeltaProduct token, built by explicit matrix products.

TEST INFRASTRUCTURE ONLY (see the package docstring). Pure numpy fp64, no
shared code with ``recurrence.c``.

DeltaProduct paper, Sec.4, Eq.(3) and its expansion:
  F_{i,j} = I - beta_{i,j} k_{i,j} k_{i,j}^T        (generalised Householder)
  C_{i,j} = beta_{i,j} k_{i,j} v_{i,j}^T
  A_i = F_{i,n_h} ... F_{i,1}                       (earliest factor rightmost)
  B_i = sum_j F_{i,n_h} ... F_{i,j+1} C_{i,j}        (empty product = I)
  H_i = A_i H_{i-1} + B_i
Gated variant (Sec.4): H_{i,0} = g_i H_{i-1}, so A_i = g_i F_{i,n_h}...F_{i,1}
and B_i is unchanged.
"""
import numpy as np


def householder(k, b):
    """F = I - b k k^T."""
    k = np.asarray(k, dtype=np.float64)
    return np.eye(k.shape[0]) - b * np.outer(k, k)


def token_transition(keys, values, betas, gate=None):
    """(A_i, B_i) for one token with keys [nh,Dk], values [nh,Dv], betas [nh]."""
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    nh, Dk = keys.shape
    Fs = [householder(keys[j], betas[j]) for j in range(nh)]
    A = np.eye(Dk)
    for j in range(nh):
        A = Fs[j] @ A                      # later factors multiply on the left
    Bm = np.zeros((Dk, values.shape[1]))
    for j in range(nh):
        tail = np.eye(Dk)
        for m in range(j + 1, nh):
            tail = Fs[m] @ tail
        Bm = Bm + tail @ (betas[j] * np.outer(keys[j], values[j]))
    if gate is not None:
        A = gate * A
    return A, Bm


def forward(q, k, v, beta, g=None, h0=None):
    """Whole-sequence run of H_i = A_i H_{i-1} + B_i, o_i = H_i^T q_i.

    Same shapes and layouts as ``oracle.forward``; meant for tiny inputs.
    """
    q, k, v, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, beta))
    B, T, H, nh, Dk = k.shape
    Dv = v.shape[-1]
    o = np.zeros((B, T, H, Dv))
    hf = np.zeros((B, H, Dk, Dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((Dk, Dv)) if h0 is None else np.array(h0[b, h], dtype=np.float64)
            for t in range(T):
                gate = None if g is None else float(g[b, t, h])
                A, Bm = token_transition(k[b, t, h], v[b, t, h], beta[b, t, h], gate)
                S = A @ S + Bm
                o[b, t, h] = S.T @ q[b, t, h]
            hf[b, h] = S
    return o, hf
