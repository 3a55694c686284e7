"""Chunked UT/WY form of the DeltaProduct recurrence, in numpy fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring). This restates, on the
CPU and in plain numpy, the algebra the GPU path is built on, so that the
derivation itself is checked against the sequential recurrence before any
kernel is trusted. It shares no code with the CUDA library.

Sources:
* Extended sequence (DeltaProduct paper, Sec.5.1): the n_h keys/values/betas of
  every token are laid out one after another, giving a DeltaNet sequence of
  length T*n_h; the gate is expanded to (g_1, 1, ..., 1, g_2, 1, ...), and only
  the last output of every token's group is kept.
* Chunk transform (OSDN paper, App.A.2 and App.C, with the write key equal to
  the read key, in the H = S^T convention):
      T = (I + tril(diag(beta) K K^T, -1))^{-1},  W = T diag(beta) K,
      U = T diag(beta) V,  H_next = H + K^T (U - W H).
* Gate (DeltaProduct paper, Sec.4; OSDN paper, App.B: the residual is taken
  on the gated state). With Gamma_r the gate product from the chunk start to
  row r inclusive and E_rs = Gamma_r / Gamma_s (s <= r), induction on
  u_r = beta_r (v_r - (gamma_r H_{r-1})^T k_r) gives
      G   = tril(diag(beta) (K K^T * E), -1),  T = (I + G)^{-1}
      W   = T diag(beta * Gamma) K,  U = T diag(beta) V,  U_new = U - W H0
      H_C = Gamma_C H0 + K^T diag(E_{C,.}) U_new
      o_r = Gamma_r H0^T q + sum_{s<=r} E_rs (q . k_s) u_new_s
  which reduces to the ungated formulas above when every gate is 1.
Ratios E are formed as products of the gates between s and r, so a gate of
exactly zero (a reset) needs no special case here.
"""
import numpy as np


def _chunk_bounds(T, nh, chunk, token_aligned):
    N = T * nh
    if token_aligned:
        per = max(1, chunk // nh)          # whole tokens per chunk
        step = per * nh
    else:
        step = chunk
    return [(s, min(s + step, N)) for s in range(0, N, step)]


def forward(q, k, v, beta, g=None, h0=None, chunk=64, token_aligned=False):
    """Chunked forward. Same shapes/layouts as ``oracle.forward``.

    ``token_aligned=False`` cuts the extended sequence every ``chunk`` rows
    (chunks may straddle a token); ``True`` cuts after floor(chunk/nh) whole
    tokens. Both give the recurrence's result up to rounding.
    """
    q, k, v, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, beta))
    B, T, H, nh, Dk = k.shape
    Dv = v.shape[-1]
    N = T * nh
    o = np.zeros((B, T, H, Dv))
    hf = np.zeros((B, H, Dk, Dv))
    for b in range(B):
        for h in range(H):
            K = k[b, :, h].reshape(N, Dk)
            V = v[b, :, h].reshape(N, Dv)
            bet = beta[b, :, h].reshape(N)
            gam = np.ones(N)
            if g is not None:
                gam[0::nh] = np.asarray(g[b, :, h], dtype=np.float64)
            S = np.zeros((Dk, Dv)) if h0 is None else np.array(h0[b, h], dtype=np.float64)
            for (c0, c1) in _chunk_bounds(T, nh, chunk, token_aligned):
                C = c1 - c0
                Kc, Vc, bc, gc = K[c0:c1], V[c0:c1], bet[c0:c1], gam[c0:c1]
                # E[r, s] = prod(gc[s+1 .. r]) for s <= r; Gamma[r] = prod(gc[0 .. r])
                E = np.zeros((C, C))
                for r in range(C):
                    acc = 1.0
                    E[r, r] = 1.0
                    for s in range(r - 1, -1, -1):
                        acc *= gc[s + 1]
                        E[r, s] = acc
                Gam = np.cumprod(gc)
                G = np.tril((bc[:, None] * (Kc @ Kc.T)) * E, -1)
                Tm = np.linalg.inv(np.eye(C) + G)
                W = Tm @ ((bc * Gam)[:, None] * Kc)
                U = Tm @ (bc[:, None] * Vc)
                Un = U - W @ S
                for r in range(C):
                    if (c0 + r) % nh == nh - 1:          # last sub-step of a token
                        t = (c0 + r) // nh
                        qt = q[b, t, h]
                        scores = (Kc[: r + 1] @ qt) * E[r, : r + 1]
                        o[b, t, h] = Gam[r] * (S.T @ qt) + scores @ Un[: r + 1]
                S = Gam[-1] * S + Kc.T @ (E[C - 1][:, None] * Un)
            hf[b, h] = S
    return o, hf
