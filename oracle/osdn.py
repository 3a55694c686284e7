"""OSDN write keys: the phase-1 preconditioner scan and the write-key forward.

TEST INFRASTRUCTURE ONLY (see the package docstring). numpy fp64 for the
scan; the recurrence is the C oracle with write keys.

OSDN paper (Improving Delta Rule with Provable Online Preconditioning),
Sec.4.1/4.3 Eqs.(2)/(5), Lemma 4.1 / Eq.(3), Alg.1, App.A.3:
  s_t = k_t (.) k_t, n_t = ||k_t||^2, nbar_t = max(n_t, eps)
  emit the write key k~_t = d_t (.) k_t with the CURRENT d_t, then
  d_{t+1} = clamp(r_t d_t + eta beta_t (1 - beta_t <d_t, s_t>) / nbar_t * s_t,
                  d_lo, d_hi)                         (projection onto [d_lo, d_hi]^K)
with d_1 = 1, eta = 0.003, [d_lo, d_hi] = [0.5, 2], eps = 1e-6 (the paper's
final configuration), r_t = 1 without APF and the given retention r_{t,h}
with APF (Sec.4.4). Phase 2 writes the state along k~ while the residual
still reads with k: H_t = H_{t-1} + beta_t k~_t (v_t - H_{t-1}^T k_t)^T.

Reading for DeltaProduct (n_h keys per token): the scan runs over the
extended sequence of T*n_h rows in order (one row per Householder step,
with its own key and beta); an APF retention r_{t,h} is per token and is
applied on the token's first row (like the gate, once per token).
"""
import numpy as np

ETA, D_LO, D_HI, EPS = 0.003, 0.5, 2.0, 1e-6


def dscan(k, beta, r=None, d0=None, eta=ETA, d_lo=D_LO, d_hi=D_HI, eps=EPS):
    """Returns (kw [B,T,H,nh,Dk], d_final [B,H,Dk]) for keys k [B,T,H,nh,Dk],
    betas [B,T,H,nh], APF retention r [B,T,H] or None, d0 [B,H,Dk] or None (ones)."""
    k = _f64(k)
    beta = _f64(beta)
    B, T, H, nh, Dk = k.shape
    d = np.ones((B, H, Dk)) if d0 is None else _f64(d0).copy()
    r = None if r is None else _f64(r)
    kw = np.zeros_like(k)
    for t in range(T):
        for j in range(nh):
            kk = k[:, t, :, j]                                   # [B,H,Dk]
            bt = beta[:, t, :, j][..., None]                     # [B,H,1]
            kw[:, t, :, j] = d * kk                              # emit with the current d
            s = kk * kk
            n = np.maximum(np.sum(s, axis=-1, keepdims=True), eps)
            a = bt * np.sum(d * s, axis=-1, keepdims=True)
            keep = r[:, t, :][..., None] if (r is not None and j == 0) else 1.0
            d = np.clip(keep * d + eta * bt * (1.0 - a) / n * s, d_lo, d_hi)
    return kw, d


def forward(q, k, v, beta, g=None, h0=None, r=None, d0=None, threads=None, **scan):
    """Phase 1 (d-scan) then phase 2 (write-key recurrence). Returns
    (o, h_final, kw, d_final)."""
    from . import forward as recurrence
    kw, d = dscan(k, beta, r, d0, **scan)
    o, hf = recurrence(q, k, v, beta, g, h0, threads=threads, kw=kw)
    return o, hf, kw, d


def _f64(x):
    if hasattr(x, "detach"):
        return x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)
