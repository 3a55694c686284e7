"""The chunked backward's formulas, checked in fp64 against the oracle's
backward (CPU only).

The CUDA chunked backward (csrc/backward_chunk.cu) differentiates the
chunk form of the recurrence (OSDN paper, App.A.2, with the gated decays of
the DeltaProduct paper, Sec.4): per chunk of ct tokens, A = I + tril(B (K
K^T o E), -1), T = A^-1, W = T diag(beta Gamma) K, U = T B V, U' = U - W S0,
S1 = Gamma_C S0 + Kd^T U' with Kd = diag(Gamma_C / Gamma) K, O =
diag(Gamma_last(t)) Q S0 + (Q K^T o E_last(t),s) U'. This file restates
those per-chunk gradient formulas in numpy (written here, sharing nothing
with the CUDA sources) and requires them to reproduce the oracle's
recurrent backward to 1e-10 for several chunk sizes, gated and not. It also
checks the direct form of dg the kernel uses (decay factors without the
gate, no division by it) against dlog(g) / g.
"""
import numpy as np
import pytest

import oracle


def chunked_backward(q, k, v, beta, g, h0, d_o, dhf, ct):
    B, T, H, nh, D = k.shape
    Dv = v.shape[-1]
    gated = g is not None
    dq, dk, dv, db = (np.zeros_like(x) for x in (q, k, v, beta))
    dg = np.zeros_like(g) if gated else None
    dg_direct = np.zeros_like(g) if gated else None
    dh0 = np.zeros((B, H, D, Dv))
    for b in range(B):
        for h in range(H):
            nc = -(-T // ct)
            S = h0[b, h].copy()
            saved = []
            for c in range(nc):                                  # forward: states at chunk starts
                t0, t1 = c * ct, min(T, (c + 1) * ct)
                nt = t1 - t0
                R = nt * nh
                K = k[b, t0:t1, h].reshape(R, D)
                V = v[b, t0:t1, h].reshape(R, Dv)
                be = beta[b, t0:t1, h].reshape(R)
                Q = q[b, t0:t1, h]
                lg = np.zeros(R)
                if gated:
                    lg[0::nh] = np.log(g[b, t0:t1, h])
                L = np.cumsum(lg)
                Gm = np.exp(L)
                gC = Gm[-1]
                E = np.exp(L[:, None] - L[None, :])
                KK = K @ K.T
                Tm = np.linalg.inv(np.eye(R) + np.tril(be[:, None] * KK * E, -1))
                W = Tm @ ((be * Gm)[:, None] * K)
                Up = Tm @ (be[:, None] * V) - W @ S
                last = np.arange(nt) * nh + nh - 1
                M = (np.arange(R)[None, :] <= last[:, None]).astype(float)
                Eq = E[last] * M
                Pr = (Q @ K.T) * M
                Kd = (gC / Gm)[:, None] * K
                saved.append((t0, t1, K, V, be, Q, lg, Gm, gC, E, KK, Tm, W, Up, last, M, Eq, Pr, Kd, S.copy()))
                S = gC * S + Kd.T @ Up
            dS = dhf[b, h].copy()
            for c in reversed(range(nc)):                        # reverse chain and per-chunk gradients
                t0, t1, K, V, be, Q, lg, Gm, gC, E, KK, Tm, W, Up, last, M, Eq, Pr, Kd, S0 = saved[c]
                nt = t1 - t0
                R = nt * nh
                dO = d_o[b, t0:t1, h]
                Gq = Gm[last]
                dS1 = dS
                dUp = (Pr * Eq).T @ dO + Kd @ dS1
                dS = gC * dS1 + Q.T @ (Gq[:, None] * dO) - W.T @ dUp
                dPe = dO @ Up.T * M
                dP = dPe * Eq
                dQ0 = dO @ S0.T
                dQ = Gq[:, None] * dQ0 + dP @ K
                dK = dP.T @ Q
                dGq = np.sum(Q * dQ0, 1)
                dEq = dPe * Pr
                dKd = Up @ dS1.T
                ratio = gC / Gm
                dK += ratio[:, None] * dKd
                dratio = np.sum(K * dKd, 1)
                dgC = np.sum(dS1 * S0)
                dW = -dUp @ S0.T
                dT = dW @ ((be * Gm)[:, None] * K).T + dUp @ (be[:, None] * V).T
                TdW, TdU = Tm.T @ dW, Tm.T @ dUp
                dK += (be * Gm)[:, None] * TdW
                dV = be[:, None] * TdU
                dbg = np.sum(K * TdW, 1)
                dbe = dbg * Gm + np.sum(V * TdU, 1)
                dG = np.tril(-Tm.T @ dT @ Tm.T, -1)
                dbe += np.sum(dG * KK * E, 1)
                Mx = be[:, None] * dG * E
                dK += Mx @ K + Mx.T @ K
                dq[b, t0:t1, h] = dQ
                dk[b, t0:t1, h] = dK.reshape(nt, nh, D)
                dv[b, t0:t1, h] = dV.reshape(nt, nh, Dv)
                db[b, t0:t1, h] = dbe.reshape(nt, nh)
                if not gated:
                    continue
                # coefficients of the decay factors
                cG = dbg * be                                    # of Gamma_r
                cG[last] += dGq
                cE = be[:, None] * dG * KK                       # of E[r][s], s < r
                np.add.at(cE, last, dEq)                         # the scores' decays sit on row last(t)
                cE = np.tril(cE, -1)                             # E[r][r] = 1 carries no gate
                # log-space: dL_r, then d log gamma = reverse cumsum, dg = / g
                dL = cG * Gm
                EE = cE * E
                dL += EE.sum(1) - EE.sum(0)
                dL -= dratio * ratio
                dL[-1] += np.sum(dratio * ratio) + dgC * gC
                dlg = np.cumsum(dL[::-1])[::-1]
                dg[b, t0:t1, h] = dlg[0::nh] / g[b, t0:t1, h]
                # direct: every factor containing gamma_r', without it
                for i in range(nt):
                    rp = i * nh
                    skip = lambda lo, hi: sum(lg[x] for x in range(lo, hi) if x != rp)
                    tot = dgC * np.exp(skip(0, R))
                    for r in range(R):
                        if r >= rp:
                            tot += cG[r] * np.exp(skip(0, r + 1))
                            for s in range(rp):
                                tot += cE[r, s] * np.exp(skip(s + 1, r + 1))
                        else:
                            tot += dratio[r] * np.exp(skip(r + 1, R))
                    dg_direct[b, t0 + i, h] = tot
            dh0[b, h] = dS
    return dict(dq=dq, dk=dk, dv=dv, dbeta=db, dg=dg, dh0=dh0), dg_direct


def _case(seed, B, T, H, nh, D, Dv, gated):
    rng = np.random.default_rng(seed)
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    q = rng.normal(size=(B, T, H, D))
    k = unit(rng.normal(size=(B, T, H, nh, D)))
    v = rng.normal(size=(B, T, H, nh, Dv))
    beta = rng.uniform(0.1, 1.9, size=(B, T, H, nh))
    g = rng.uniform(0.5, 0.99, size=(B, T, H)) if gated else None
    h0 = rng.normal(size=(B, H, D, Dv))
    d_o = rng.normal(size=(B, T, H, Dv))
    dhf = rng.normal(size=(B, H, D, Dv))
    return q, k, v, beta, g, h0, d_o, dhf


@pytest.mark.parametrize("gated", [False, True], ids=["ungated", "gated"])
@pytest.mark.parametrize("nh,ct", [(1, 7), (2, 5), (3, 1), (4, 13)])
def test_chunked_backward_matches_oracle(gated, nh, ct):
    q, k, v, beta, g, h0, d_o, dhf = _case(10 * nh + ct, 2, 13, 2, nh, 6, 5, gated)
    got, dg_direct = chunked_backward(q, k, v, beta, g, h0, d_o, dhf, ct)
    ref = oracle.backward(q, k, v, beta, g, h0, d_o, dhf, threads=1)
    for name in ("dq", "dk", "dv", "dbeta", "dg", "dh0"):
        if ref[name] is None:
            assert got[name] is None
            continue
        err = np.abs(got[name] - ref[name]).max()
        assert err <= 1e-10 * max(1.0, np.abs(ref[name]).max()), (name, err)
    if gated:
        assert np.abs(dg_direct - ref["dg"]).max() <= 1e-10 * max(1.0, np.abs(ref["dg"]).max())


def test_chunked_backward_gate_reductions():
    """g = 1 reduces the gated chunk form to the ungated one, and a gate
    below 1 moves every gradient (so the gated check above is not vacuous)."""
    q, k, v, beta, g, h0, d_o, dhf = _case(7, 1, 9, 1, 2, 4, 3, True)
    got, _ = chunked_backward(q, k, v, beta, g, h0, d_o, dhf, 4)
    ones = np.ones_like(g)
    got1, _ = chunked_backward(q, k, v, beta, ones, h0, d_o, dhf, 4)
    got0, _ = chunked_backward(q, k, v, beta, None, h0, d_o, dhf, 4)
    for name in ("dq", "dk", "dv", "dbeta", "dh0"):
        assert np.abs(got1[name] - got0[name]).max() < 1e-10
        assert np.abs(got[name] - got0[name]).max() > 1e-3
