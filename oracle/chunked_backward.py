"""Independent f64 chunked evaluation of the KDA backward.  TEST INFRASTRUCTURE.

The gradients of the chunked form (``oracle.chunked``) taken chunk by chunk in reverse:
the same function as ``oracle.backward`` (reverse mode through the token recurrence),
organised as the chunk-level adjoint equations.  Per chunk, with S the state entering it,
G the in-chunk cumulative log decay, Gamma = e^G, gamma = e^{G_last}, Kg = K Gamma,
Qg = Q Gamma, Kt = K e^{G_last - G}, A'[t,i] = sum_c k_tc k_ic e^{G_tc - G_ic} (i < t),
M[t,i] = sum_c q_tc k_ic e^{G_tc - G_ic} (i <= t), T = (I + diag(beta) A')^{-1},
R = V - Kg S and Delta = T diag(beta) R, the forward is
    o = scale (Qg S + M Delta),   S_out = diag(gamma) S + Kt^T Delta,
and with dS the adjoint of S_out and dO that of the chunk's outputs:
    dDelta = Kt dS + scale M^T dO,    dY = T^T dDelta,    dR = diag(beta) dY,
    dKt = Delta dS^T,  dgamma = rowsum(S .* dS),  dQg = scale dO S^T,  dKg = -dR S^T,
    dM = scale dO Delta^T (i <= t),   dB = -dY Delta^T (i < t),  dA' = diag(beta) dB,
    dbeta = rowsum(R .* dY) + rowsum(A' .* dB),   dV = dR,
    the pairwise terms of dA' and dM, the Gamma factors, and
    dS <- diag(gamma) dS + scale Qg^T dO - Kg^T dR;
dg is the reverse in-chunk cumulative sum of dG.  The tests check it against the token
reverse mode to f64 round-off at several chunk sizes and ragged lengths.
"""
from __future__ import annotations

import numpy as np

from . import f64
from .chunked import _pairwise_decay, forward_substitution_inverse


def chunked_backward(q, k, v, g, beta, scale, h0, d_o, dhT=None, chunk: int = 16) -> dict:
    """Gradients dq, dk, dv, dg (B,H,T,.), dbeta (B,H,T) and dh0 (B,H,K,V), given the log
    decay g (the gate's own derivative is elementwise and not repeated here)."""
    q, k, v, g, beta, h0, d_o, dhT = (f64(a) for a in (q, k, v, g, beta, h0, d_o, dhT))
    B, H, T, K = q.shape
    V = v.shape[-1]
    out = {n: np.zeros((B, H, T, K)) for n in ("dq", "dk", "dg")}
    out["dv"] = np.zeros((B, H, T, V))
    out["dbeta"] = np.zeros((B, H, T))
    out["dh0"] = np.zeros((B, H, K, V))
    starts = list(range(0, T, chunk))
    for b in range(B):
        for h in range(H):
            # forward: the state entering each chunk
            S = np.zeros((K, V)) if h0 is None else h0[b, h].copy()
            states = []
            for s in starts:
                e = min(s + chunk, T)
                states.append(S.copy())
                G = np.cumsum(g[b, h, s:e], axis=0)
                D = _pairwise_decay(G)
                kc, bc = k[b, h, s:e], beta[b, h, s:e]
                Ap = np.tril(np.einsum("tc,ic,tic->ti", kc, kc, D), -1)
                Tm = forward_substitution_inverse(bc[:, None] * Ap)
                R = v[b, h, s:e] - (kc * np.exp(G)) @ S
                Dl = Tm @ (bc[:, None] * R)
                S = np.exp(G[-1])[:, None] * S + (kc * np.exp(G[-1][None, :] - G)).T @ Dl
            # reverse
            dS = np.zeros((K, V)) if dhT is None else dhT[b, h].copy()
            for n in range(len(starts) - 1, -1, -1):
                s = starts[n]
                e = min(s + chunk, T)
                S = states[n]
                qc, kc, vc, bc = q[b, h, s:e], k[b, h, s:e], v[b, h, s:e], beta[b, h, s:e]
                doc = d_o[b, h, s:e]
                G = np.cumsum(g[b, h, s:e], axis=0)
                Gam, gl = np.exp(G), G[-1]
                gam = np.exp(gl)
                eL = np.exp(gl[None, :] - G)
                D = _pairwise_decay(G)
                Ap = np.tril(np.einsum("tc,ic,tic->ti", kc, kc, D), -1)
                M = np.tril(np.einsum("tc,ic,tic->ti", qc, kc, D))
                Tm = forward_substitution_inverse(bc[:, None] * Ap)
                Kg, Qg, Kt = kc * Gam, qc * Gam, kc * eL
                R = vc - Kg @ S
                Dl = Tm @ (bc[:, None] * R)
                # adjoints
                dDl = Kt @ dS + scale * M.T @ doc
                dY = Tm.T @ dDl
                dR = bc[:, None] * dY
                dKt = Dl @ dS.T
                dgam = (S * dS).sum(axis=1)
                dQg = scale * doc @ S.T
                dKg = -dR @ S.T
                dM = np.tril(scale * doc @ Dl.T)
                dB = np.tril(-dY @ Dl.T, -1)
                dAp = bc[:, None] * dB
                # pairwise terms: A'_ti and M_ti as functions of k_t, q_t (row) and k_i (column)
                row_a = np.einsum("ti,ic,tic->tc", dAp, kc, D)
                row_m = np.einsum("ti,ic,tic->tc", dM, kc, D)
                col_a = np.einsum("ti,tc,tic->ic", dAp, kc, D)
                col_m = np.einsum("ti,tc,tic->ic", dM, qc, D)
                dq = row_m + dQg * Gam
                dk = row_a + col_a + col_m + dKg * Gam + dKt * eL
                dG = (kc * row_a + qc * row_m - kc * (col_a + col_m)
                      + dQg * qc * Gam + dKg * kc * Gam - dKt * kc * eL)
                dG[-1] += (dKt * kc * eL).sum(axis=0) + dgam * gam
                out["dq"][b, h, s:e] = dq
                out["dk"][b, h, s:e] = dk
                out["dv"][b, h, s:e] = dR
                out["dg"][b, h, s:e] = np.cumsum(dG[::-1], axis=0)[::-1]
                out["dbeta"][b, h, s:e] = (R * dY).sum(axis=1) + (Ap * dB).sum(axis=1)
                dS = gam[:, None] * dS + scale * Qg.T @ doc - Kg.T @ dR
            out["dh0"][b, h] = dS
    return out
