"""Independent f64 chunked (WY) evaluation of the KDA forward.  TEST INFRASTRUCTURE.

This is the same function as :func:`oracle.recurrent`, reorganised over chunks
of C tokens exactly as the method states it; the tests check that the two forms
agree to f64 round-off (one chunk, two chunks, many chunks, ragged tail).  It
shares no code with the recurrence or with the CUDA library.

Per chunk, with S the state entering the chunk and, per key channel c,
G_t = sum_{s <= t} g_s the in-chunk cumulative log decay (G_t <= 0) and
Gamma_t = exp(G_t):

    A[t, i] = beta_t * sum_c k[t,c] k[i,c] exp(G[t,c] - G[i,c])      (i < t)
    Tm      = (I + A)^{-1}                     (forward substitution)
    W       = Tm @ diag(beta) (K * Gamma)      U = Tm @ diag(beta) V
    Delta   = U - W @ S
    M[t, i] = sum_c q[t,c] k[i,c] exp(G[t,c] - G[i,c])               (i <= t)
    o       = scale * ((Q * Gamma) @ S + M @ Delta)
    S'      = diag(Gamma_last) S + (K * exp(G_last - G))^T @ Delta

The carry factor exp(G_last - G) is the one the kda-adjoint-2026-10-01 page
(section 2 and section 5b) fixes: a single exponential of the log-space
difference (its bug was exponentiating an already exponentiated G_last).
Every exponent used is <= 0, so nothing overflows.
"""
from __future__ import annotations

import numpy as np

from . import f64


def carry_decay(G: np.ndarray) -> np.ndarray:
    """exp(G_last - G) per token and channel for one chunk's cumulative log decay G (c, K)."""
    return np.exp(G[-1][None, :] - G)


def forward_substitution_inverse(A: np.ndarray) -> np.ndarray:
    """(I + A)^{-1} for strictly lower-triangular A, row by row (unit lower triangular)."""
    n = A.shape[0]
    Tm = np.zeros_like(A)
    for t in range(n):
        Tm[t, t] = 1.0
        # row t of (I + A) Tm = I:  Tm[t, :] = e_t - sum_{i<t} A[t, i] Tm[i, :]
        for i in range(t):
            Tm[t, :] -= A[t, i] * Tm[i, :]
    return Tm


def _pairwise_decay(G: np.ndarray) -> np.ndarray:
    """D[t, i, c] = exp(G[t,c] - G[i,c]) for i <= t, 0 above the diagonal."""
    c = G.shape[0]
    diff = G[:, None, :] - G[None, :, :]
    lower = np.tril(np.ones((c, c), dtype=bool))[:, :, None]
    return np.where(lower, np.exp(np.where(lower, diff, 0.0)), 0.0)


def chunk_step(S, q, k, v, g, beta, scale):
    """One chunk: returns (o_chunk, S_next).  Shapes: q,k,g (c,K); v (c,V); beta (c,)."""
    G = np.cumsum(g, axis=0)
    Gam = np.exp(G)
    D = _pairwise_decay(G)
    kk = np.einsum("tc,ic,tic->ti", k, k, D)
    A = beta[:, None] * np.tril(kk, -1)
    M = np.tril(np.einsum("tc,ic,tic->ti", q, k, D))
    Tm = forward_substitution_inverse(A)
    W = Tm @ (beta[:, None] * k * Gam)
    U = Tm @ (beta[:, None] * v)
    Delta = U - W @ S
    o = scale * ((q * Gam) @ S + M @ Delta)
    S_next = Gam[-1][:, None] * S + (k * carry_decay(G)).T @ Delta
    return o, S_next


def chunked_wy(q, k, v, g, beta, scale, h0=None, chunk: int = 16):
    """Chunked-form forward given the log decay g.  Returns (o, hT) in float64.

    T need not be a multiple of ``chunk``: the last chunk is simply shorter.
    """
    q, k, v, g, beta, h0 = (f64(a) for a in (q, k, v, g, beta, h0))
    B, H, T, K = q.shape
    V = v.shape[-1]
    o = np.zeros((B, H, T, V))
    hT = np.zeros((B, H, K, V))
    for b in range(B):
        for h in range(H):
            S = np.zeros((K, V)) if h0 is None else h0[b, h].copy()
            for s in range(0, T, chunk):
                e = min(s + chunk, T)
                o[b, h, s:e], S = chunk_step(S, q[b, h, s:e], k[b, h, s:e], v[b, h, s:e],
                                             g[b, h, s:e], beta[b, h, s:e], scale)
            hT[b, h] = S
    return o, hT
