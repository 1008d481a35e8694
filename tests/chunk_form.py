"""Chunkwise-parallel form of the KDA recurrence, fp64 numpy (test helper).

The page's update ("Kimi (AI)", section "Kimi Delta Attention (KDA)") expands
to S_t = D_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T with
D_t = diag(alpha_t).  D_t acts on the left (value channels) and the projector
on the right (key channels), so they commute: every row of S runs a scalar-
gated delta rule with its own gate.  Inside a chunk of C tokens, with
gamma_t = prod_{j<=t} alpha_j (elementwise, per value channel), rescaling the
state by 1/gamma turns each row into a plain delta rule on values v_t/gamma_t,
whose C steps have the WY/UT form

    A = I + diag(beta) strict_lower(K K^T),   T = A^{-1}
    X = diag(beta) (V / Gamma - K S^T)        (C x d_v)
    U = T X
    O = Gamma * (Q S^T + tril_incl(Q K^T) U)
    S <- diag(gamma_C) (S + U^T K)

Padding a partial last chunk with alpha = 1, beta = 0 leaves S unchanged and
its rows are not emitted.  This file exists to check that derivation against
the oracle; it is not used by the CUDA path.
"""
from __future__ import annotations

import numpy as np


def run_sequence(q, k, v, alpha, beta, S0, C):
    """One (sequence, head): q, k [L, d_k]; v, alpha [L, d_v]; beta [L]; S0 [d_v, d_k]."""
    q, k, v, alpha, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, alpha, beta))
    L, d_k = k.shape
    d_v = v.shape[1]
    S = np.zeros((d_v, d_k)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((L, d_v))
    for c0 in range(0, L, C):
        n = min(C, L - c0)
        Kc = np.zeros((C, d_k)); Kc[:n] = k[c0:c0 + n]
        Qc = np.zeros((C, d_k)); Qc[:n] = q[c0:c0 + n]
        Vc = np.zeros((C, d_v)); Vc[:n] = v[c0:c0 + n]
        Ac = np.ones((C, d_v)); Ac[:n] = alpha[c0:c0 + n]
        bc = np.zeros(C); bc[:n] = beta[c0:c0 + n]
        G = np.cumprod(Ac, axis=0)
        A = np.eye(C) + bc[:, None] * np.tril(Kc @ Kc.T, -1)
        T = np.linalg.inv(A)
        X = bc[:, None] * (Vc / G - Kc @ S.T)
        U = T @ X
        O = G * (Qc @ S.T + np.tril(Qc @ Kc.T) @ U)
        S = G[-1][:, None] * (S + U.T @ Kc)
        o[c0:c0 + n] = O[:n]
    return o, S


def run_packed(q, k, v, alpha, beta, S0, cu_seqlens, C):
    """Packed batch: q, k [T, H, d_k]; v, alpha [T, H, d_v]; beta [T, H]; S0 [N, H, d_v, d_k] or None."""
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = len(cu_seqlens) - 1
    o = np.zeros((T, H, d_v))
    S_T = np.zeros((N, H, d_v, d_k))
    for n in range(N):
        a, b = int(cu_seqlens[n]), int(cu_seqlens[n + 1])
        for h in range(H):
            s0 = None if S0 is None else S0[n, h]
            o[a:b, h], S_T[n, h] = run_sequence(q[a:b, h], k[a:b, h], v[a:b, h],
                                                alpha[a:b, h], beta[a:b, h], s0, C)
    return o, S_T
