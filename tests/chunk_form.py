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


def run_sequence(q, k, v, alpha, beta, S0, C, additive=False):
    """One (sequence, head): q, k [L, d_k]; v, alpha [L, d_v]; beta [L]; S0 [d_v, d_k].

    additive=True: the additive update of linear attention (no prediction), whose
    chunk form is this one with T = I and no K S^T term in X."""
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
        if additive:
            T = np.eye(C)
            X = bc[:, None] * (Vc / G)
        else:
            A = np.eye(C) + bc[:, None] * np.tril(Kc @ Kc.T, -1)
            T = np.linalg.inv(A)
            X = bc[:, None] * (Vc / G - Kc @ S.T)
        U = T @ X
        O = G * (Qc @ S.T + np.tril(Qc @ Kc.T) @ U)
        S = G[-1][:, None] * (S + U.T @ Kc)
        o[c0:c0 + n] = O[:n]
    return o, S


def run_packed(q, k, v, alpha, beta, S0, cu_seqlens, C, additive=False):
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
                                                alpha[a:b, h], beta[a:b, h], s0, C, additive)
    return o, S_T


def backward_sequence(q, k, v, alpha, beta, S0, dO, dS_T, C):
    """Reverse mode of ``run_sequence``, chunk by chunk, as the CUDA backward does it.

    One (sequence, head).  A forward sweep keeps the state at every chunk
    start; the backward sweep walks the chunks in reverse carrying
    D = dL/d(state at the chunk's end).  Inside a chunk, with the forward
    quantities Gamma, T, M = tril_incl(Q K^T), Y = V / Gamma - K S^T,
    U = T diag(beta) Y and P = Q S^T + M U (so O = Gamma * P):

        dS^ = diag(gamma_C) D                  (S_C = diag(gamma_C) (S + U^T K))
        dP  = Gamma * dO
        dU  = M^T dP + K dS^^T
        dX  = T^T dU,  dY = diag(beta) dX,  dT = dU (diag(beta) Y)^T
        dA  = -T^T dT T^T,  sdA = strict_lower(dA)
        dM  = tril_incl(dP U^T)
        dq  = dP S + dM K
        dk  = dM^T Q + U dS^ - dY S + diag(beta) sdA K + sdA^T diag(beta) K
        dv  = dY / Gamma
        dbeta_r = sum_i dX_ri Y_ri + k_r . (sdA K)_r
        E   = dO * Gamma * P - dY * V / Gamma,   E[C-1] += rowsum(dS^ * (S + U^T K))
        dalpha = reverse_cumsum(E) / alpha
        D   <- dS^ + dP^T Q - dY^T K           (gradient at the chunk's start)
    """
    q, k, v, alpha, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, alpha, beta))
    L, d_k = k.shape
    d_v = v.shape[1]
    S = np.zeros((d_v, d_k)) if S0 is None else np.array(S0, dtype=np.float64)
    nc = (L + C - 1) // C
    states = []
    chunks = []
    for c in range(nc):
        c0 = c * C
        n = min(C, L - c0)
        Kc = np.zeros((C, d_k)); Kc[:n] = k[c0:c0 + n]
        Qc = np.zeros((C, d_k)); Qc[:n] = q[c0:c0 + n]
        Vc = np.zeros((C, d_v)); Vc[:n] = v[c0:c0 + n]
        Ac = np.ones((C, d_v)); Ac[:n] = alpha[c0:c0 + n]
        bc = np.zeros(C); bc[:n] = beta[c0:c0 + n]
        dOc = np.zeros((C, d_v)); dOc[:n] = dO[c0:c0 + n]
        chunks.append((c0, n, Kc, Qc, Vc, Ac, bc, dOc))
        states.append(S.copy())
        G = np.cumprod(Ac, axis=0)
        T = np.linalg.inv(np.eye(C) + bc[:, None] * np.tril(Kc @ Kc.T, -1))
        U = T @ (bc[:, None] * (Vc / G - Kc @ S.T))
        S = G[-1][:, None] * (S + U.T @ Kc)
    dq = np.zeros((L, d_k)); dk = np.zeros((L, d_k))
    dv = np.zeros((L, d_v)); dal = np.zeros((L, d_v)); db = np.zeros(L)
    D = np.zeros((d_v, d_k)) if dS_T is None else np.array(dS_T, dtype=np.float64)
    for c in range(nc - 1, -1, -1):
        c0, n, Kc, Qc, Vc, Ac, bc, dOc = chunks[c]
        S = states[c]
        G = np.cumprod(Ac, axis=0)
        T = np.linalg.inv(np.eye(C) + bc[:, None] * np.tril(Kc @ Kc.T, -1))
        M = np.tril(Qc @ Kc.T)
        Y = Vc / G - Kc @ S.T
        U = T @ (bc[:, None] * Y)
        P = Qc @ S.T + M @ U
        dS_hat = G[-1][:, None] * D
        dP = G * dOc
        dU = M.T @ dP + Kc @ dS_hat.T
        dX = T.T @ dU
        dY = bc[:, None] * dX
        dT = dU @ (bc[:, None] * Y).T
        sdA = np.tril(-T.T @ dT @ T.T, -1)
        dM = np.tril(dP @ U.T)
        Z = sdA @ Kc
        dq_c = dP @ S + dM @ Kc
        dk_c = dM.T @ Qc + U @ dS_hat - dY @ S + bc[:, None] * Z + sdA.T @ (bc[:, None] * Kc)
        dv_c = dY / G
        db_c = np.sum(dX * Y, axis=1) + np.sum(Kc * Z, axis=1)
        E = dOc * G * P - dY * Vc / G
        E[-1] += np.sum(dS_hat * (S + U.T @ Kc), axis=1)
        dal_c = np.cumsum(E[::-1], axis=0)[::-1] / Ac
        D = dS_hat + dP.T @ Qc - dY.T @ Kc
        dq[c0:c0 + n] = dq_c[:n]; dk[c0:c0 + n] = dk_c[:n]
        dv[c0:c0 + n] = dv_c[:n]; dal[c0:c0 + n] = dal_c[:n]; db[c0:c0 + n] = db_c[:n]
    return dq, dk, dv, dal, db, D


def backward_packed(q, k, v, alpha, beta, S0, cu_seqlens, dO, dS_T, C):
    """``backward_sequence`` over a packed batch; returns a dict like ``oracle.backward``."""
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = len(cu_seqlens) - 1
    out = {"dq": np.zeros((T, H, d_k)), "dk": np.zeros((T, H, d_k)),
           "dv": np.zeros((T, H, d_v)), "dalpha": np.zeros((T, H, d_v)),
           "dbeta": np.zeros((T, H)), "dS0": np.zeros((N, H, d_v, d_k))}
    for n in range(N):
        a, b = int(cu_seqlens[n]), int(cu_seqlens[n + 1])
        for h in range(H):
            s0 = None if S0 is None else S0[n, h]
            ds = None if dS_T is None else dS_T[n, h]
            r = backward_sequence(q[a:b, h], k[a:b, h], v[a:b, h], alpha[a:b, h],
                                  beta[a:b, h], s0, dO[a:b, h], ds, C)
            for name, x in zip(("dq", "dk", "dv", "dalpha", "dbeta"), r[:5]):
                out[name][a:b, h] = x
            out["dS0"][n, h] = r[5]
    return out
