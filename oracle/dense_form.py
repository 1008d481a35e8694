"""Second oracle form: the KDA step as one explicit dense matrix product.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Substituting forget gating and predict into memory updating ("Kimi (AI)",
section "Kimi Delta Attention (KDA)") gives, per step,

    S_t = diag(alpha_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
    o_t = S_t q_t.

This module evaluates that expression with dense d x d numpy matrices in
fp64.  It is algebraically equal to the three-line form in ``kda_oracle.c``
but computed by a different route (one d_k x d_k projector per step), so the
two agreeing checks the C code's loops.  Cost is O(T d_v d_k^2): tiny sizes only.
"""
from __future__ import annotations

import numpy as np


def run(q, k, v, alpha, beta, S0=None):
    """One sequence, one head.  q, k: [T, d_k]; v, alpha: [T, d_v]; beta: [T].

    All inputs are float64 arrays.  Returns (o [T, d_v], S_T [d_v, d_k]).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    alpha = np.asarray(alpha, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    T, d_k = k.shape
    d_v = v.shape[1]
    S = np.zeros((d_v, d_k)) if S0 is None else np.array(S0, dtype=np.float64)
    eye = np.eye(d_k)
    o = np.zeros((T, d_v))
    for t in range(T):
        D = np.diag(alpha[t])
        projector = eye - beta[t] * np.outer(k[t], k[t])
        S = D @ S @ projector + beta[t] * np.outer(v[t], k[t])
        o[t] = S @ q[t]
    return o, S
