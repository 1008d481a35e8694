"""Pins for the oracle's reverse mode: facts fixed by calculus and by the page.

Each pin returns the largest relative deviation of ``oracle.backward`` from
something computed without it:

* central finite differences of the loss L = sum(dO * o) + sum(dS_T * S_T)
  through the dense matrix form of the recurrence (``oracle/dense_form.py``,
  itself pinned to the page in ``oracle_pins.py``), element by element on a
  tiny packed batch and along random directions on a larger one;
* closed forms: with beta = 0 the recurrence is pure decay, S_t = Gamma_t S0,
  so every gradient has an explicit formula; with alpha = 1, beta = 1, S0 = 0
  and orthonormal keys it is the page's naive linear attention, which fixes
  dq and dv.

Source: "Kimi (AI)" (Wikipedia mirror), section "Kimi Delta Attention (KDA)"
(the three-line update and the naive linear attention equation before it).
``test_oracle_mutants.py`` plants mistakes in the reverse-mode code and
checks that each one trips a pin.
"""
from __future__ import annotations

import numpy as np

import oracle
from oracle import dense_form
from oracle_pins import _f32, _hadamard, _rel, _random_problem

NAMES = ("dq", "dk", "dv", "dalpha", "dbeta", "dS0")


def _dense_loss(q, k, v, alpha, beta, S0, cu, dO, dS_T) -> float:
    """L = sum(dO * o) + sum(dS_T * S_T) through the dense matrix form, fp64."""
    H, d_k = q.shape[1], q.shape[2]
    d_v = v.shape[2]
    total = 0.0
    for n in range(len(cu) - 1):
        a, b = int(cu[n]), int(cu[n + 1])
        for h in range(H):
            s0 = np.zeros((d_v, d_k)) if S0 is None else S0[n, h]
            if b > a:
                o, S = dense_form.run(q[a:b, h], k[a:b, h], v[a:b, h], alpha[a:b, h],
                                      beta[a:b, h], s0)
                total += float(np.sum(dO[a:b, h] * o))
            else:
                S = s0
            if dS_T is not None:
                total += float(np.sum(dS_T[n, h] * S))
    return total


def _problem(rng, lengths, H, d_k, d_v, extra_tokens=0):
    q, k, v, alpha, beta, S0, cu = _random_problem(rng, lengths, H, d_k, d_v)
    if extra_tokens:
        pad = lambda x: np.concatenate([x, x[:extra_tokens] * 0 + 0.5], axis=0).astype(x.dtype)
        q, k, v, alpha, beta = (pad(x) for x in (q, k, v, alpha, beta))
    T = q.shape[0]
    dO = rng.standard_normal((T, H, d_v))
    dS_T = rng.standard_normal((len(lengths), H, d_v, d_k))
    return q, k, v, alpha, beta, S0, cu, dO, dS_T


def _as_f64(*xs):
    return [None if x is None else np.asarray(x, dtype=np.float64) for x in xs]


def pin_finite_differences_elementwise(lib) -> float:
    """Every gradient entry against a central difference of the dense-form loss,
    on two heads of a packed batch with an empty sequence and a token past the
    last sequence (whose gradients must be zero)."""
    rng = np.random.default_rng(21)
    lengths, H, d_k, d_v = [3, 0, 5], 2, 4, 3
    q, k, v, alpha, beta, S0, cu, dO, dS_T = _problem(rng, lengths, H, d_k, d_v, extra_tokens=1)
    g = oracle.backward(q, k, v, alpha, beta, S0, cu, dO, dS_T, lib=lib)
    xs = dict(zip(("q", "k", "v", "alpha", "beta", "S0"), _as_f64(q, k, v, alpha, beta, S0)))
    h = 1e-6
    err = 0.0
    for name, gname in zip(("q", "k", "v", "alpha", "beta", "S0"), NAMES):
        x = xs[name]
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = _dense_loss(xs["q"], xs["k"], xs["v"], xs["alpha"], xs["beta"], xs["S0"], cu,
                             dO, dS_T)
            x[idx] = old - h
            lm = _dense_loss(xs["q"], xs["k"], xs["v"], xs["alpha"], xs["beta"], xs["S0"], cu,
                             dO, dS_T)
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        err = max(err, _rel(g[gname], fd))
    return err


def pin_finite_differences_directional(lib) -> float:
    """<grad L, delta> against (L(x + h delta) - L(x - h delta)) / 2h for random
    directions delta in all six inputs at once, on a larger varlen batch."""
    rng = np.random.default_rng(22)
    lengths, H, d_k, d_v = [9, 1, 0, 14], 2, 8, 6
    q, k, v, alpha, beta, S0, cu, dO, dS_T = _problem(rng, lengths, H, d_k, d_v)
    g = oracle.backward(q, k, v, alpha, beta, S0, cu, dO, dS_T, lib=lib)
    base = _as_f64(q, k, v, alpha, beta, S0)
    h = 1e-6
    err = 0.0
    for _ in range(4):
        dirs = [rng.standard_normal(x.shape) for x in base]
        plus = [x + h * d for x, d in zip(base, dirs)]
        minus = [x - h * d for x, d in zip(base, dirs)]
        fd = (_dense_loss(*plus, cu, dO, dS_T) - _dense_loss(*minus, cu, dO, dS_T)) / (2 * h)
        an = sum(float(np.sum(g[n] * d)) for n, d in zip(NAMES, dirs))
        err = max(err, abs(an - fd) / max(abs(fd), 1.0))
    return err


def pin_pure_decay_gradients(lib) -> float:
    """beta = 0: S_t = diag(Gamma_t) S0 with Gamma_t = prod_{j<=t} alpha_j, so
    o_t = Gamma_t * (S0 q_t) and, writing D_t = sum_{s>=t} diag(Gamma_s / Gamma_t)
    dO_s q_s^T + diag(Gamma_T / Gamma_t) dS_T (the gradient reaching S_t):
      dq_t = S_t^T dO_t,  dk_t = 0,  dv_t = 0,
      dbeta_t = (v_t - S~_t k_t)^T D_t k_t with S~_t = diag(Gamma_t) S0,
      dS0 = sum_t diag(Gamma_t) dO_t q_t^T + diag(Gamma_T) dS_T,
      dalpha_t = (sum_{s>=t} dO_s * Gamma_s * (S0 q_s) + Gamma_T * rowsum(dS_T * S0)) / alpha_t."""
    rng = np.random.default_rng(23)
    lengths, H, d_k, d_v = [10], 2, 6, 5
    q, k, v, alpha, beta, S0, cu, dO, dS_T = _problem(rng, lengths, H, d_k, d_v)
    beta = np.zeros_like(beta)
    g = oracle.backward(q, k, v, alpha, beta, S0, cu, dO, dS_T, lib=lib)
    qf, kf, vf, af = _as_f64(q, k, v, alpha)
    T = lengths[0]
    err = max(_rel(g["dk"], np.zeros_like(g["dk"])), _rel(g["dv"], np.zeros_like(g["dv"])))
    for h in range(H):
        s0 = S0[0, h]
        gam = np.cumprod(af[:, h], axis=0)            # [T, d_v]
        dq = np.stack([(gam[t][:, None] * s0).T @ dO[t, h] for t in range(T)])
        dS0 = sum(np.outer(gam[t] * dO[t, h], qf[t, h]) for t in range(T)) + gam[-1][:, None] * dS_T[0, h]
        per_tok = np.stack([dO[t, h] * gam[t] * (s0 @ qf[t, h]) for t in range(T)])
        tail = gam[-1] * np.sum(dS_T[0, h] * s0, axis=1)
        rev = np.cumsum(per_tok[::-1], axis=0)[::-1] + tail
        dalpha = rev / af[:, h]
        dbeta = np.zeros(T)
        for t in range(T):
            D = gam[-1][:, None] / gam[t][:, None] * dS_T[0, h]
            for s in range(t, T):
                D = D + np.outer(gam[s] / gam[t] * dO[s, h], qf[s, h])
            u = vf[t, h] - (gam[t][:, None] * s0) @ kf[t, h]
            dbeta[t] = u @ (D @ kf[t, h])
        err = max(err, _rel(g["dq"][:, h], dq), _rel(g["dS0"][0, h], dS0),
                  _rel(g["dalpha"][:, h], dalpha), _rel(g["dbeta"][:, h], dbeta))
    return err


def pin_naive_linear_attention_gradients(lib) -> float:
    """alpha = 1, beta = 1, S0 = 0, orthonormal keys: the page's naive linear
    attention, S_t = sum_{i<=t} v_i k_i^T.  Perturbing v_i adds e k_i^T to every
    later state (the later projectors leave k_i alone), so
      dv_i = sum_{t>=i} (k_i . q_t) dO_t + dS_T k_i,   dq_t = sum_{i<=t} (v_i . dO_t) k_i."""
    rng = np.random.default_rng(24)
    T, H, d = 12, 2, 16
    had = _hadamard(d) / 4.0
    perm = np.stack([rng.permutation(d)[:T] for _ in range(H)], axis=1)
    k = _f32(np.stack([had[perm[:, h]] for h in range(H)], axis=1))
    q = _f32(rng.standard_normal((T, H, d)))
    v = _f32(rng.standard_normal((T, H, d)))
    alpha = np.ones((T, H, d), np.float32)
    beta = np.ones((T, H), np.float32)
    cu = np.array([0, T], np.int32)
    dO = rng.standard_normal((T, H, d))
    dS_T = rng.standard_normal((1, H, d, d))
    g = oracle.backward(q, k, v, alpha, beta, None, cu, dO, dS_T, lib=lib)
    qf, kf, vf = _as_f64(q, k, v)
    err = 0.0
    for h in range(H):
        dv = np.stack([sum((kf[i, h] @ qf[t, h]) * dO[t, h] for t in range(i, T)) +
                       dS_T[0, h] @ kf[i, h] for i in range(T)])
        dq = np.stack([sum((vf[i, h] @ dO[t, h]) * kf[i, h] for i in range(t + 1))
                       for t in range(T)])
        err = max(err, _rel(g["dv"][:, h], dv), _rel(g["dq"][:, h], dq))
    return err


def pin_gate_layout_chain_rules(lib) -> float:
    """One gate per head drives every value channel, so its gradient is the sum
    of the per-channel gradients; for log alpha it is alpha times the
    per-channel gradient.  Both checked by central differences of the dense-form
    loss with the gate expanded (the reductions the gate-layout tests apply to
    the oracle's per-channel gradient)."""
    rng = np.random.default_rng(25)
    lengths, H, d_k, d_v = [4, 3], 2, 4, 3
    q, k, v, alpha, beta, S0, cu, dO, dS_T = _problem(rng, lengths, H, d_k, d_v)
    T = q.shape[0]
    head = alpha[:, :, :1].astype(np.float64)                     # [T, H, 1]
    logs = np.log(alpha.astype(np.float64))                         # [T, H, d_v]
    a_head = np.ascontiguousarray(np.broadcast_to(head, (T, H, d_v)), dtype=np.float32)
    g_head = oracle.backward(q, k, v, a_head, beta, S0, cu, dO, dS_T, lib=lib)["dalpha"].sum(axis=2)
    g_log = oracle.backward(q, k, v, alpha, beta, S0, cu, dO, dS_T, lib=lib)["dalpha"] * np.exp(logs)
    qf, kf, vf, bf, s0 = _as_f64(q, k, v, beta, S0)
    h = 1e-6
    fd_head = np.zeros((T, H))
    for t in range(T):
        for hh in range(H):
            pm = []
            for sgn in (1, -1):
                a = np.broadcast_to(head, (T, H, d_v)).copy()
                a[t, hh, :] += sgn * h
                pm.append(_dense_loss(qf, kf, vf, a, bf, s0, cu, dO, dS_T))
            fd_head[t, hh] = (pm[0] - pm[1]) / (2 * h)
    fd_log = np.zeros((T, H, d_v))
    for idx in np.ndindex(T, H, d_v):
        pm = []
        for sgn in (1, -1):
            lg = logs.copy()
            lg[idx] += sgn * h
            pm.append(_dense_loss(qf, kf, vf, np.exp(lg), bf, s0, cu, dO, dS_T))
        fd_log[idx] = (pm[0] - pm[1]) / (2 * h)
    return max(_rel(g_head, fd_head), _rel(g_log, fd_log))


# name -> (function, tolerance).  Finite differences with h = 1e-6 in fp64 are
# good to about 1e-9 relative here; the closed forms to a few hundred roundings.
PINS = {
    "fd_elementwise": (pin_finite_differences_elementwise, 1e-7),
    "fd_directional": (pin_finite_differences_directional, 1e-7),
    "pure_decay_gradients": (pin_pure_decay_gradients, 1e-12),
    "naive_linear_attention_gradients": (pin_naive_linear_attention_gradients, 1e-12),
    "gate_layout_chain_rules": (pin_gate_layout_chain_rules, 1e-7),
}


def failing_pins(lib) -> list[str]:
    """Names of reverse-mode pins that a given oracle build violates."""
    bad = []
    for name, (fn, tol) in PINS.items():
        try:
            err = fn(lib)
        except Exception:
            bad.append(name)
            continue
        if not np.isfinite(err) or err > tol:
            bad.append(name)
    return bad
