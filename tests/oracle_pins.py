"""Pins for the KDA oracle: facts fixed by the page and by mathematics.

Each pin builds inputs for which the answer is known without running the
recurrence (a closed form, a reduction to the page's naive linear attention,
an identity of the delta rule) or an invariant the recurrence must satisfy,
runs the oracle, and returns the largest relative deviation.  The same
functions run against deliberately broken copies of the oracle in
``test_oracle_mutants.py``: every planted mistake must trip at least one pin.

Source: "Kimi (AI)" (Wikipedia mirror), section "Kimi Delta Attention (KDA)":
the naive linear attention equation o_t = (sum_{i<=t} v_i k_i^T) q_t with
S_t = S_{t-1} + v_t k_t^T, and the three-line update (forget gating, predict,
memory updating).
"""
from __future__ import annotations

import numpy as np

import oracle
from oracle import dense_form


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (nearest-even) and return the bit patterns."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def _f32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _hadamard(n: int) -> np.ndarray:
    h = np.array([[1.0]])
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def _rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def pin_naive_linear_attention(lib) -> float:
    """alpha = 1, beta = 1, S0 = 0 and mutually orthonormal keys: the prediction
    S~_t k_t is zero, so KDA reduces to the page's naive linear attention
    o_t = (sum_{i<=t} v_i k_i^T) q_t.  Keys are scaled Hadamard rows (exact in
    bf16), q and v random bf16."""
    rng = np.random.default_rng(1)
    T, H, d = 16, 2, 16
    had = _hadamard(d) / 4.0                     # rows are orthonormal, entries +-1/4
    perm = np.stack([rng.permutation(d)[:T] for _ in range(H)], axis=1)   # [T, H]
    k = np.stack([had[perm[:, h]] for h in range(H)], axis=1)           # [T, H, d]
    q_bits = _bf16_bits(rng.standard_normal((T, H, d)))
    v_bits = _bf16_bits(rng.standard_normal((T, H, d)))
    k_bits = _bf16_bits(k)
    alpha = np.ones((T, H, d), np.float32)
    beta = np.ones((T, H), np.float32)
    cu = np.array([0, T], np.int32)
    o, S_T = oracle.prefill(q_bits, k_bits, v_bits, alpha, beta, None, cu, lib=lib)
    qf, kf, vf = (oracle.bf16_bits_to_f64(x) for x in (q_bits, k_bits, v_bits))
    err = 0.0
    for h in range(H):
        M = np.zeros((d, d))
        for t in range(T):
            M = M + np.outer(vf[t, h], kf[t, h])
            err = max(err, _rel(o[t, h], M @ qf[t, h]))
        err = max(err, _rel(S_T[0, h], M))
    return err


def pin_pure_decay(lib) -> float:
    """beta = 0 removes memory updating: S_t = diag(prod_{j<=t} alpha_j) S0 and
    o_t = S_t q_t.  Random per-channel alpha and a random S0 make the side of
    diag(alpha) visible (rows = value channels)."""
    rng = np.random.default_rng(2)
    T, H, d_k, d_v = 12, 3, 8, 8
    q = _f32(rng.standard_normal((T, H, d_k)))
    k = _f32(rng.standard_normal((T, H, d_k)))
    v = _f32(rng.standard_normal((T, H, d_v)))
    alpha = _f32(rng.uniform(0.3, 1.0, (T, H, d_v)))
    beta = np.zeros((T, H), np.float32)
    S0 = rng.standard_normal((1, H, d_v, d_k))
    o, S_T = oracle.prefill(q, k, v, alpha, beta, S0, np.array([0, T], np.int32), lib=lib)
    err = 0.0
    for h in range(H):
        g = np.ones(d_v)
        for t in range(T):
            g = g * alpha[t, h].astype(np.float64)
            St = g[:, None] * S0[0, h]
            err = max(err, _rel(o[t, h], St @ q[t, h].astype(np.float64)))
        err = max(err, _rel(S_T[0, h], g[:, None] * S0[0, h]))
    return err


def pin_delta_write(lib) -> float:
    """One step from a known state with a unit key and q = k.  Memory updating
    gives S_1 k = (1 - beta) S~ k + beta v with S~ = diag(alpha) S0 (the
    prediction uses the decayed state), so o_1 = (1 - beta) diag(alpha) S0 k + beta v;
    with beta = 1 the output is exactly v.  Many independent length-1 sequences."""
    rng = np.random.default_rng(3)
    N, H, d = 40, 2, 16
    had = _hadamard(d) / 4.0
    k = had[rng.integers(0, d, (N, H))] * rng.choice([-1.0, 1.0], (N, H, 1))
    k_bits = _bf16_bits(k)
    v_bits = _bf16_bits(rng.standard_normal((N, H, d)))
    alpha = _f32(rng.uniform(0.2, 1.0, (N, H, d)))
    beta = _f32(rng.uniform(0.0, 1.0, (N, H)))
    beta[: N // 2] = 1.0
    S0 = rng.standard_normal((N, H, d, d))
    cu = np.arange(N + 1, dtype=np.int32)
    o, S_T = oracle.prefill(k_bits, k_bits, v_bits, alpha, beta, S0, cu, lib=lib)
    kf, vf = oracle.bf16_bits_to_f64(k_bits), oracle.bf16_bits_to_f64(v_bits)
    err = 0.0
    for n in range(N):
        for h in range(H):
            b = float(beta[n, h])
            pred = alpha[n, h].astype(np.float64) * (S0[n, h] @ kf[n, h])
            expect = (1.0 - b) * pred + b * vf[n, h]
            err = max(err, _rel(o[n, h], expect))
            err = max(err, _rel(S_T[n, h] @ kf[n, h], expect))
    return err


def pin_scalar_geometric(lib) -> float:
    """d_k = d_v = 1 with constant alpha, beta, k = 1 and v: the update is
    s_t = a s_{t-1} + beta v with a = alpha (1 - beta), a geometric series with
    closed form s_t = a^t s_0 + beta v (1 - a^t) / (1 - a); o_t = s_t q_t."""
    T = 40
    alpha_c, beta_c, v_c, q_c, s0 = 0.875, 0.375, 1.5, -0.75, 2.0
    q = np.full((T, 1, 1), q_c, np.float32)
    k = np.ones((T, 1, 1), np.float32)
    v = np.full((T, 1, 1), v_c, np.float32)
    alpha = np.full((T, 1, 1), alpha_c, np.float32)
    beta = np.full((T, 1), beta_c, np.float32)
    S0 = np.full((1, 1, 1, 1), s0)
    o, S_T = oracle.prefill(q, k, v, alpha, beta, S0, np.array([0, T], np.int32), lib=lib)
    a = alpha_c * (1.0 - beta_c)
    t = np.arange(1, T + 1, dtype=np.float64)
    s = a ** t * s0 + beta_c * v_c * (1.0 - a ** t) / (1.0 - a)
    return max(_rel(o[:, 0, 0], s * q_c), _rel(S_T[0, 0, 0, 0], s[-1]))


def _random_problem(rng, lengths, H, d_k, d_v, s0=True, unit_keys=False):
    T = int(sum(lengths))
    q = _f32(rng.standard_normal((T, H, d_k)))
    k = rng.standard_normal((T, H, d_k))
    if unit_keys:
        k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    k = _f32(k * (1.0 if unit_keys else 0.4))
    v = _f32(rng.standard_normal((T, H, d_v)))
    alpha = _f32(rng.uniform(0.5, 1.0, (T, H, d_v)))
    beta = _f32(rng.uniform(0.0, 1.0, (T, H)))
    N = len(lengths)
    S0 = rng.standard_normal((N, H, d_v, d_k)) * 0.3 if s0 else None
    cu = np.zeros(N + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    return q, k, v, alpha, beta, S0, cu


def pin_dense_matrix_form(lib) -> float:
    """The oracle's loops against the same recurrence written as one dense
    matrix product per step, S_t = D_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
    (oracle/dense_form.py), on small random problems with d_k != d_v."""
    rng = np.random.default_rng(4)
    lengths = [7, 1, 13]
    H, d_k, d_v = 2, 5, 6
    q, k, v, alpha, beta, S0, cu = _random_problem(rng, lengths, H, d_k, d_v)
    o, S_T = oracle.prefill(q, k, v, alpha, beta, S0, cu, lib=lib)
    err = 0.0
    for n in range(len(lengths)):
        a, b = cu[n], cu[n + 1]
        for h in range(H):
            od, Sd = dense_form.run(q[a:b, h], k[a:b, h], v[a:b, h], alpha[a:b, h],
                                    beta[a:b, h], S0[n, h])
            err = max(err, _rel(o[a:b, h], od), _rel(S_T[n, h], Sd))
    return err


def pin_row_permutation(lib) -> float:
    """Rows of S (value channels) never mix: permuting the value channels of
    (v, alpha, S0) permutes the rows of o and S_T the same way."""
    rng = np.random.default_rng(5)
    lengths = [9, 4]
    H, d_k, d_v = 2, 6, 7
    q, k, v, alpha, beta, S0, cu = _random_problem(rng, lengths, H, d_k, d_v)
    o, S_T = oracle.prefill(q, k, v, alpha, beta, S0, cu, lib=lib)
    p = rng.permutation(d_v)
    o2, S2 = oracle.prefill(q, k, _f32(v[..., p]), _f32(alpha[..., p]), beta,
                            S0[:, :, p, :], cu, lib=lib)
    return max(_rel(o2, o[..., p]), _rel(S2, S_T[:, :, p, :]))


def pin_split_resume(lib) -> float:
    """Constant memory: the state carries everything.  Running T1 + T2 tokens
    equals running T2 tokens from the state left after T1."""
    rng = np.random.default_rng(6)
    T1, T2, H, d_k, d_v = 11, 9, 2, 6, 5
    q, k, v, alpha, beta, S0, _ = _random_problem(rng, [T1 + T2], H, d_k, d_v)
    o, S_T = oracle.prefill(q, k, v, alpha, beta, S0, np.array([0, T1 + T2], np.int32), lib=lib)
    o1, S1 = oracle.prefill(q[:T1], k[:T1], v[:T1], alpha[:T1], beta[:T1], S0,
                            np.array([0, T1], np.int32), lib=lib)
    o2, S2 = oracle.prefill(q[T1:], k[T1:], v[T1:], alpha[T1:], beta[T1:], S1,
                            np.array([0, T2], np.int32), lib=lib)
    return max(_rel(np.concatenate([o1, o2]), o), _rel(S2, S_T))


def pin_varlen_independence(lib) -> float:
    """A packed batch equals its sequences run one by one; a zero-length
    sequence returns its initial state unchanged."""
    rng = np.random.default_rng(7)
    lengths = [5, 0, 8, 3, 0]
    H, d_k, d_v = 2, 4, 6
    q, k, v, alpha, beta, S0, cu = _random_problem(rng, lengths, H, d_k, d_v)
    o, S_T = oracle.prefill(q, k, v, alpha, beta, S0, cu, lib=lib)
    err = 0.0
    for n, L in enumerate(lengths):
        a, b = cu[n], cu[n + 1]
        if L == 0:
            err = max(err, _rel(S_T[n], S0[n]))
            continue
        on, Sn = oracle.prefill(q[a:b], k[a:b], v[a:b], alpha[a:b], beta[a:b], S0[n:n + 1],
                                np.array([0, L], np.int32), lib=lib)
        err = max(err, _rel(o[a:b], on), _rel(S_T[n], Sn[0]))
    return err


def pin_additive_is_naive_linear_attention(lib) -> float:
    """The additive update with alpha = beta = 1 and S0 = 0 is the page's naive
    linear attention, o_t = (sum_{i<=t} v_i k_i^T) q_t, for any keys (here
    random, not orthogonal: the delta rule would differ)."""
    rng = np.random.default_rng(8)
    T, H, d_k, d_v = 14, 2, 6, 5
    q = _f32(rng.standard_normal((T, H, d_k)))
    k = _f32(rng.standard_normal((T, H, d_k)))
    v = _f32(rng.standard_normal((T, H, d_v)))
    alpha = np.ones((T, H, d_v), np.float32)
    beta = np.ones((T, H), np.float32)
    o, S_T = oracle.prefill(q, k, v, alpha, beta, None, np.array([0, T], np.int32), lib=lib,
                            additive=True)
    err = 0.0
    for h in range(H):
        M = np.zeros((d_v, d_k))
        for t in range(T):
            M = M + np.outer(v[t, h].astype(np.float64), k[t, h].astype(np.float64))
            err = max(err, _rel(o[t, h], M @ q[t, h].astype(np.float64)))
        err = max(err, _rel(S_T[0, h], M))
    return err


def pin_additive_gated_closed_form(lib) -> float:
    """The gated additive update unrolled: S_t = diag(G_t) S0 +
    sum_{i<=t} diag(G_t / G_i) beta_i v_i k_i^T with G_t = prod_{j<=t} alpha_j."""
    rng = np.random.default_rng(9)
    T, H, d_k, d_v = 11, 2, 4, 6
    q = _f32(rng.standard_normal((T, H, d_k)))
    k = _f32(rng.standard_normal((T, H, d_k)))
    v = _f32(rng.standard_normal((T, H, d_v)))
    alpha = _f32(rng.uniform(0.4, 1.0, (T, H, d_v)))
    beta = _f32(rng.uniform(0.0, 1.0, (T, H)))
    S0 = rng.standard_normal((1, H, d_v, d_k))
    o, S_T = oracle.prefill(q, k, v, alpha, beta, S0, np.array([0, T], np.int32), lib=lib,
                            additive=True)
    err = 0.0
    for h in range(H):
        G = np.cumprod(alpha[:, h].astype(np.float64), axis=0)
        for t in range(T):
            St = G[t][:, None] * S0[0, h]
            for i in range(t + 1):
                St = St + (G[t] / G[i])[:, None] * float(beta[i, h]) * np.outer(
                    v[i, h].astype(np.float64), k[i, h].astype(np.float64))
            err = max(err, _rel(o[t, h], St @ q[t, h].astype(np.float64)))
        err = max(err, _rel(S_T[0, h], St))
    return err


# name -> (function, tolerance).  Tolerances are a few hundred fp64 roundings.
def pin_decode_continuation(lib) -> float:
    """A decode step is the recurrence over sequences of length one: a packed
    prefill of each sequence's first tokens, then n batched decode steps (one
    token of every sequence per step), equals the prefill of all the tokens,
    sequence by sequence; under both update rules."""
    rng = np.random.default_rng(10)
    lens, n, H, d_k, d_v = [5, 8, 3], 4, 2, 6, 5
    B = len(lens)
    q, k, v, alpha, beta, S0, cu_full = _random_problem(rng, [L + n for L in lens], H, d_k, d_v)
    head = np.concatenate([np.arange(cu_full[b], cu_full[b] + lens[b]) for b in range(B)])
    cu = np.zeros(B + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    err = 0.0
    for additive in (False, True):
        o_full, S_full = oracle.prefill(q, k, v, alpha, beta, S0, cu_full, lib=lib,
                                        additive=additive)
        o_p, S = oracle.prefill(q[head], k[head], v[head], alpha[head], beta[head], S0, cu,
                                lib=lib, additive=additive)
        err = max(err, _rel(o_p, o_full[head]))
        for j in range(n):
            tok = np.array([cu_full[b] + lens[b] + j for b in range(B)])
            o_d, S = oracle.decode_step(q[tok], k[tok], v[tok], alpha[tok], beta[tok], S,
                                        additive, lib=lib)
            err = max(err, _rel(o_d, o_full[tok]))
        err = max(err, _rel(S, S_full))
    return err


PINS = {
    "naive_linear_attention": (pin_naive_linear_attention, 1e-12),
    "pure_decay": (pin_pure_decay, 1e-12),
    "delta_write": (pin_delta_write, 1e-12),
    "scalar_geometric": (pin_scalar_geometric, 1e-12),
    "dense_matrix_form": (pin_dense_matrix_form, 1e-11),
    "row_permutation": (pin_row_permutation, 1e-13),
    "split_resume": (pin_split_resume, 1e-13),
    "varlen_independence": (pin_varlen_independence, 1e-13),
    "decode_continuation": (pin_decode_continuation, 1e-13),
    "additive_is_naive_linear_attention": (pin_additive_is_naive_linear_attention, 1e-12),
    "additive_gated_closed_form": (pin_additive_gated_closed_form, 1e-12),
}


def failing_pins(lib) -> list[str]:
    """Names of pins that a given oracle build violates (errors count as failures)."""
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
