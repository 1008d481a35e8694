"""Pins for the Attention Residuals oracle (``oracle/attnres.py``).

Source: "Kimi (AI)" (Wikipedia mirror), section "Attention Residuals": the
plain form h_i = SoftmaxAttention(q_i, K_i, V_i) with K_i = V_i = the
earlier outputs, and the blocked form whose sources are block sums.

Each pin takes the oracle module (so that planted mistakes in a copy can be
checked) and returns the largest relative deviation from something computed
without the function under test: PyTorch's scaled dot-product attention, a
closed form, an invariance, or the page's formula run a second way.
"""
from __future__ import annotations

import numpy as np
import torch


def _rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def pin_library_attention(ar) -> float:
    """softmax_attention against torch's scaled_dot_product_attention: one
    query per token (the layer's q), the m sources of that token as keys and
    values."""
    rng = np.random.default_rng(41)
    m, T, d = 5, 37, 24
    S = rng.standard_normal((m, T, d))
    q = rng.standard_normal(d)
    scale = 0.37
    got = ar.softmax_attention(q, S, scale)
    qt = torch.from_numpy(np.broadcast_to(q, (T, 1, d)).copy())
    kv = torch.from_numpy(np.ascontiguousarray(S.transpose(1, 0, 2)))   # [T, m, d]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kv, kv, scale=scale)[:, 0]
    return _rel(got, ref.numpy())


def pin_zero_query_is_mean(ar) -> float:
    """q = 0: all logits equal, the output is the mean of the sources."""
    rng = np.random.default_rng(42)
    S = rng.standard_normal((6, 11, 8))
    return _rel(ar.softmax_attention(np.zeros(8), S, 1.0), S.mean(axis=0))


def pin_one_source_is_identity(ar) -> float:
    """A single source gets weight 1."""
    rng = np.random.default_rng(43)
    S = rng.standard_normal((1, 9, 16))
    return _rel(ar.softmax_attention(rng.standard_normal(16), S, 0.25), S[0])


def pin_two_sources_closed_form(ar) -> float:
    """Two sources: weight sigmoid(scale q.(s0 - s1)) on s0."""
    rng = np.random.default_rng(44)
    S = rng.standard_normal((2, 13, 10))
    q = rng.standard_normal(10)
    scale = 0.7
    w0 = 1.0 / (1.0 + np.exp(-scale * (S[0] - S[1]) @ q))
    expect = w0[:, None] * S[0] + (1 - w0)[:, None] * S[1]
    return _rel(ar.softmax_attention(q, S, scale), expect)


def pin_source_order(ar) -> float:
    """The sources form a set: permuting them leaves the output unchanged."""
    rng = np.random.default_rng(45)
    S = rng.standard_normal((7, 10, 12))
    q = rng.standard_normal(12)
    perm = rng.permutation(7)
    return _rel(ar.softmax_attention(q, S[perm], 0.3), ar.softmax_attention(q, S, 0.3))


def _layer_fn(d, seed):
    """A fixed nonlinear layer per index (a stand-in for the network's layers)."""
    rng = np.random.default_rng(seed)
    W = [rng.standard_normal((d, d)) / np.sqrt(d) for _ in range(64)]
    return lambda i, h: np.tanh(h @ W[i % 64]) + 0.1 * h


def pin_unit_blocks_are_plain(ar) -> float:
    """Blocks of one layer each: every block sum is one output, so the blocked
    network is the plain one."""
    rng = np.random.default_rng(46)
    T, d, L = 7, 16, 6
    h0 = rng.standard_normal((T, d))
    qs = rng.standard_normal((L, d))
    f = _layer_fn(d, 1)
    _, o_plain = ar.plain_network(h0, f, qs, 0.25)
    _, o_block = ar.blocked_network(h0, f, qs, [1] * L, 0.25)
    return max(_rel(a, b) for a, b in zip(o_block, o_plain))


def pin_incremental_matches_formula(ar) -> float:
    """The layer-by-layer bookkeeping (stored block sums, a running partial sum
    of the current block, the previous output added on the fly) against the
    page's formula rebuilt from all outputs, over uneven blocks."""
    rng = np.random.default_rng(47)
    T, d = 9, 12
    sizes = [3, 1, 4, 2]
    L = sum(sizes)
    h0 = rng.standard_normal((T, d))
    qs = rng.standard_normal((L, d))
    f = _layer_fn(d, 2)
    ins_ref, _ = ar.blocked_network(h0, f, qs, sizes, 0.3)
    blocks = [h0]
    err, layer = 0.0, 0
    partial = h_last = None
    for n_size in sizes:
        for i in range(n_size):
            h, P = ar.layer_step(np.stack(blocks), partial, h_last, qs[layer], 0.3)
            if i == 0 and P is not None:      # P is the previous block's sum
                blocks.append(P)
                P = None
            err = max(err, _rel(h, ins_ref[layer]))
            layer += 1
            partial, h_last = P, f(layer, h)
    return err


def _constant_layer_inputs(h0, c, qs, sizes, scale):
    """Closed form of every layer's input in a blocked network whose layers all
    output the same array c (whatever their input).  A finished block of n
    layers then sums to n c, and a block's partial sum after i layers is i c,
    so layer (block, i) attends over h0 and multiples m_j c of c:

        h = (w_0 h0 + (sum_j w_j m_j) c),   w = softmax(scale q.h0, scale m_j q.c)

    with multipliers m_j = the finished blocks' sizes, then i when i >= 1.
    Returns the inputs and, per layer, the multiplier of the running sum the
    layer forms (i at i >= 1; at a block's first layer, the size of the block
    just finished; None for the first block's first layer)."""
    ins, run_mult = [], []
    finished, layer, prev = [], 0, None
    for n_size in sizes:
        for i in range(n_size):
            q = qs[layer]
            mults = list(finished) + ([i] if i >= 1 else [])
            a0 = scale * (h0 @ q)                        # [T]
            ac = scale * (c @ q)                         # [T]
            logits = np.stack([a0] + [m * ac for m in mults], axis=1)
            logits = logits - logits.max(axis=1, keepdims=True)
            w = np.exp(logits)
            w = w / w.sum(axis=1, keepdims=True)
            cm = sum(w[:, 1 + j] * m for j, m in enumerate(mults)) if mults else 0.0
            ins.append(w[:, :1] * h0 + np.asarray(cm)[..., None] * c)
            run_mult.append(i if i >= 1 else prev)
            layer += 1
        finished.append(n_size)
        prev = n_size
    return ins, run_mult


def _constant_case():
    rng = np.random.default_rng(48)
    T, d = 8, 10
    sizes = [3, 1, 4, 2]
    h0 = rng.standard_normal((T, d))
    c = rng.standard_normal((T, d))
    qs = rng.standard_normal((sum(sizes), d))
    return h0, c, qs, sizes, 0.4


def pin_constant_layers_blocked(ar) -> float:
    """The blocked network's inputs against the closed form for layers that
    all output the same array (block sums are integer multiples of it)."""
    h0, c, qs, sizes, scale = _constant_case()
    expect, _ = _constant_layer_inputs(h0, c, qs, sizes, scale)
    got, _ = ar.blocked_network(h0, lambda i, h: c, qs, sizes, scale)
    return max(_rel(a, b) for a, b in zip(got, expect))


def pin_constant_layers_step(ar) -> float:
    """layer_step driven as a model drives it (stored block sums, the running
    sum carried between layers) on the same network: each input and each
    running sum it returns against the closed form."""
    h0, c, qs, sizes, scale = _constant_case()
    expect, mult = _constant_layer_inputs(h0, c, qs, sizes, scale)
    blocks, partial, h_last = [h0], None, None
    err, layer = 0.0, 0
    for n_size in sizes:
        for i in range(n_size):
            h, P = ar.layer_step(np.stack(blocks), partial, h_last, qs[layer], scale)
            err = max(err, _rel(h, expect[layer]))
            if mult[layer] is None:
                err = max(err, 0.0 if P is None else 1.0)
            else:
                err = max(err, _rel(P, mult[layer] * c))
            if i == 0 and P is not None:      # P is the previous block's sum
                blocks.append(P)
                P = None
            layer += 1
            partial, h_last = P, c
    return err


PINS = {
    "library_attention": (pin_library_attention, 1e-12),
    "zero_query_is_mean": (pin_zero_query_is_mean, 1e-14),
    "one_source_is_identity": (pin_one_source_is_identity, 1e-15),
    "two_sources_closed_form": (pin_two_sources_closed_form, 1e-13),
    "source_order": (pin_source_order, 1e-14),
    "unit_blocks_are_plain": (pin_unit_blocks_are_plain, 1e-13),
    "incremental_matches_formula": (pin_incremental_matches_formula, 1e-13),
    "constant_layers_blocked": (pin_constant_layers_blocked, 1e-13),
    "constant_layers_step": (pin_constant_layers_step, 1e-13),
}


def failing_pins(ar) -> list[str]:
    bad = []
    for name, (fn, tol) in PINS.items():
        try:
            err = fn(ar)
        except Exception:
            bad.append(name)
            continue
        if not np.isfinite(err) or err > tol:
            bad.append(name)
    return bad
