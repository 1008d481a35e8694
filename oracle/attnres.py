"""Attention Residuals, plain and blocked: fp64 numpy reference.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU arms may import it.

What it computes ("Kimi (AI)", section "Attention Residuals").  Layer i has
input h_i and output h'_i; h'_0 is the network's input.  Plain Attention
Residuals feed layer i with

    h_i = SoftmaxAttention(q_i, K_i, V_i),   K_i = V_i = [h'_0, ..., h'_{i-1}],

q_i a learned vector per layer.  The blocked variant cuts the layers into
consecutive blocks (n_1, n_2, ... layers); layer i of block n attends over
the sums of the outputs of every earlier block and, from its second layer
on, the sum of the earlier outputs of its own block.

Readings (the pages leave these open):
* The first layer of the first block would attend over an empty list; the
  network input h'_0 is read as block 0, a block of one output, so its
  summary h'_0 leads every list (the other page describes the first block's
  layers as fed from "input0").
* SoftmaxAttention is standard scaled dot-product attention, per token
  (attention runs over depth, not over positions): weights
  softmax_j(scale * q . k_j), scale = 1 / sqrt(d) unless given.
"""
from __future__ import annotations

import numpy as np


def softmax_attention(q, sources, scale):
    """Per token: sum_j softmax_j(scale * q . s_j[t]) s_j[t].

    q: [d]; sources: [m, T, d] (K = V = sources).  Returns [T, d] (fp64).
    """
    q = np.asarray(q, dtype=np.float64)
    S = np.asarray(sources, dtype=np.float64)
    logits = scale * np.einsum("mtd,d->tm", S, q)            # [T, m]
    logits = logits - logits.max(axis=1, keepdims=True)
    w = np.exp(logits)
    w = w / w.sum(axis=1, keepdims=True)
    return np.einsum("tm,mtd->td", w, S)


def default_scale(d: int) -> float:
    return 1.0 / np.sqrt(d)


def plain_network(h0, layer_fn, queries, scale):
    """Run L layers with plain Attention Residuals.

    h0: [T, d] (= h'_0); layer_fn(i, h) -> h'_i for layer i = 1..L; queries[i-1]
    is q_i.  Returns (inputs [h_1..h_L], outputs [h'_0..h'_L])."""
    outs = [np.asarray(h0, dtype=np.float64)]
    ins = []
    for i, q in enumerate(queries, start=1):
        h = softmax_attention(q, np.stack(outs), scale)
        ins.append(h)
        outs.append(np.asarray(layer_fn(i, h), dtype=np.float64))
    return ins, outs


def blocked_network(h0, layer_fn, queries, block_sizes, scale):
    """Run sum(block_sizes) layers with Blocked Attention Residuals, straight
    from the page's formula: the source list of layer (n, i) is rebuilt from
    all outputs so far.  Returns (inputs, outputs) like ``plain_network``."""
    outs = [np.asarray(h0, dtype=np.float64)]
    blocks = [[0]]          # output indices of each block; block 0 = {h'_0}
    ins = []
    layer = 0
    for n_size in block_sizes:
        cur = []
        for i in range(n_size):
            summaries = [sum(outs[j] for j in blk) for blk in blocks]
            if i >= 1:
                summaries.append(sum(outs[j] for j in cur))
            h = softmax_attention(queries[layer], np.stack(summaries), scale)
            ins.append(h)
            layer += 1
            outs.append(np.asarray(layer_fn(layer, h), dtype=np.float64))
            cur.append(len(outs) - 1)
        blocks.append(cur)
    return ins, outs


def layer_step(blocks, partial, h_last, q, scale):
    """One layer of the blocked scheme as it runs in a network, with the block
    summaries stored and the current block's partial sum carried.

    blocks: [nb, T, d] summaries of the finished blocks (block 0 first);
    partial: [T, d] sum of the current block's outputs before the previous
    layer, or None; h_last: [T, d] output of the previous layer when it belongs
    to the current block, or None (first layer of a block).  The running sum
    P = partial + h_last (whichever are given) joins the sources last.
    Returns (h [T, d], P or None)."""
    srcs = [np.asarray(b, dtype=np.float64) for b in blocks]
    P = None
    if partial is not None or h_last is not None:
        P = 0.0
        if partial is not None:
            P = P + np.asarray(partial, dtype=np.float64)
        if h_last is not None:
            P = P + np.asarray(h_last, dtype=np.float64)
        srcs.append(P)
    return softmax_attention(q, np.stack(srcs), scale), P
