"""Helpers shared by the GPU parity tests: run the oracle on chosen
(sequence, head) pairs of a synthetic problem and compare slices.

Error metric: rel_F(x) = ||x - x_ref||_F / ||x_ref||_F per (sequence, head)
slice, separately for o and for the final state; the gate is the maximum over
slices.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from gated_delta_rule_45_gb300 import synth

# Gate on bf16 storage: max over (sequence, head) slices of the relative
# Frobenius error, for o and for the final state.
TOL_BF16 = 2e-3
# fp32 storage: no output rounding to bf16; the fp32 chunk arithmetic alone
# stays near 1e-6, so a tighter gate.
TOL_FP32 = 2e-5


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    if den == 0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / den)


def _np(x: torch.Tensor):
    return synth.bf16_bits(x.cpu()) if x.dtype == torch.bfloat16 else x.cpu().contiguous().numpy()


def oracle_pairs(d: dict, pairs, S0=None, nthreads: int = 0):
    """Run the oracle on the listed (n, h) pairs of a prefill problem `d`.

    The pairs are gathered into one packed batch with H = 1 (each pair becomes
    its own sequence), so the oracle sees exactly the same values.  S0 (float64
    [N, H, d_v, d_k]) defaults to d["S0"].  Returns {(n, h): (o [L, d_v], S_T [d_v, d_k])}.
    """
    cu = d["cu_seqlens"].numpy()
    if S0 is None and d.get("S0") is not None:
        S0 = d["S0"].double().numpy()
    qs, ks, vs, als, bes, s0s, lens = [], [], [], [], [], [], []
    for n, h in pairs:
        a, b = int(cu[n]), int(cu[n + 1])
        qs.append(d["q"][a:b, h:h + 1])
        ks.append(d["k"][a:b, h:h + 1])
        vs.append(d["v"][a:b, h:h + 1])
        als.append(d["alpha"][a:b, h:h + 1])
        bes.append(d["beta"][a:b, h:h + 1])
        lens.append(b - a)
        if S0 is not None:
            s0s.append(np.asarray(S0[n, h], dtype=np.float64))
    q = _np(torch.cat(qs))
    k = _np(torch.cat(ks))
    v = _np(torch.cat(vs))
    al = torch.cat(als).numpy()
    be = torch.cat(bes).numpy()
    pcu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    s0 = np.stack(s0s)[:, None] if S0 is not None else None
    o, S_T = oracle.prefill(q, k, v, al, be, s0, pcu, nthreads=nthreads)
    out = {}
    for i, (n, h) in enumerate(pairs):
        out[(n, h)] = (o[pcu[i]:pcu[i + 1], 0], S_T[i, 0])
    return out


# A slice shorter than this is gated against the oracle value rounded to the
# storage dtype: with few values, rounding even the exact result to bf16 can
# exceed 2e-3 by itself (measured: max 2.2e-3 over 8192 single-token slices of
# 128 values).  Longer slices are gated against the exact fp64 value.
SHORT_SLICE = 4096


def round_to(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Round float64 values to `dtype` (nearest-even) and widen back."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).double().numpy()


def rel_gate(o_gpu: np.ndarray, o_ref: np.ndarray, store_dtype: torch.dtype) -> float:
    """The error a slice of o is gated on (see SHORT_SLICE)."""
    if store_dtype == torch.bfloat16 and o_ref.size < SHORT_SLICE:
        return rel(o_gpu, round_to(o_ref, torch.bfloat16))
    return rel(o_gpu, o_ref)


def compare_pairs(d: dict, o_gpu: torch.Tensor, S_gpu: torch.Tensor, ref: dict):
    """Max over the given pairs of the gated error for o and of rel_F for S_T."""
    cu = d["cu_seqlens"].numpy()
    o_cpu = o_gpu.float().cpu()
    S_cpu = S_gpu.cpu()
    worst_o = worst_s = 0.0
    for (n, h), (o_ref, s_ref) in ref.items():
        a, b = int(cu[n]), int(cu[n + 1])
        if b > a:
            worst_o = max(worst_o, rel_gate(o_cpu[a:b, h].numpy(), o_ref, o_gpu.dtype))
        worst_s = max(worst_s, rel(S_cpu[n, h].numpy(), s_ref))
    return worst_o, worst_s


def to_device(d: dict, device="cuda") -> dict:
    out = {}
    for key in ("q", "k", "v", "alpha", "beta", "S0", "cu_seqlens", "S"):
        if d.get(key) is not None:
            out[key] = d[key].to(device)
        else:
            out[key] = None
    return out
