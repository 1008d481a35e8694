"""The chunkwise form the kernels implement, in fp64, against the oracle (CPU only).

This checks the derivation (row-independent decay, 1/gamma rescaling, WY/UT
triangular solve, inclusive intra-chunk mask, padding of partial chunks and
varlen resets) before any CUDA is involved.
"""
import numpy as np
import pytest
import torch

import chunk_form
import oracle
from gated_delta_rule_45_gb300 import synth


def _np_inputs(d):
    f = lambda x: synth.bf16_bits(x)
    S0 = None if d["S0"] is None else d["S0"].double().numpy()
    return (f(d["q"]), f(d["k"]), f(d["v"]), d["alpha"].numpy(), d["beta"].numpy(), S0,
            d["cu_seqlens"].numpy())


def _widen(x):
    return oracle.bf16_bits_to_f64(x) if x.dtype == np.uint16 else x.astype(np.float64)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.mark.parametrize("C", [16, 32, 64])
def test_chunk_form_matches_recurrence_varlen(oracle_lib, C):
    spec = synth.PrefillSpec(num_seqs=5, len_lo=1, len_hi=150, H=2, d_k=32, d_v=48,
                             alpha_mu=2.0, s0_std=0.3, seed=3)
    q, k, v, a, b, S0, cu = _np_inputs(synth.prefill_inputs(spec))
    o_ref, S_ref = oracle.prefill(q, k, v, a, b, S0, cu, lib=oracle_lib)
    o, S = chunk_form.run_packed(_widen(q), _widen(k), _widen(v), a, b, S0, cu, C)
    assert _rel(o, o_ref) < 1e-11
    assert _rel(S, S_ref) < 1e-11


def test_chunk_form_tiny_workload(oracle_lib):
    d = synth.prefill_inputs(synth.TINY)
    q, k, v, a, b, S0, cu = _np_inputs(d)
    o_ref, S_ref = oracle.prefill(q, k, v, a, b, S0, cu, lib=oracle_lib)
    o, S = chunk_form.run_packed(_widen(q), _widen(k), _widen(v), a, b, S0, cu, 16)
    assert _rel(o, o_ref) < 1e-12 and _rel(S, S_ref) < 1e-12


def test_chunk_form_zero_length_and_exact_multiple(oracle_lib):
    rng = np.random.default_rng(0)
    lengths = [0, 64, 128, 0, 65]
    H, d_k, d_v = 1, 16, 16
    T = sum(lengths)
    q = rng.standard_normal((T, H, d_k)).astype(np.float32)
    k = rng.standard_normal((T, H, d_k)).astype(np.float32)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, d_v)).astype(np.float32)
    a = rng.uniform(0.6, 1.0, (T, H, d_v)).astype(np.float32)
    b = rng.uniform(0, 1, (T, H)).astype(np.float32)
    S0 = rng.standard_normal((len(lengths), H, d_v, d_k))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    o_ref, S_ref = oracle.prefill(q, k, v, a, b, S0, cu, lib=oracle_lib)
    o, S = chunk_form.run_packed(q.astype(np.float64), k.astype(np.float64),
                                 v.astype(np.float64), a, b, S0, cu, 64)
    assert _rel(o, o_ref) < 1e-11 and _rel(S, S_ref) < 1e-11
    assert np.array_equal(S[0], S0[0]) and np.array_equal(S[3], S0[3])


def test_synth_is_deterministic():
    a = synth.prefill_inputs(synth.PrefillSpec(num_seqs=3, len_lo=2, len_hi=9, H=2, d_k=8, d_v=8))
    b = synth.prefill_inputs(synth.PrefillSpec(num_seqs=3, len_lo=2, len_hi=9, H=2, d_k=8, d_v=8))
    for key in ("q", "k", "v", "alpha", "beta", "cu_seqlens"):
        assert torch.equal(a[key], b[key])
    assert a["q"].dtype == torch.bfloat16 and a["alpha"].dtype == torch.float32
    norms = a["k"].float().norm(dim=-1)
    assert torch.allclose(norms, torch.ones_like(norms), atol=1e-2)
    assert float(a["alpha"].min()) > 0 and float(a["alpha"].max()) < 1


@pytest.mark.parametrize("C", [16, 64])
def test_chunk_backward_matches_reverse_mode(oracle_lib, C):
    """The chunkwise reverse mode the CUDA backward implements against the
    oracle's token-by-token reverse mode, on a varlen batch with an empty
    sequence, ragged tails and nonzero S0 and dS_T."""
    spec = synth.PrefillSpec(num_seqs=4, len_lo=1, len_hi=150, H=2, d_k=32, d_v=48,
                             alpha_mu=2.0, s0_std=0.3, seed=5)
    q, k, v, a, b, S0, cu = _np_inputs(synth.prefill_inputs(spec))
    cu = np.concatenate([cu[:2], cu[1:2], cu[2:]]).astype(np.int32)   # an empty sequence
    S0 = np.concatenate([S0[:1], S0[:1] * 0.5, S0[1:]])
    rng = np.random.default_rng(6)
    dO = rng.standard_normal(v.shape)
    dS_T = rng.standard_normal(S0.shape)
    ref = oracle.backward(q, k, v, a, b, S0, cu, dO, dS_T, lib=oracle_lib)
    got = chunk_form.backward_packed(_widen(q), _widen(k), _widen(v), a, b, S0, cu, dO, dS_T, C)
    for name in ref:
        assert _rel(got[name], ref[name]) < 1e-10, name


@pytest.mark.parametrize("C", [16, 64])
def test_chunk_form_of_the_additive_update(oracle_lib, C):
    """The additive update's chunk form (T = I, no K S^T term in X), which both
    chunk kernels implement, against the oracle's additive recurrence."""
    spec = synth.PrefillSpec(num_seqs=4, len_lo=1, len_hi=150, H=2, d_k=32, d_v=48,
                             alpha_mu=2.0, s0_std=0.3, seed=8)
    q, k, v, a, b, S0, cu = _np_inputs(synth.prefill_inputs(spec))
    o_ref, S_ref = oracle.prefill(q, k, v, a, b, S0, cu, lib=oracle_lib, additive=True)
    o, S = chunk_form.run_packed(_widen(q), _widen(k), _widen(v), a, b, S0, cu, C,
                                 additive=True)
    assert _rel(o, o_ref) < 1e-11
    assert _rel(S, S_ref) < 1e-11
