"""The GPU workloads at full size, in the launch configuration the bench
times (kernel choice "auto"), checked against the oracle on sampled
(sequence, head) pairs, each over its whole sequence."""
import numpy as np
import pytest
import torch

import oracle
import parity
from gated_delta_rule_45_gb300 import kda, synth

pytestmark = pytest.mark.gpu


def _sample_pairs(num_seqs, H, count, seed):
    rng = np.random.default_rng(seed)
    all_pairs = [(n, h) for n in range(num_seqs) for h in range(H)]
    idx = rng.choice(len(all_pairs), size=min(count, len(all_pairs)), replace=False)
    return sorted(all_pairs[i] for i in idx)


def test_prefill_workload_full():
    """B = 8, H = 32, T = 4096, d = 128, chunk 64, bf16, S0 = 0."""
    spec = synth.PREFILL
    d = synth.prefill_inputs(spec)
    dev = parity.to_device(d)
    o, S_T = kda.prefill(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], None,
                         dev["cu_seqlens"], chunk=spec.chunk, check_device_status=True)
    # 64 of the 256 (sequence, head) pairs, each over its whole sequence, plus
    # every head of the first sequence and every sequence of the last head
    pairs = _sample_pairs(spec.num_seqs, spec.H, 64, 0) \
        + [(0, h) for h in range(spec.H)] + [(n, spec.H - 1) for n in range(spec.num_seqs)]
    pairs = sorted(set(pairs))
    assert len(pairs) >= 64
    ref = parity.oracle_pairs(d, pairs)
    wo, ws = parity.compare_pairs(d, o, S_T, ref)
    assert wo <= parity.TOL_BF16 and ws <= parity.TOL_BF16, (wo, ws)
    assert torch.isfinite(o.float()).all() and torch.isfinite(S_T).all()


def test_long_context_workload_full():
    """B = 1, H = 32, T = 131072, d = 128, chunk 64, S0 ~ N(0, 0.1^2), alpha = sigmoid(N(5, 1))."""
    spec = synth.LONG
    d = synth.prefill_inputs(spec)
    dev = parity.to_device(d)
    o, S_T = kda.prefill(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], dev["S0"],
                         dev["cu_seqlens"], chunk=spec.chunk, check_device_status=True)
    # every one of the 32 chains, each over all 131072 tokens
    pairs = [(0, h) for h in range(spec.H)]
    ref = parity.oracle_pairs(d, pairs)
    wo, ws = parity.compare_pairs(d, o, S_T, ref)
    assert wo <= parity.TOL_BF16 and ws <= parity.TOL_BF16, (wo, ws)
    assert torch.isfinite(o.float()).all() and torch.isfinite(S_T).all()


def test_varlen_workload_with_decode_continuation():
    """64 sequences, lengths U[128, 8192], H = 16, d_k = 128, d_v = 256, S0 ~ N(0, 0.1^2);
    then 32 decode steps per sequence from the returned states.  The decode
    continuation is checked against the oracle run over prefill + decode tokens."""
    spec = synth.VARLEN
    d = synth.prefill_inputs(spec)
    steps = synth.decode_sequence_inputs(synth.VARLEN_DECODE_STEPS, spec.num_seqs, spec.H,
                                         spec.d_k, spec.d_v, spec.dtype, spec.alpha_mu,
                                         d["generator"])
    dev = parity.to_device(d)
    o, S_T = kda.prefill(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], dev["S0"],
                         dev["cu_seqlens"], chunk=spec.chunk, check_device_status=True)
    S = S_T.clone()
    outs = []
    for st in steps:
        sd = {k_: st[k_].cuda() for k_ in ("q", "k", "v", "alpha", "beta")}
        outs.append(kda.decode_step(sd["q"], sd["k"], sd["v"], sd["alpha"], sd["beta"], S))
    torch.cuda.synchronize()

    lengths = d["lengths"]
    longest = int(np.argmax(lengths))
    shortest = int(np.argmin(lengths))
    # 32 sampled pairs plus the longest and the shortest sequence under every head
    pairs = sorted(set(_sample_pairs(spec.num_seqs, spec.H, 32, 1)
                       + [(longest, h) for h in range(spec.H)]
                       + [(shortest, h) for h in range(spec.H)]))
    assert len(pairs) >= 64
    ref = parity.oracle_pairs(d, pairs)
    wo, ws = parity.compare_pairs(d, o, S_T, ref)
    assert wo <= parity.TOL_BF16 and ws <= parity.TOL_BF16, (wo, ws)

    # oracle over the same pairs: continue from its own prefill state through the
    # decode tokens; a slice is one (sequence, head) over its 32 decode tokens
    worst_o = worst_s = 0.0
    S_gpu = S.cpu().numpy()
    for (n, h) in pairs:
        s_ref = ref[(n, h)][1]
        o_refs, o_gpus = [], []
        for i, st in enumerate(steps):
            q = parity._np(st["q"][n:n + 1, h:h + 1])
            k = parity._np(st["k"][n:n + 1, h:h + 1])
            v = parity._np(st["v"][n:n + 1, h:h + 1])
            o_r, S_r = oracle.decode_step(q, k, v, st["alpha"][n:n + 1, h:h + 1].numpy(),
                                          st["beta"][n:n + 1, h:h + 1].numpy(),
                                          s_ref[None, None])
            s_ref = S_r[0, 0]
            o_refs.append(o_r[0, 0])
            o_gpus.append(outs[i][n, h].float().cpu().numpy())
        worst_o = max(worst_o, parity.rel_gate(np.stack(o_gpus), np.stack(o_refs), torch.bfloat16))
        worst_s = max(worst_s, parity.rel(S_gpu[n, h], s_ref))
    assert worst_o <= parity.TOL_BF16 and worst_s <= parity.TOL_BF16, (worst_o, worst_s)


def test_l2_resident_contraction_case():
    """The bench's L2-resident case (152 chains of 384 tokens, H = 1): every chain
    against the oracle."""
    spec = synth.L2_RESIDENT
    d = synth.prefill_inputs(spec)
    dev = parity.to_device(d)
    o, S_T = kda.prefill(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], dev["S0"],
                         dev["cu_seqlens"], chunk=spec.chunk, check_device_status=True)
    ref = parity.oracle_pairs(d, [(n, 0) for n in range(spec.num_seqs)])
    wo, ws = parity.compare_pairs(d, o, S_T, ref)
    assert wo <= parity.TOL_BF16 and ws <= parity.TOL_BF16, (wo, ws)


@pytest.mark.gpu
def test_cuda_path_matches_the_fixture():
    """The stored small case (two sequences of 3 and 6 tokens, d = 16, fp32,
    chunk 16) against its outputs, written by the oracle alone."""
    from test_golden import load_fixture

    _, x, y = load_fixture()
    dev = lambda a, dt=torch.float32: torch.from_numpy(a).to(dt).cuda()
    o, S_T = kda.prefill(dev(x["q"]), dev(x["k"]), dev(x["v"]), dev(x["alpha"]),
                         dev(x["beta"]), dev(x["S0"]), dev(x["cu_seqlens"], torch.int32),
                         chunk=16, check_device_status=True)
    torch.cuda.synchronize()
    o, S_T = o.double().cpu().numpy(), S_T.double().cpu().numpy()
    cu = x["cu_seqlens"]
    for n in range(len(cu) - 1):
        assert parity.rel(o[cu[n]:cu[n + 1]], y["o"][cu[n]:cu[n + 1]]) <= parity.TOL_FP32
        assert parity.rel(S_T[n], y["S_T"][n]) <= parity.TOL_FP32
