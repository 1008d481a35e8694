"""The GPU steps of the cross-process sequence split, on one GPU: each
segment's map from special prefills, kda_segment_combine scanning them, and
the segments' prefills from the scanned states, against the oracle over the
whole sequences (the exchange between processes is tested on CPU ranks)."""
import numpy as np
import pytest
import torch

import oracle
import parity
import seqpar_reference as ref
from gated_delta_rule_45_gb300 import kda, seqpar, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("world,d_k,d_v,mu", [(2, 128, 128, 3.0), (3, 128, 256, 4.0),
                                              (4, 64, 48, 3.0)])
def test_segments_scanned_on_one_gpu(world, d_k, d_v, mu):
    spec = synth.PrefillSpec(num_seqs=3, len_lo=100, len_hi=700, H=2, d_k=d_k, d_v=d_v,
                             alpha_mu=mu, s0_std=0.1, seed=61)
    d = synth.prefill_inputs(spec)
    segs = ref.split_batch(d, world)
    be = seqpar.LibraryBackend()
    maps = []
    for seg in segs:
        g = {k_: seg[k_].cuda() for k_ in ("q", "k", "v", "alpha", "beta", "cu_seqlens")}
        maps.append(seqpar.segment_map(be, g["q"], g["k"], g["v"], g["alpha"], g["beta"],
                                       g["cu_seqlens"]))
    S = d["S0"].cuda()
    o_ref, S_ref = oracle.prefill(synth.bf16_bits(d["q"]), synth.bf16_bits(d["k"]),
                                  synth.bf16_bits(d["v"]), d["alpha"].numpy(), d["beta"].numpy(),
                                  d["S0"].double().numpy(), d["cu_seqlens"].numpy())
    cu = d["cu_seqlens"].numpy()
    for r, seg in enumerate(segs):
        g = {k_: seg[k_].cuda() for k_ in ("q", "k", "v", "alpha", "beta", "cu_seqlens")}
        o, S_end = be.prefill(g["q"], g["k"], g["v"], g["alpha"], g["beta"], S, g["cu_seqlens"])
        torch.cuda.synchronize()
        idx = seg["idx"].numpy()
        o_r = o.float().cpu().numpy()
        scu = seg["cu_seqlens"].numpy()
        for n in range(spec.num_seqs):
            a, b = int(scu[n]), int(scu[n + 1])
            for h in range(spec.H):
                if b > a:
                    assert parity.rel_gate(o_r[a:b, h], o_ref[idx[a:b], h], torch.bfloat16) \
                        <= parity.TOL_BF16, (r, n, h)
        if r + 1 < world:   # the next segment starts from this one's map applied
            S = kda.segment_combine(S, *maps[r])
    torch.cuda.synchronize()
    for n in range(spec.num_seqs):
        for h in range(spec.H):
            assert parity.rel(S_end[n, h].cpu().numpy(), S_ref[n, h]) <= parity.TOL_BF16


def test_segment_combine_against_numpy():
    gen = torch.Generator().manual_seed(3)
    N, H, d_k, d_v = 2, 3, 128, 80
    S = torch.randn(N, H, d_v, d_k, generator=gen)
    g = torch.rand(N, H, d_v, generator=gen)
    P = torch.randn(N, H, d_k, d_k, generator=gen) / 11
    R = torch.randn(N, H, d_v, d_k, generator=gen)
    ref_out = ref.OracleBackend().combine(S, g, P, R).numpy()
    out = kda.segment_combine(S.cuda(), g.cuda(), P.cuda(), R.cuda())
    np.testing.assert_allclose(out.cpu().numpy(), ref_out, rtol=1e-4, atol=1e-4)
    Sc = S.cuda()   # in place
    kda.segment_combine(Sc, g.cuda(), P.cuda(), R.cuda(), Sc)
    np.testing.assert_allclose(Sc.cpu().numpy(), ref_out, rtol=1e-4, atol=1e-4)
