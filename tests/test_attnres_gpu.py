"""attnres_layer against the Attention Residuals oracle (GPU).

Single layers in bf16 and fp32 (with and without the running sum, written
in place and as a finished block), a whole network run layer by layer the
way a model would (stored block sums, an in-place running sum) against the
page's formula, and sampled tokens of the full-size layer.  Gate: relative
Frobenius error <= 2e-3 for bf16 outputs (the bf16 rounding of the exact
output alone costs about 1.1e-3) and <= 1e-5 for fp32.
"""
import numpy as np
import pytest
import torch

import parity
from gated_delta_rule_45_gb300 import kda, synth
from oracle import attnres as ar

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 2e-3, torch.float32: 1e-5}


def _np(x):
    return x.double().cpu().numpy()


def _layer_case(T, d, nb, with_partial, with_last, dtype, seed, inplace=False, block_out=False):
    g = torch.Generator(device="cpu").manual_seed(seed)
    blocks = torch.randn(nb, T, d, generator=g).to(dtype)
    partial = torch.randn(T, d, generator=g) * 2 if with_partial else None
    h_last = torch.randn(T, d, generator=g).to(dtype) if with_last else None
    q = torch.randn(d, generator=g)
    scale = 1.0 / np.sqrt(d)
    dev = lambda x: None if x is None else x.cuda()
    bd, pd, hd, qd = dev(blocks), dev(partial), dev(h_last), dev(q)
    has_p = with_partial or with_last
    pout = None
    if has_p:
        pout = pd if (inplace and pd is not None) else torch.empty(T, d, device="cuda")
    bout = torch.empty(T, d, dtype=dtype, device="cuda") if (block_out and has_p) else None
    h = kda.attnres_layer(bd, qd, partial=pd, h_last=hd, partial_out=pout, block_out=bout,
                          scale=scale)
    torch.cuda.synchronize()
    h_ref, P_ref = ar.layer_step(_np(blocks), None if partial is None else _np(partial),
                                 None if h_last is None else _np(h_last), _np(q), scale)
    assert parity.rel(_np(h), h_ref) <= TOL[dtype]
    if has_p:
        assert parity.rel(_np(pout), P_ref) <= 1e-6
    if bout is not None:
        assert parity.rel(_np(bout), P_ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("case", [
    dict(T=300, d=256, nb=1, with_partial=False, with_last=False),    # one source
    dict(T=257, d=512, nb=5, with_partial=False, with_last=False),    # a block's first layer, n > 1
    dict(T=130, d=2048, nb=4, with_partial=False, with_last=True),    # a block's second layer
    dict(T=99, d=1024, nb=3, with_partial=True, with_last=True),      # later layers
    dict(T=64, d=4096, nb=2, with_partial=True, with_last=True),      # several pieces per thread
    dict(T=40, d=64, nb=63, with_partial=True, with_last=False),      # 64 sources, narrow rows
    dict(T=48, d=8192, nb=2, with_partial=True, with_last=True),      # wide rows, four pieces per thread
])
def test_attnres_layer_matches_oracle(case, dtype):
    _layer_case(**case, dtype=dtype, seed=hash(tuple(case.values())) % 1000)


def test_attnres_running_sum_in_place_and_block_out():
    _layer_case(T=200, d=768, nb=2, with_partial=True, with_last=True, dtype=torch.bfloat16,
                seed=7, inplace=True, block_out=True)
    _layer_case(T=200, d=768, nb=2, with_partial=False, with_last=True, dtype=torch.float32,
                seed=8, block_out=True)


def test_attnres_network_matches_formula():
    """Twelve layers in blocks of 3, 4 and 5, run as a model would: block sums
    stored as they complete, the current block's running sum updated in place.
    fp32 storage, so the stored block sums are exact up to fp32."""
    spec = synth.AttnResSpec(T=96, d=256, block_sizes=(3, 4, 5), dtype="fp32", seed=3)
    x = synth.attnres_inputs(spec)
    L = sum(spec.block_sizes)
    scale = 1.0 / np.sqrt(spec.d)
    outs_np = _np(x["outs"])
    ins_ref, _ = ar.blocked_network(_np(x["h0"]), lambda i, h: outs_np[i - 1],
                                    _np(x["queries"]), list(spec.block_sizes), scale)
    nblk = len(spec.block_sizes)
    blocks = torch.empty(nblk + 1, spec.T, spec.d, device="cuda")
    blocks[0] = x["h0"].cuda()
    running = torch.empty(spec.T, spec.d, device="cuda")
    outs = x["outs"].cuda()
    qs = x["queries"].cuda()
    layer, worst = 0, 0.0
    for n, size in enumerate(spec.block_sizes, start=1):
        for i in range(size):
            if i == 0 and n == 1:
                h = kda.attnres_layer(blocks[:1], qs[layer], scale=scale)
            elif i == 0:   # previous block finishes: its sum is the last source and is stored
                h = kda.attnres_layer(blocks[:n - 1], qs[layer], partial=running,
                                      h_last=outs[layer - 1], block_out=blocks[n - 1],
                                      scale=scale)
            elif i == 1:
                h = kda.attnres_layer(blocks[:n], qs[layer], h_last=outs[layer - 1],
                                      partial_out=running, scale=scale)
            else:
                h = kda.attnres_layer(blocks[:n], qs[layer], partial=running,
                                      h_last=outs[layer - 1], partial_out=running, scale=scale)
            torch.cuda.synchronize()
            worst = max(worst, parity.rel(_np(h), ins_ref[layer]))
            layer += 1
    assert worst <= 1e-5, worst


def test_attnres_full_size_layer_sampled():
    """A full-size layer of the bench network (16384 tokens, width 2048, the
    eighth block's later layers: 7 stored blocks + the running sum), the
    oracle on 64 sampled tokens."""
    spec = synth.ATTNRES
    g = torch.Generator(device="cuda").manual_seed(9)
    T, d = spec.T, spec.d
    blocks = torch.randn(8, T, d, device="cuda", generator=g).to(torch.bfloat16)
    partial = torch.randn(T, d, device="cuda", generator=g) * 2
    h_last = torch.randn(T, d, device="cuda", generator=g).to(torch.bfloat16)
    q = torch.randn(d, device="cuda", generator=g)
    h = kda.attnres_layer(blocks, q, partial=partial, h_last=h_last)
    torch.cuda.synchronize()
    idx = torch.randperm(T, generator=torch.Generator().manual_seed(1))[:64]
    h_ref, _ = ar.layer_step(_np(blocks[:, idx]), _np(partial[idx]), _np(h_last[idx]), _np(q),
                             1.0 / np.sqrt(d))
    assert parity.rel(_np(h[idx]), h_ref) <= 2e-3
