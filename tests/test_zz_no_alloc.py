"""kda_prefill_noalloc, the entry point for callers that cannot allocate
device memory (its scratch is built into the library), against kda_prefill
with a caller-provided workspace.

Both calls run the same kernels on the same inputs, so their outputs must be
identical bit for bit; one batch is also checked against the oracle.  Two
calls in a row on different batches: the second must not be disturbed by
what the first left in the shared scratch.  A call whose cu_seqlens the
device rejects must leave its outputs unwritten, and the good call after it
must not see the error word the failed call left behind.  Kept in its own
file, collected last."""
import ctypes

import pytest
import torch

import parity
from gated_delta_rule_45_gb300 import kda, synth

pytestmark = pytest.mark.gpu

SPECS = [
    synth.PrefillSpec(num_seqs=5, len_lo=1, len_hi=300, H=2, d_k=128, d_v=256, chunk=64,
                      s0_std=0.1, seed=21),
    synth.PrefillSpec(num_seqs=3, len_lo=40, len_hi=200, H=3, d_k=128, d_v=128, chunk=64,
                      s0_std=0.1, seed=22),
]


def _noalloc_via_c_abi(lib, dev, o, S_T, chunk, cu=None):
    T, H, d_k = dev["q"].shape
    d_v = dev["v"].shape[2]
    cu = dev["cu_seqlens"] if cu is None else cu
    N = cu.numel() - 1
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return lib.kda_prefill_noalloc(p(dev["q"]), p(dev["k"]), p(dev["v"]), p(dev["alpha"]),
                                   p(dev["beta"]), p(dev["S0"]), p(cu), N, T, H,
                                   d_k, d_v, kda.BF16, chunk, p(o), p(S_T),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _reference(dev, spec):
    return kda.prefill(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], dev["S0"],
                       dev["cu_seqlens"], chunk=spec.chunk, check_device_status=True)


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    lib = kda.load()
    for i, spec in enumerate(SPECS):
        d = synth.prefill_inputs(spec)
        dev = parity.to_device(d)
        o_ref, S_ref = _reference(dev, spec)
        o = torch.full_like(o_ref, float("nan"))
        S_T = torch.full_like(S_ref, float("nan"))
        assert _noalloc_via_c_abi(lib, dev, o, S_T, spec.chunk) == kda.OK
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(S_T, S_ref)
        if i == 0:
            pairs = [(n, h) for n in range(spec.num_seqs) for h in range(spec.H)]
            wo, ws = parity.compare_pairs(d, o, S_T, parity.oracle_pairs(d, pairs))
            assert wo <= parity.TOL_BF16 and ws <= parity.TOL_BF16, (wo, ws)


def test_noalloc_recovers_after_a_rejected_call():
    lib = kda.load()
    spec = SPECS[1]
    d = synth.prefill_inputs(spec)
    dev = parity.to_device(d)
    o_ref, S_ref = _reference(dev, spec)
    # cu_seqlens that decreases: the planner flags it and no output is written
    cu = dev["cu_seqlens"].cpu().tolist()
    cu[1], cu[2] = cu[2], cu[1]
    bad = torch.tensor(cu, dtype=torch.int32, device="cuda")
    assert cu[2] < cu[1]
    o = torch.full_like(o_ref, float("nan"))
    S_T = torch.full_like(S_ref, float("nan"))
    assert _noalloc_via_c_abi(lib, dev, o, S_T, spec.chunk, cu=bad) == kda.OK
    torch.cuda.synchronize()
    assert torch.isnan(o.float()).all() and torch.isnan(S_T).all()
    # the next call clears the error word it finds and runs normally
    assert _noalloc_via_c_abi(lib, dev, o, S_T, spec.chunk) == kda.OK
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(S_T, S_ref)


def test_noalloc_rejects_too_many_sequences():
    lib = kda.load()
    fake = ctypes.c_void_p(0x10000)
    st = lib.kda_prefill_noalloc(fake, fake, fake, fake, fake, None, fake,
                                 kda.NOALLOC_MAX_SEQS + 1, 64, 1, 128, 128, kda.BF16, 64,
                                 fake, fake, None)
    assert st == kda.ERR_UNSUPPORTED
