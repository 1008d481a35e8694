"""kda_prefill_noalloc, the entry point for callers that cannot allocate
device memory (its scratch is built into the library), against kda_prefill
with a caller-provided workspace.  Two calls in a row on different batches:
the second must not be disturbed by what the first left in the shared
scratch.  Kept in its own file, collected last."""
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


def _noalloc_via_c_abi(lib, dev, o, S_T, chunk):
    T, H, d_k = dev["q"].shape
    d_v = dev["v"].shape[2]
    N = dev["cu_seqlens"].numel() - 1
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return lib.kda_prefill_noalloc(p(dev["q"]), p(dev["k"]), p(dev["v"]), p(dev["alpha"]),
                                   p(dev["beta"]), p(dev["S0"]), p(dev["cu_seqlens"]), N, T, H,
                                   d_k, d_v, kda.BF16, chunk, p(o), p(S_T),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    lib = kda.load()
    for spec in SPECS:
        d = synth.prefill_inputs(spec)
        dev = parity.to_device(d)
        o_ref, S_ref = kda.prefill(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"],
                                   dev["S0"], dev["cu_seqlens"], chunk=spec.chunk,
                                   check_device_status=True)
        o = torch.full_like(o_ref, float("nan"))
        S_T = torch.full_like(S_ref, float("nan"))
        assert _noalloc_via_c_abi(lib, dev, o, S_T, spec.chunk) == kda.OK
        torch.cuda.synchronize()
        assert torch.isfinite(o.float()).all() and torch.isfinite(S_T).all()
        assert parity.rel(o.float().cpu().numpy(), o_ref.float().cpu().numpy()) <= parity.TOL_BF16
        assert parity.rel(S_T.cpu().numpy(), S_ref.cpu().numpy()) <= parity.TOL_BF16


def test_noalloc_rejects_too_many_sequences():
    lib = kda.load()
    fake = ctypes.c_void_p(0x10000)
    st = lib.kda_prefill_noalloc(fake, fake, fake, fake, fake, None, fake,
                                 kda.NOALLOC_MAX_SEQS + 1, 64, 1, 128, 128, kda.BF16, 64,
                                 fake, fake, None)
    assert st == kda.ERR_UNSUPPORTED
