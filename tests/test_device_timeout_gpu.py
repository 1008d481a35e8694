"""The device-side wait limit of the tensor-core prefill, run on purpose.

kda_check_wait_timeout enqueues one CTA that allocates tensor memory as the
prefill kernel does, waits with a 1 ms limit on an mbarrier nothing arrives
on, and waits on a second one with the prefill's own 2 s limit until the
first warp's failure stops it.  Nothing faults or hangs: the kernel returns,
the workspace's status word reads KDA_ERR_DEVICE_TIMEOUT, the tensor memory
is free again for the next launch, and a prefill right after is correct."""
import time

import pytest
import torch

import parity
from gated_delta_rule_45_gb300 import kda, synth

pytestmark = pytest.mark.gpu


def _timeout_once(ws):
    kda.check_wait_timeout(ws, 1_000_000)
    with pytest.raises(kda.KdaError) as e:
        kda.device_status(ws)
    assert e.value.status == kda.ERR_DEVICE_TIMEOUT


def test_wait_runs_out_and_the_context_stays_usable():
    ws = torch.empty(kda.workspace_size(0), dtype=torch.uint8, device="cuda")
    _timeout_once(ws)
    # a second launch allocates the tensor memory again: the first one freed it;
    # its second warp ends through the abort flag, well before its own 2 s limit
    t0 = time.perf_counter()
    _timeout_once(ws)
    assert time.perf_counter() - t0 < 1.5
    # a normal prefill afterwards is unaffected
    spec = synth.PrefillSpec(num_seqs=3, len_lo=60, len_hi=200, H=2, d_k=128, d_v=128,
                             s0_std=0.1, seed=31)
    d = synth.prefill_inputs(spec)
    dev = parity.to_device(d)
    o, S_T = kda.prefill(dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"], dev["S0"],
                         dev["cu_seqlens"], chunk=64, kernel="tc", check_device_status=True)
    pairs = [(n, h) for n in range(spec.num_seqs) for h in range(spec.H)]
    wo, ws_ = parity.compare_pairs(d, o, S_T, parity.oracle_pairs(d, pairs))
    assert wo <= parity.TOL_BF16 and ws_ <= parity.TOL_BF16, (wo, ws_)


def test_timeout_check_rejects_bad_arguments():
    ws = torch.empty(kda.workspace_size(0), dtype=torch.uint8, device="cuda")
    for bad in (10, 2_000_000_000):
        with pytest.raises(kda.KdaError) as e:
            kda.check_wait_timeout(ws, bad)
        assert e.value.status == kda.ERR_INVALID_ARG
