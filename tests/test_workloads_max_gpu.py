"""The largest sizes each entry point documents, against the oracle (GPU).

kda_prefill: d_k = 128 and d_v = 1024 (every kernel that takes the shape);
kda_decode_step: d_k = 256 and d_v = 4096; kda_backward: d_v = 1024.  Short
ragged sequences keep the oracle's share to a fraction of a second.
"""
import pytest

import parity
import test_backward_gpu as backward_cases
import test_decode_gpu as decode_cases
import test_prefill_gpu as prefill_cases
from gated_delta_rule_45_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,chunk", [("bf16", 64), ("fp32", 32)])
def test_prefill_widest_value_dimension(dtype, chunk):
    spec = synth.PrefillSpec(num_seqs=2, len_lo=70, len_hi=150, H=1, d_k=128, d_v=1024,
                             dtype=dtype, chunk=chunk, s0_std=0.1, seed=61)
    for kernel in prefill_cases._kernels_for(spec):
        prefill_cases._check(spec, kernel)


def test_decode_widest_state():
    spec = synth.DecodeSpec(B=2, H=1, d_k=256, d_v=4096, dtype="bf16", seed=62)
    wo, ws = decode_cases._run(spec)
    assert wo <= parity.TOL_BF16 and ws <= parity.TOL_BF16, (wo, ws)


def test_backward_widest_value_dimension():
    spec = synth.PrefillSpec(num_seqs=2, len_lo=70, len_hi=140, H=1, d_k=128, d_v=1024,
                             s0_std=0.1, seed=63)
    backward_cases._run(spec)
