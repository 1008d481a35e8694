"""The sequence axis split across processes (gated_delta_rule_45_gb300.seqpar)
on two gloo ranks on CPU, each step taken by the oracle: every rank's segment
output and the batch's final state against the oracle over the whole
sequences.  This checks the exchange (the all-gather of the segment maps), the
scan over the ranks before each one and the maps' construction from special
prefills; the GPU version of each step is checked in test_seqpar_gpu.py."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from gated_delta_rule_45_gb300 import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


SPEC = synth.PrefillSpec(num_seqs=3, len_lo=40, len_hi=150, H=2, d_k=16, d_v=24,
                         s0_std=0.3, alpha_mu=2.0, seed=51)


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    from gated_delta_rule_45_gb300 import seqpar
    import seqpar_reference as ref
    dist.init_process_group("gloo", rank=rank, world_size=world)
    d = synth.prefill_inputs(SPEC)
    seg = ref.split_batch(d, world)[rank]
    o, S_T = seqpar.prefill_sequence_parallel(
        seg["q"], seg["k"], seg["v"], seg["alpha"], seg["beta"],
        d["S0"] if rank == 0 else None, seg["cu_seqlens"], backend=ref.OracleBackend())
    out[rank] = (seg["idx"].numpy(), o.numpy(), S_T.numpy())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ranks_match_the_whole_sequence(world):
    """With 3 ranks the last one chains two earlier segments' maps."""
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    d = synth.prefill_inputs(SPEC)
    o_ref, S_ref = oracle.prefill(synth.bf16_bits(d["q"]), synth.bf16_bits(d["k"]),
                                  synth.bf16_bits(d["v"]), d["alpha"].numpy(), d["beta"].numpy(),
                                  d["S0"].double().numpy(), d["cu_seqlens"].numpy())
    for r in range(world):
        idx, o, S_T = out[r]
        np.testing.assert_allclose(o, o_ref[idx], rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(S_T, S_ref, rtol=1e-9, atol=1e-11)
