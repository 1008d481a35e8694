"""The bench's multi-process aggregation on CPU: two gloo ranks, each with
its own elapsed time and unit count; every rank must see the maximum time
and the summed units (weak scaling: value = all ranks' units / slowest rank)."""
import os
import socket

import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    bench.init_dist("gloo")
    bench.barrier()
    t, u = bench.reduce_max_sum(elapsed_s=1.5 + rank, units=100.0 * (rank + 1))
    out[rank] = (t, u)
    torch.distributed.destroy_process_group()


def test_two_rank_max_time_and_sum_of_units():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()   # no fork of this multi-threaded process
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0] == out[1] == (2.5, 300.0)


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max_sum(3.0, 7.0) == (3.0, 7.0)
    assert bench.dist_env()[0] >= 1
