"""Multi-rank host logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

Every rank runs its own batch (weak scaling, no collective on the data path); the only
exchanges are the max of the ranks' times and the sum of their work, taken after the timed
region.  The reference arm runs on rank 0 alone.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, result_q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_setup(None)
        local_ms = [12.5, 20.0][rank]           # rank 1 is the slow one
        local_flops = [3.0e12, 5.0e12][rank]
        total_ms = bench.max_over_ranks(local_ms)
        total_flops = bench.sum_over_ranks(local_flops)
        value = bench.job_tflops(total_flops, total_ms)

        class Args:
            pass

        # the reference arm: ranks other than 0 return at once, without touching the oracle
        skipped = bench.run_reference(Args(), w, r) is None if r != 0 else True
        result_q.put((rank, w, r, local, total_ms, total_flops, value, skipped))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_time_and_work():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    for rank, w, r, local, total_ms, total_flops, value, skipped in results:
        assert (w, r, local) == (world, rank, rank)
        assert total_ms == 20.0                 # the slowest rank's time
        assert total_flops == 8.0e12            # the work of both ranks
        assert value == pytest.approx(8.0e12 / 20.0e-3 / 1e12)
        assert skipped


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5) == 3.5 and bench.sum_over_ranks(2.0) == 2.0
    assert bench.job_tflops(1.0337e12, 1.078) == pytest.approx(958.9, rel=1e-3)
