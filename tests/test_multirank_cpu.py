"""Multi-rank host logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

Every rank runs its own batch (weak scaling, no collective on the data path); the only
exchanges are the max of the ranks' times and the sum of their work, taken after the timed
region.  The reference arm runs on rank 0 alone.  A batch can also be split by rows across the
ranks (row_shard): the shards partition the rows, and the per-shard results are exactly the
rows of the whole batch's result.
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


def _shard_main(rank, world, port, result_q):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import numpy as np
    import oracle
    import workloads as W
    from sparse_mla_attention_fwd_gb300 import row_shard
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = W.random_case(61, 23, 300, 64, 512, 90, with_len=True, with_sink=True)
        r0, r1 = row_shard(23, rank, world)
        # each rank computes its own rows only (the oracle stands in for the GPU here)
        out, lse, mx = oracle.sparse_mla_fwd(w["q"], w["kv"], w["indices"], w["topk_length"], w["attn_sink"],
                                             w["sm_scale"], rows=np.arange(r0, r1), threads=1)
        gathered = [None] * world
        dist.all_gather_object(gathered, (rank, r0, r1, lse.tolist()))
        result_q.put((rank, r0, r1, gathered))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_row_shards_partition_the_batch_and_reproduce_it(world):
    import numpy as np
    sys.path.insert(0, ROOT)
    import oracle
    import workloads as W
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    gathered = sorted(results[0][3])
    edges = [(r0, r1) for _, r0, r1, _ in gathered]
    assert edges[0][0] == 0 and edges[-1][1] == 23
    assert all(a[1] == b[0] for a, b in zip(edges, edges[1:]))          # contiguous, disjoint
    assert max(r1 - r0 for r0, r1 in edges) - min(r1 - r0 for r0, r1 in edges) <= 1
    w = W.random_case(61, 23, 300, 64, 512, 90, with_len=True, with_sink=True)
    _, lse_all, _ = oracle.sparse_mla_fwd(w["q"], w["kv"], w["indices"], w["topk_length"], w["attn_sink"],
                                          w["sm_scale"], threads=1)
    stitched = np.concatenate([np.array(l) for _, _, _, l in gathered])
    assert np.array_equal(stitched, lse_all)


def test_row_shard_edges():
    from sparse_mla_attention_fwd_gb300 import row_shard
    assert [row_shard(10, r, 4) for r in range(4)] == [(0, 3), (3, 6), (6, 8), (8, 10)]
    assert row_shard(0, 0, 2) == (0, 0) and row_shard(3, 2, 5) == (2, 3) and row_shard(3, 3, 5) == (3, 3)
    with pytest.raises(ValueError):
        row_shard(5, 2, 2)
