"""The N > 1 host path of the bench on CPU: two gloo ranks (no GPU).

Decode shards by sequence with no exchange on the data path; the only
collectives are the bench's barrier and the max-over-ranks of the timings.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w = bench.init_dist("gloo")
    assert (r, w) == (rank, world)
    bench.barrier()
    slowest = bench.max_over_ranks(10.0 + rank)          # rank 1 is the slow one
    # the reference arm: rank 0 alone works, the others return without work
    skipped = bench.dist_env()[0] != 0 and bench.run_reference(None) is None
    results[rank] = (slowest, skipped)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_only_rank0_reports():
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(2, port, results), nprocs=2, join=True)
        res = dict(results)
    assert res[0][0] == pytest.approx(11.0) and res[1][0] == pytest.approx(11.0)
    assert res[1][1] is True


def test_single_process_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    bench.barrier()
