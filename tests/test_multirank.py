"""The bench's multi-rank host logic on CPU: two processes over gloo.

With N > 1 every rank verifies its own rows (replicas, no data-path
collective); the only exchange is the timing: each rank's elapsed time is
reduced to the maximum, and the whole-job rate counts the rows of all ranks.
The reference arm runs on rank 0 alone. Runs without a GPU.
"""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, _ = bench.dist_env()
    local_ms = 1.0 + 0.5 * rank          # the last rank is the slowest
    m = bench.max_over_ranks(local_ms)
    rate = bench.job_rate(w, 256, 4, m)
    skipped = bench.run_reference(None, rank, w, 1.0) if rank != 0 else "rank 0"
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, r, w, m, rate, skipped))


@pytest.mark.parametrize("world", [2, 3])
def test_ranks_reduce_to_the_slowest(world):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=180) for _ in ps)
    for p in ps:
        p.join(timeout=60)
    assert all(p.exitcode == 0 for p in ps)
    slowest = 1.0 + 0.5 * (world - 1)
    for rank, r, w, m, rate, skipped in res:
        assert r == rank and w == world
        assert m == slowest                                    # every rank sees the max
        assert rate == pytest.approx(world * 256 * 4 / (slowest / 1e3))
        if rank != 0:
            assert skipped is None                              # no reference work off rank 0


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.job_rate(1, 256, 4, 0.5) == pytest.approx(256 * 4 / 0.5e-3)
