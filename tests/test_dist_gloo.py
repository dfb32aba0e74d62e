"""Host-side logic of the multi-GPU benchmark path, on CPU with gloo.

The hot path shards by batch: every rank verifies and realigns its own
independent batch, so the only cross-rank traffic is timing (a barrier and a
max-reduction of the elapsed time).  Two gloo ranks check the seed split, the
max-over-ranks reduction and the whole-job aggregation.
"""
import os

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_env()
        seed = bench.rank_seed(1002, r)
        t = 1.0 + r * 0.5  # rank 1 is slower
        tmax = bench.max_over_ranks(t, True)
        dist.barrier()
        q.put((r, lr, w, seed, tmax, bench.aggregate(50, tmax, w)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 2000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, lr0, w0, s0, t0, v0), (r1, lr1, w1, s1, t1, v1) = res
    assert (r0, r1, w0, w1) == (0, 1, 2, 2)
    assert s0 != s1  # independent batches
    assert t0 == t1 == 1.5  # the slowest rank's time
    assert v0 == v1 == pytest.approx(2 * 50 / 1.5)
