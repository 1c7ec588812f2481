"""The N-rank bench path on CPU: two gloo ranks combine their timings and counts
the way bench.py does under torchrun (slowest rank's time, summed work), and
each rank draws its own batch.  No GPU is used."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        ms = 10.0 + 5.0 * rank           # rank 1 is the slower one
        units = [24 + rank, 100.0 * (rank + 1)]
        ms_max, totals = bench.across_ranks(ms, units, w)
        queue.put((r, w, local, ms_max, totals, bench.rank_seed(622, r)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_bench():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, l0, ms0, tot0, seed0), (r1, w1, l1, ms1, tot1, seed1) = out
    assert (r0, r1, w0, w1, l0, l1) == (0, 1, 2, 2, 0, 1)
    assert ms0 == ms1 == 15.0                 # max over ranks
    assert tot0 == tot1 == [49.0, 300.0]      # sums over ranks
    assert seed0 == 622 and seed1 != seed0    # rank 0 keeps the 1-GPU batch


def test_single_rank_needs_no_process_group():
    import bench
    ms, tot = bench.across_ranks(3.5, [1, 2], 1)
    assert ms == 3.5 and tot == [1.0, 2.0]
