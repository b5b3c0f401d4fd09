"""The multi-GPU path is replicas (weak scaling): each rank runs its own batch and only the timing
and byte totals cross ranks.  This checks that host logic with two gloo ranks on the CPU."""
import os
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r moved (r+1) GB and 10*(r+1) sequences in (r+1) * 0.5 s
    gbs, seqs, elapsed = bench.aggregate((rank + 1) * 1e9, 10.0 * (rank + 1), 0.5 * (rank + 1), world)
    q.put((rank, gbs, seqs, elapsed))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_weak_scaling_aggregation_over_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slowest = 0.5 * world
    total_gb = sum(r + 1 for r in range(world))
    for _, gbs, seqs, elapsed in res:
        assert elapsed == pytest.approx(slowest)
        assert gbs == pytest.approx(total_gb / slowest)
        assert seqs == pytest.approx(10.0 * total_gb / slowest)


def test_single_rank_aggregation_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(2e9, 32.0, 0.25, 1) == pytest.approx((8.0, 128.0, 0.25))
