"""The N>1 benchmark path on CPU: two gloo ranks agree on the max time and the whole-job sum."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    mx = bench.max_over_ranks(1.5 + rank, w)  # per-rank step times 1.5, 2.5
    sm = bench.sum_over_ranks(100.0 * (rank + 1), w)  # per-rank bytes
    dist.destroy_process_group()
    q.put((r, w, lr, mx, sm))


@pytest.mark.parametrize("world", [2])
def test_replica_aggregation_over_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, w, lr, mx, sm) in enumerate(res):
        assert (rank, w, lr) == (r, world, r)
        assert mx == 2.5 and sm == 300.0


def test_single_process_identity():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0 and bench.sum_over_ranks(7.0, 1) == 7.0
