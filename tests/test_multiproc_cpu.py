"""The multi-rank path of bench.py on CPU: two gloo ranks, barrier and
max-over-ranks timing, whole-job aggregation (replicas, weak scaling)."""
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


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, lr, w = bench.dist_env()
    assert (r, lr, w) == (rank, rank, world)
    bench.dist_init("gloo")
    bench.dist_barrier()
    my_ms = 10.0 + 5.0 * rank                    # the slower rank decides
    mx = bench.dist_max(my_ms)
    value = bench.aggregate(100.0, mx / 1e3, w)
    q.put((rank, mx, value))
    import torch.distributed as dist
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(120) if hasattr(pytest.mark, "timeout") else (lambda f: f)
def test_two_gloo_ranks_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, mx, value in res:
        assert mx == 15.0
        assert abs(value - 2 * 100.0 / 0.015) < 1e-6
