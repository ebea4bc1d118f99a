"""The benchmark's multi-rank plumbing on CPU: two gloo ranks, barrier and max-over-ranks
timing. The data path itself has no collective (each rank decodes its own batch)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, lr = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    bench.barrier(w)
    t = bench.max_over_ranks(1.5 + rank, w, "cpu")
    tokens = w * 256 * 16 * 10
    q.put((r, lr, t, tokens / t))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=100) for _ in range(2))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1] and [o[1] for o in out] == [0, 1]
    assert all(o[2] == 2.5 for o in out)                 # max over ranks
    assert all(abs(o[3] - 2 * 256 * 16 * 10 / 2.5) < 1e-6 for o in out)
