"""The replica path of bench.py with two gloo ranks on the CPU: each rank trains its own
views (no view trained twice in a step, every view of the dealt batches covered) and the
timing is the maximum over the ranks."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        batch, n_views, steps = 4, 64, 10
        mine = torch.tensor([bench.rank_views(s, rank, world, batch, n_views) for s in range(steps)])
        got = [torch.zeros_like(mine) for _ in range(world)]
        dist.all_gather(got, mine)
        t = bench.max_over_ranks(1.5 + rank, dist, "cpu")
        if rank == 0:
            out.put(([g.tolist() for g in got], t))
    finally:
        dist.destroy_process_group()


def test_replica_views_and_max_timing():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    views, t = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert t == 2.5  # the slower rank's time
    for s in range(10):
        step = [v for r in range(world) for v in views[r][s]]
        assert len(set(step)) == len(step)  # no view trained twice in a step
        # the ranks' batches are consecutive slices of the view list
        assert sorted(step) == sorted(((s * world) * 4 + b) % 64 for b in range(world * 4))
    assert bench_single_rank_is_identity()


def bench_single_rank_is_identity():
    import bench
    return bench.max_over_ranks(3.0, None, "cpu") == 3.0 and bench.rank_views(2, 0, 1, 4, 64) == [8, 9, 10, 11]
