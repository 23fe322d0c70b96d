"""The N > 1 path of bench.py on CPU: two gloo ranks run the same replica
logic the GPU ranks run (barrier, max over ranks of the step time, whole-job
GB/s), with different local step times."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q) -> None:
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        local = [0.004, 0.005][rank]                 # rank 1 is the slower replica
        step = bench.slowest_rank(local, dist, "cpu")
        dist.barrier()
        q.put((rank, step, bench.job_gbps(world, 31_000_000_000, step)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_replica():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, step, gbps in got:
        assert step == pytest.approx(0.005)
        assert gbps == pytest.approx(2 * 31.0 / 0.005)


def test_single_replica_is_local():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank(0.0042, None, "cpu") == 0.0042
    assert bench.job_gbps(1, 10_000_000_000, 0.01) == pytest.approx(1000.0)
