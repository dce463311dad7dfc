"""The multi-rank side of the benchmark on the CPU (gloo, world size 2): each
rank runs the same step on its own token batch with no data exchange, and the
job's time is the slowest rank's, so the reported throughput is
world * bytes per rank / max time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, result_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r took (r + 1) * 10 ms for its steps
        t = bench.max_over_ranks(10.0 * (rank + 1), dist, "cpu")
        gbs = bench.job_gbs(world, 1e9, t)
        dist.barrier()
        result_q.put((rank, t, gbs))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_time_and_job_throughput():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, t, gbs in got:
        assert t == pytest.approx(20.0)  # the slower rank's time on every rank
        assert gbs == pytest.approx(2 * 1e9 / 0.020 / 1e9)


def test_single_process_is_a_no_op():
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.job_gbs(1, 6e9, 1.0) == pytest.approx(6000.0)
