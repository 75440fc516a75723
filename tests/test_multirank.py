"""The benchmark's cross-rank step: each rank runs the whole step on its own
GPU, the job's time is the slowest rank's and its work is world x one step.
Checked with two gloo ranks on the CPU (the GPU run uses NCCL; the host logic
is the same)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, ms, flops, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        q.put((rank, bench.over_ranks(ms[rank], flops, dist, "cpu")))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run(world, ms, flops):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, ms, flops, q)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        got = dict(q.get(timeout=120) for _ in range(world))
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    return got


def test_two_ranks_slowest_time_and_whole_job_throughput():
    flops = 3.0e12
    got = _run(2, [1.25, 2.5], flops)
    want = (2.5, flops * 2 / 2.5e-3 / 1e12)
    assert got[0] == pytest.approx(want) and got[1] == pytest.approx(want)


def test_equal_ranks_scale_weakly():
    """Equal per-rank times: the job's throughput is world x one rank's."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    flops = 1.0e12
    one_ms, one_value = bench.over_ranks(4.0, flops)
    got = _run(2, [4.0, 4.0], flops)
    assert got[0][0] == one_ms and got[0][1] == pytest.approx(2 * one_value)
