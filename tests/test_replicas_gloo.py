"""The multi-GPU path of bench.py is replicas only: N independent copies of
the decode step, one per GPU, timed between barriers, the job's time the
slowest rank's. Its host-side pieces run here as two gloo ranks on the CPU:
the max over ranks that every rank must agree on, the whole-job rate, and the
reference arm's rule that ranks other than 0 do no work."""

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


def _rank_main(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        dist.barrier()
        mx = bench.max_over_ranks(torch, dist, times[rank], torch.device("cpu"))
        rate = bench.job_rate(world, 20, 655_097_856, mx)

        class A:
            gpus, steps, warmup = world, 1, 0
        ref = bench.run_reference(A, rank, world) if rank != 0 else "skipped"
        out.put((rank, mx, rate, ref))
    finally:
        dist.destroy_process_group()


def test_two_replicas_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    times = [2.75, 3.125]   # ms of the timed steps on each rank
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, rate, ref in res:
        assert mx == max(times)
        # two replicas, 20 steps of 655.1 MB each, over the slower rank's 3.125 ms
        assert rate == pytest.approx(2 * 20 * 655_097_856 / 3.125e-3 / 1e9)
    # the reference arm's other ranks return without work (and print nothing)
    assert res[1][3] is None
