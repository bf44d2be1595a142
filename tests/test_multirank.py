"""The bench's multi-rank path on the CPU: two gloo ranks on 127.0.0.1.

Every (layer, b, h) unit is independent, so N GPUs run N replicas with no
collective on the data path; the only cross-rank steps are the barriers
around the timed region and the max over ranks of the measured time. These
run here with the gloo backend: the slowest rank's time is what every rank
reports, and the whole-job throughput counts all ranks' units.
"""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        w, r, lr = bench._dist()
        assert (w, r, lr) == (world, rank, rank)
        dist.barrier()
        ms = bench.max_over_ranks(times[rank], device="cpu")
        value = bench.job_throughput(w, 1000.0, ms)
        out.put((rank, ms, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_time_and_the_whole_job():
    world, times = 2, [3.0, 5.0]
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, ms, value in got:
        assert ms == 5.0                                  # every rank reports the slowest rank
        assert value == pytest.approx(2 * 1000.0 / 5e-3)  # all ranks' units over that time


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(4.5, device="cpu") == 4.5
    assert bench.job_throughput(1, 10.0, 2.0) == pytest.approx(5000.0)
