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


# ---------------------------------------------------------------------------
# The batch-row partition of the long-context stream: rank r owns rows
# rank_rows(r) of the global batch; the union of the ranks' kept caches and
# the sum of their byte accounting equal one process over the whole batch.
# ---------------------------------------------------------------------------
SHARD = dict(rows=2, heads=2, block=192, blocks=3, budget=128)


def _shard_results(first_row, rows):
    from kv_cache_token_bf16_gb300 import synth
    from oracle import calibrate as ocal
    from oracle.cache import OracleCache
    import numpy as np
    H = SHARD["heads"]
    filt = ocal.calibrate(synth.long_context_queries(H, n_samples=300), H).astype(np.float32)
    out = {}
    for method, kw in (("knorm", {}), ("qfilters", {"filters": filt}), ("curdkv", {"rank_cap": 16})):
        c = OracleCache(method, rows, H, budget=SHARD["budget"], n_sink=4, **kw)
        for blk in range(SHARD["blocks"]):
            k, v = synth.long_context_block(blk, rows, H, SHARD["block"], first_row=first_row)
            c.update_and_fetch(k, v)
        out[method] = (c.pos.copy(), c.k.copy(), np.asarray(c.score, np.float64).copy(), c.stats())
    return out


def _shard_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        first, rows = bench.rank_rows(rank, world, SHARD["rows"])
        res = _shard_results(first, rows)
        dist.barrier()                                    # no data crosses ranks: only the host results
        out.put((rank, first, res))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_partition_the_batch_rows():
    import numpy as np
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((out.get(timeout=300) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [0, SHARD["rows"]]
    whole = _shard_results(0, world * SHARD["rows"])
    for method, (pos, k, score, stats) in whole.items():
        parts = [g[2][method] for g in got]
        assert np.array_equal(np.concatenate([p[0] for p in parts]), pos), method
        assert np.array_equal(np.concatenate([p[1] for p in parts]), k), method
        assert np.array_equal(np.concatenate([p[2] for p in parts]), score), method
        # byte accounting: the global cache's bytes are the ranks' sums; the calibrated filter is
        # one per layer, held by every rank
        filt = SHARD["heads"] * 128 * 4 if method == "qfilters" else 0
        assert sum(p[3]["kept_bytes"] - filt for p in parts) + filt == stats["kept_bytes"]
        assert sum(p[3]["full_seq_bytes"] for p in parts) == stats["full_seq_bytes"]
        assert all(p[3]["tokens_seen"] == stats["tokens_seen"] for p in parts)


def test_rank_rows_cover_the_batch_once():
    import bench
    rows = [bench.rank_rows(r, 8, 4) for r in range(8)]
    covered = [i for first, n in rows for i in range(first, first + n)]
    assert covered == list(range(32))
    with pytest.raises(ValueError):
        bench.rank_rows(8, 8, 4)
