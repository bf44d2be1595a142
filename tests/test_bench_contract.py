"""The bench's host-side contract on the CPU: the algorithmic work behind the roofline, and the
reference arm's JSON line (the CPU oracle on a bounded sample)."""
import json
import os
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class _FakeBinding:
    """Stands in for the library: the last update moved `old` kept rows and wrote `new` rows."""

    def __init__(self, old, new):
        self.old, self.new = old, new

    def evict_compaction_rows(self, h):
        return self.old, self.new


class _FakeRun:
    def __init__(self, w, rows_per_call):
        self.w, self.rows_per_call, self.handles = w, rows_per_call, [object()]


def test_algorithmic_bytes_of_the_stack_step():
    w = bench.WORKLOADS["qfilters_stack"]
    run = _FakeRun(w, w["seq"])
    units = w["layers"] * w["batch"] * w["heads"]
    survivors = units * w["budget"]
    work = bench.algorithmic_work(run, _FakeBinding(0, survivors))
    # score: every key read once (128 bf16), its fp32 score written
    assert work["score"]["bytes"] == units * w["seq"] * (128 * 2 + 4)
    # compaction of a prefill: each survivor's K and V read and written, plus position, score, map
    assert work["compact"]["bytes"] == survivors * (4 * 128 * 2 + 16)
    # selection: n scores read, the budget-long map written, the flags of the 64-row compaction
    # chunks and the chunk counter reset, the metadata
    flags = w["budget"] // 64 + 1
    assert work["select"]["bytes"] == units * (4 * w["seq"] + 4 * w["budget"] + 4 * flags + 8)


@pytest.mark.parametrize("method,per_row", [("h2o", 128 * 2 + 16), ("curdkv", 128 * 2 + 4)])
def test_algorithmic_bytes_of_the_short_block_attention(method, per_row):
    # a decode step: every unit reads its budget + 1 key rows once and writes their column sums
    w = dict(bench.WORKLOADS["decode"], method=method)
    units = w["batch"] * w["heads"]
    work = bench.algorithmic_work(_FakeRun(w, w["budget"] + 1), _FakeBinding(0, 0))
    assert work["curdkv_attn_small"]["bytes"] == units * (w["budget"] + 1) * per_row
    # per-token mode: each launch sees the budget's rows plus the token, whatever the call's rows
    w = dict(bench.WORKLOADS["curdkv_planted"], method=method, per_token=True)
    units = w["batch"] * w["heads"]
    work = bench.algorithmic_work(_FakeRun(w, w["existing"] + w["incoming"]), _FakeBinding(0, 0))
    assert work["curdkv_attn_small"]["bytes"] == units * (w["budget"] + 1) * per_row


def test_throughput_and_rank_helpers():
    assert bench.job_throughput(4, 1000.0, 2.0) == pytest.approx(2.0e6)
    assert bench.max_over_ranks(3.25, device="cpu") == 3.25


def test_reference_arm_prints_the_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "knorm_single",
                          "--steps", "1", "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads([l for l in out.stdout.splitlines() if l.startswith("{")][-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["config"]["workload"] == "knorm_single"
