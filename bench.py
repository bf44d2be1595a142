"""Throughput of block KV-cache eviction on GB300 through libevict.

Default run (the largest single-GPU workload, every scorer): the long-context
chunked prefill. B=4 sequences, 8 KV heads, D=128, bf16; a 131072-token
stream arrives in 16 blocks of 8192 tokens; budget 4096, n_sink 4, recent 0.
One step = the whole hot path over that batch for all three scorers: a KNorm
cache (keep low), a calibrated Q-Filters cache (filters from the GPU
calibration on the workload's queries, run once before timing) and a CurDKV
cache (rank 16, proxy queries = each block's keys) are each reset and absorb
the 16 blocks (score, protected top-k, order-preserving compaction).

Metric: cache tokens evicted-and-compacted per second, summed over the
scorers, blocks and (b, h) units (each update counts the k + m rows it
scores and selects from), with the dominant kernel's achieved rate against
its roofline and every scorer's whole-path fraction of its binding resource.

The same JSON line carries, under "configs", the other single-GPU workloads,
each with its own step time, rooflines, clocks and CPU baseline:
  qfilters_stack  28 Llama-3.2-3B-like layers (24 query / 8 KV heads), one
                  8192-token prefill per layer, budget 1024, one grouped call;
  decode          B=32, H=8, 2048-token prefill then single-token steps,
                  budget 512, recent 128 (KNorm; the whole 4096-step stream is
                  also replayed as captured CUDA graphs, "stream");
  curdkv_planted  B=H=8, 16384 kept rows + a 512-token block, budget 2048.

--workload picks one of them (or knorm_single) alone; --method picks one
scorer for long_context / decode (knorm, qfilters, qfilters_fallback, curdkv,
h2o) or curdkv_planted (curdkv, h2o); --per-token runs curdkv_planted through
the pages' token-by-token loop.

Arms:
  --impl ours       (default) libevict on the GPU
  --impl reference  the CPU oracle (numpy), as it stands, on a bounded sample
                    of the same workload; prints the same JSON line.

Multi-GPU (torchrun): the batch is partitioned by sequence. Rank r owns rows
4r .. 4r+3 of a global batch of 4N sequences (each row is drawn from its own
seeded stream, so the shards are exactly the rows of the global batch); no
collective touches the data path. value = all ranks' tokens / the slowest
rank's time ("scaling": "weak"). The sub-records run at N=1 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from kv_cache_token_bf16_gb300 import synth  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# fp32 FMA peak: 152 SMs x 128 fp32 lanes x 2 flops x 2.07 GHz maximum SM clock
FP32_FMA_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
METRIC = "cache tokens evicted-and-compacted/sec per layer; achieved HBM GB/s vs roofline"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 512 << 20          # written between timed steps where the inputs could sit in L2
HEADLINE = "long_context"
SUB_CONFIGS = ("qfilters_stack", "decode", "curdkv_planted")


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------
WORKLOADS = {
    "long_context": dict(scorers=("knorm", "qfilters", "curdkv"), layers=1, batch=4, heads=8, block=8192,
                         blocks=16, budget=4096, n_sink=4, recent=0, rank_cap=16, dtype="bf16"),
    "qfilters_stack": dict(method="qfilters", layers=28, batch=1, heads=8, q_heads=24, seq=8192, budget=1024,
                           n_sink=4, recent=0, dtype="bf16"),
    "decode": dict(method="knorm", layers=1, batch=32, heads=8, prefill=2048, steps=4096, budget=512, n_sink=4,
                   recent=128, dtype="bf16"),
    "curdkv_planted": dict(method="curdkv", layers=1, batch=8, heads=8, existing=16384, incoming=512,
                           budget=2048, n_sink=4, recent=0, rank_cap=16, dtype="bf16"),
    "knorm_single": dict(method="knorm", layers=1, batch=1, heads=1, seq=1024, budget=512, n_sink=4, recent=0,
                         dtype="fp32"),
}


def max_over_ranks(x: float, device: str = "cuda") -> float:
    """The largest value of x over the ranks (x itself without a process group): every rank's
    timed region is bracketed by the same barriers, so the slowest rank sets the job's time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_rank: float, ms_per_step: float) -> float:
    """Whole-job throughput: the units all ranks processed (weak scaling: each rank a fixed
    share) divided by the slowest rank's time per step."""
    return world * units_per_rank / (ms_per_step / 1e3)


def rank_rows(rank: int, world: int, rows_per_rank: int):
    """Batch rows of the global batch (rows_per_rank * world sequences) that `rank` owns:
    a contiguous slice, disjoint across ranks, together the whole batch."""
    if not 0 <= rank < world:
        raise ValueError("rank outside the world")
    return rank * rows_per_rank, rows_per_rank


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _peaks():
    """Roofline denominators: the measured copy bandwidth and bf16 GEMM rate."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"])}, \
            "measured (MEASURED_PEAKS.json: HBM copy bandwidth; bf16 GEMM burst)"
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS}, "fallback"


def _source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "kv_cache_token_bf16_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _ncu_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("source_hash") != _source_hash(*rec.get("sources", [])):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)                 # the first sample lands inside the region
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        self.tmp.flush()
        with open(self.tmp.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.tmp.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if len(r) > 2 and r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if len(r) > 2 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ----------------------------------------------------------------------------
# GPU arm: one class per workload
# ----------------------------------------------------------------------------
class StackRun:
    """Q-Filters layer stack: 28 caches updated by one grouped call per step."""

    l2_note = "inputs larger than L2 (940 MB per step)"

    def __init__(self, w, torch, binding, stream):
        self.w, self.torch, self.binding = w, torch, binding
        L, H, S = w["layers"], w["heads"], w["seq"]
        self.k, self.v = [], []
        self.filters = []
        self.calib_ms = 0.0
        for layer in range(L):
            d = synth.qfilters_layer(layer, n_q_heads=w["q_heads"], n_kv_heads=H, seq_len=S, batch=w["batch"])
            self.k.append(torch.from_numpy(d["k"].view(np.int16)).cuda().view(torch.bfloat16))
            self.v.append(torch.from_numpy(d["v"].view(np.int16)).cuda().view(torch.bfloat16))
            qd = torch.from_numpy(d["queries"].view(np.int16)).cuda()
            f = torch.empty((H, 128), dtype=torch.float32, device="cuda")
            t0 = time.perf_counter()
            binding.evict_qfilters_calibrate(qd.data_ptr(), binding.EVICT_BF16, w["q_heads"], qd.shape[1], 128, H,
                                             f.data_ptr(), stream.cuda_stream)
            self.calib_ms += (time.perf_counter() - t0) * 1e3 / L
            self.filters.append(f)
        self.caches = [binding.EvictCache("qfilters", w["batch"], H, budget=w["budget"], n_sink=w["n_sink"],
                                          recent=w["recent"], max_block=S, filters=f, sign=1,
                                          stream=stream.cuda_stream) for f in self.filters]
        self.handles = [c.handle for c in self.caches]
        self.kp = [t.data_ptr() for t in self.k]
        self.vp = [t.data_ptr() for t in self.v]
        self.tokens_per_step = L * w["batch"] * H * S
        self.calls_per_step = 1
        self.rows_per_call = S
        self.method = "qfilters"

    def step(self):
        for h in self.handles:
            self.binding.evict_reset(h)
        self.binding.evict_update_and_fetch_group(self.handles, self.kp, self.vp, None, self.w["seq"])

    # end-to-end through the public host-buffer call: inputs start in pinned host memory, and the
    # kept caches (K, V, positions) come back to pinned host memory
    def setup_e2e(self):
        torch = self.torch
        self.kh = [t.view(torch.int16).cpu().pin_memory() for t in self.k]
        self.vh = [t.view(torch.int16).cpu().pin_memory() for t in self.v]
        self.out = [_HostCache(torch, self.w["batch"], self.w["heads"], self.w["budget"]) for _ in self.caches]
        self.h2d = sum(t.numel() * 2 for t in self.kh) + sum(t.numel() * 2 for t in self.vh)
        self.d2h = sum(o.nbytes for o in self.out)

    def step_e2e(self):
        for i, h in enumerate(self.handles):
            self.binding.evict_reset(h)
            view = self.binding.evict_update_and_fetch_host(h, self.kh[i].data_ptr(), self.vh[i].data_ptr(), None,
                                                            self.w["seq"])
            self.out[i].fetch(self.binding, view, self.w["batch"], self.w["heads"])


class _HostCache:
    """Pinned host buffers for one kept cache (K, V bf16 bits, positions): the e2e read-back."""

    def __init__(self, torch, B, H, rows):
        self.k = torch.empty((B, H, rows, 128), dtype=torch.int16).pin_memory()
        self.v = torch.empty_like(self.k).pin_memory()
        self.pos = torch.empty((B, H, rows), dtype=torch.int32).pin_memory()
        self.nbytes = 2 * self.k.numel() * 2 + self.pos.numel() * 4

    def fetch(self, binding, view, B, H):
        k, v, pos, _ = binding.view_tensors(view, B, H, "bf16")
        import torch
        self.k.copy_(k.view(torch.int16), non_blocking=True)
        self.v.copy_(v.view(torch.int16), non_blocking=True)
        self.pos.copy_(pos, non_blocking=True)


def _scorer_kwargs(method, H, torch=None):
    """Cache arguments of a scorer: the library method name and extra keywords. Q-Filters on the
    decode stream: seeded unit filters; qfilters_fallback: no filters, the key-SVD fallback freezing
    after 128 keys."""
    if method == "qfilters_fallback":
        return "qfilters", {"filters": None, "calib_tokens": 128, "sign": 1}
    if method == "qfilters":
        f = synth.decode_filters(H)
        return "qfilters", {"filters": torch.from_numpy(f).cuda() if torch else f, "sign": 1}
    if method == "curdkv":
        return "curdkv", {"rank_cap": 16}
    return method, {}                     # knorm, h2o


class DecodeRun:
    """Decode streaming: after a 2048-token prefill, one step = one single-token update.
    Before each timed step the L2 is flushed (outside the timed events), so a step reads the
    kept cache from HBM."""

    l2_note = "L2 flushed before every timed step (512 MB write outside the events)"
    flush_l2 = True

    def __init__(self, w, torch, binding, stream):
        self.w, self.torch, self.binding = w, torch, binding
        B, H = w["batch"], w["heads"]
        self.method = w["method"]
        k0, v0 = synth.decode_prefill(B, H, w["prefill"])
        self.k0 = torch.from_numpy(k0.view(np.int16)).cuda().view(torch.bfloat16)
        self.v0 = torch.from_numpy(v0.view(np.int16)).cuda().view(torch.bfloat16)
        ks, vs = synth.decode_steps(0, w["steps"], B, H)
        self.ks = torch.from_numpy(ks.view(np.int16)).cuda().view(torch.bfloat16)
        self.vs = torch.from_numpy(vs.view(np.int16)).cuda().view(torch.bfloat16)
        meth, extra = _scorer_kwargs(self.method, H, torch)
        self.cache = binding.EvictCache(meth, B, H, budget=w["budget"], n_sink=w["n_sink"],
                                        recent=w["recent"], max_block=w["prefill"], stream=stream.cuda_stream,
                                        **extra)
        self.handle = self.cache.handle
        self.handles = [self.handle]
        self.cache.update_and_fetch(self.k0, self.v0)
        self.i = 0
        self.tokens_per_step = B * H * (w["budget"] + 1)
        self.calls_per_step = 1
        self.rows_per_call = w["budget"] + 1

    def step(self):
        s = self.i % self.w["steps"]
        self.binding.evict_update_and_fetch(self.handle, self.ks[s].data_ptr(), self.vs[s].data_ptr(), None, 1)
        self.i += 1

    def setup_e2e(self):
        t = self.torch
        self.kh = self.ks.view(t.int16).cpu().pin_memory()
        self.vh = self.vs.view(t.int16).cpu().pin_memory()
        self.out_h = t.empty((self.w["batch"] * self.w["heads"] * self.w["budget"],), dtype=t.int32).pin_memory()
        self.h2d = 2 * self.kh[0].numel() * 2
        self.d2h = self.out_h.numel() * 4

    def step_e2e(self):
        s = self.i % self.w["steps"]
        view = self.binding.evict_update_and_fetch_host(self.handle, self.kh[s].data_ptr(), self.vh[s].data_ptr(),
                                                        None, 1)
        self.i += 1
        pos = self.binding.view_tensors(view, self.w["batch"], self.w["heads"], "bf16")[2]
        self.out_h.copy_(pos.reshape(-1), non_blocking=True)

    def stream_leg(self, stream, per_graph=64):
        """The whole decode stream (every input step, in order, from the state after the prefill)
        captured as CUDA graphs of `per_graph` single-token steps and replayed back to back; the
        steady state keeps the kept cache in L2. Returns the per-step time over the stream."""
        torch, b = self.torch, self.binding
        steps = self.w["steps"]
        B, H = self.w["batch"], self.w["heads"]
        meth, extra = _scorer_kwargs(self.method, H, torch)
        cache = b.EvictCache(meth, B, H, budget=self.w["budget"], n_sink=self.w["n_sink"], recent=self.w["recent"],
                             max_block=self.w["prefill"], stream=stream.cuda_stream, **extra)
        with torch.cuda.stream(stream):
            cache.update_and_fetch(self.k0, self.v0)
            snap = [t.contiguous().clone() for t in cache.view()]
        off = b.evict_stats(cache.handle)["offset"]
        stream.synchronize()
        graphs = []
        launches0 = b.evict_launch_count()
        for g0 in range(0, steps, per_graph):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for s in range(g0, min(g0 + per_graph, steps)):
                    b.evict_update_and_fetch(cache.handle, self.ks[s].data_ptr(), self.vs[s].data_ptr(), None, 1)
            graphs.append(g)
        launches = b.evict_launch_count() - launches0
        times = []
        for rep in range(2):                   # the first pass warms up
            with torch.cuda.stream(stream):
                b.evict_set_state(cache.handle, snap[0].data_ptr(), snap[1].data_ptr(), snap[2].data_ptr(),
                                  snap[3].data_ptr(), snap[0].shape[2], off)
                a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for g in graphs:
                    g.replay()
                e.record(stream)
            stream.synchronize()
            times.append(a.elapsed_time(e))
        b.evict_sync(cache.handle)
        cache.close()
        ms = times[-1] / steps
        return {"steps": steps, "steps_per_graph": per_graph, "gpu_launches_per_step": launches / steps,
                "ms_per_step": round(ms, 5), "value": round(self.tokens_per_step / (ms / 1e3), 1), "unit": UNIT,
                "l2": "steady state: the 67 MB kept cache stays in L2 between steps"}


class LongContextRun:
    """Long-context chunked prefill through one scorer: one step = 16 blocks of 8192 tokens
    through one cache (reset first). `inputs` are shared device blocks when several scorers run."""

    l2_note = "inputs larger than L2 (2.1 GB of blocks per scorer per step)"

    def __init__(self, w, torch, binding, stream, method, inputs=None, first_row=0):
        self.w, self.torch, self.binding = w, torch, binding
        self.method = method
        B, H = w["batch"], w["heads"]
        self.inputs = inputs or LongContextInputs(w, torch, first_row)
        meth, extra = _scorer_kwargs(method, H, torch)
        if method == "qfilters":
            q = synth.long_context_queries(H)
            qd = torch.from_numpy(q.view(np.int16)).cuda()
            f = torch.empty((H, 128), dtype=torch.float32, device="cuda")
            binding.evict_qfilters_calibrate(qd.data_ptr(), binding.EVICT_BF16, H, q.shape[1], 128, H,
                                             f.data_ptr(), stream.cuda_stream)
            extra["filters"] = f
        # the fallback freezes once per sequence, on the first block (>= 128 keys)
        self.freeze_rows = w["block"] if method == "qfilters_fallback" else 0
        self.cache = binding.EvictCache(meth, B, H, budget=w["budget"], n_sink=w["n_sink"],
                                        recent=w["recent"], max_block=w["block"], stream=stream.cuda_stream, **extra)
        self.handle = self.cache.handle
        self.handles = [self.handle]
        kk = [min(blk * w["block"], w["budget"]) for blk in range(w["blocks"])]
        m = w["block"]
        self.logits = B * H * sum(m * k + m * (m + 1) // 2 for k in kk) if method in ("curdkv", "h2o") else None
        self.tokens_per_step = B * H * sum(k + m for k in kk)
        self.calls_per_step = w["blocks"]
        self.rows_per_call = self.tokens_per_step / (B * H * w["blocks"])

    def step(self):
        self.binding.evict_reset(self.handle)
        for k, v in zip(self.inputs.k, self.inputs.v):
            self.binding.evict_update_and_fetch(self.handle, k.data_ptr(), v.data_ptr(), None, self.w["block"])

    def setup_e2e(self):
        self.inputs.pin()
        self.out = _HostCache(self.torch, self.w["batch"], self.w["heads"], self.w["budget"])
        self.h2d = self.inputs.host_bytes
        self.d2h = self.out.nbytes

    def step_e2e(self):
        self.binding.evict_reset(self.handle)
        view = None
        for kh, vh in zip(self.inputs.kh, self.inputs.vh):
            view = self.binding.evict_update_and_fetch_host(self.handle, kh.data_ptr(), vh.data_ptr(), None,
                                                            self.w["block"])
        self.out.fetch(self.binding, view, self.w["batch"], self.w["heads"])


class LongContextInputs:
    """The 16 device blocks of the stream (and, for the end-to-end leg, pinned host copies)."""

    def __init__(self, w, torch, first_row=0):
        self.torch = torch
        self.k, self.v = [], []
        for blk in range(w["blocks"]):
            k, v = synth.long_context_block(blk, w["batch"], w["heads"], w["block"], first_row=first_row)
            self.k.append(torch.from_numpy(k.view(np.int16)).cuda().view(torch.bfloat16))
            self.v.append(torch.from_numpy(v.view(np.int16)).cuda().view(torch.bfloat16))
        self.kh = self.vh = None
        self.host_bytes = sum(x.numel() * 2 for x in self.k) * 2

    def pin(self):
        if self.kh is None:
            t = self.torch
            self.kh = [x.view(t.int16).cpu().pin_memory() for x in self.k]
            self.vh = [x.view(t.int16).cpu().pin_memory() for x in self.v]


class LongContextSuite:
    """Every scorer of the long-context workload over the same 16 blocks: one step = the stream
    through each scorer's cache in turn."""

    l2_note = LongContextRun.l2_note

    def __init__(self, w, torch, binding, stream, first_row=0):
        self.w = w
        self.inputs = LongContextInputs(w, torch, first_row)
        self.runs = [LongContextRun(w, torch, binding, stream, s, self.inputs) for s in w["scorers"]]
        self.handles = [h for r in self.runs for h in r.handles]
        self.tokens_per_step = sum(r.tokens_per_step for r in self.runs)
        self.calls_per_step = sum(r.calls_per_step for r in self.runs)

    def step(self):
        for r in self.runs:
            r.step()

    def setup_e2e(self):
        for r in self.runs:
            r.setup_e2e()
        self.h2d = sum(r.h2d for r in self.runs)
        self.d2h = sum(r.d2h for r in self.runs)

    def step_e2e(self):
        for r in self.runs:
            r.step_e2e()


class CurdkvPlantedRun:
    """CurDKV planted geometry: a 16384-row cache (reloaded before every step, outside the timed
    events, then the L2 flushed) absorbs a 512-token block whose keys are the proxy queries;
    budget 2048."""

    l2_note = "state reloaded and L2 flushed (512 MB write) before every timed step, outside the events"
    flush_l2 = True

    def __init__(self, w, torch, binding, stream):
        self.w, self.torch, self.binding = w, torch, binding
        B, H, S0, m = w["batch"], w["heads"], w["existing"], w["incoming"]
        self.method = w["method"]
        p = synth.curdkv_planted(B, H, existing=S0, incoming=m)
        dev = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.bfloat16)
        self.k0, self.v0 = dev(p["k"][:, :, :S0]), dev(p["v"][:, :, :S0])
        self.kn, self.vn = dev(p["k"][:, :, S0:]), dev(p["v"][:, :, S0:])
        self.pos0 = torch.arange(S0, dtype=torch.int32, device="cuda").expand(B, H, S0).contiguous()
        self.score0 = torch.zeros((B, H, S0), dtype=torch.float32, device="cuda")
        self.cls = p["cls"]
        self.cache = binding.EvictCache(w["method"], B, H, budget=w["budget"], n_sink=w["n_sink"],
                                        recent=w["recent"], max_block=m, max_kept=S0, rank_cap=w["rank_cap"],
                                        stream=stream.cuda_stream, per_token=w.get("per_token", False))
        self.handle = self.cache.handle
        self.handles = [self.handle]
        self.tokens_per_step = B * H * (S0 + m)
        self.calls_per_step = 1
        self.rows_per_call = S0 + m
        self.logits = B * H * (m * S0 + m * (m + 1) // 2)
        if w.get("per_token"):
            # m single-token steps: the first sees every existing row, the rest a full cache of
            # budget + 1 rows; the per-launch work of the attention kernels varies, so the kernel
            # table carries times only
            self.logits = None

    def reload(self):
        self.binding.evict_set_state(self.handle, self.k0.data_ptr(), self.v0.data_ptr(), self.pos0.data_ptr(),
                                     self.score0.data_ptr(), self.w["existing"], self.w["existing"])

    def class2_retention(self):
        """Share of class-2 (negligible-value) tokens among the kept non-sink rows after the last step
        (the pages' CurDKV-vs-H2O comparison)."""
        pos = self.cache.view()[2].cpu().numpy()
        cls = np.take_along_axis(self.cls, pos.astype(np.int64), axis=2)[:, :, self.w["n_sink"]:]
        return round(float(np.mean(cls == 2)), 4)

    def step(self):
        self.binding.evict_update_and_fetch(self.handle, self.kn.data_ptr(), self.vn.data_ptr(), None,
                                            self.w["incoming"])

    def setup_e2e(self):
        self.kh = self.kn.view(self.torch.int16).cpu().pin_memory()
        self.vh = self.vn.view(self.torch.int16).cpu().pin_memory()
        self.out = _HostCache(self.torch, self.w["batch"], self.w["heads"], self.w["budget"])
        self.h2d, self.d2h = 2 * self.kh.numel() * 2, self.out.nbytes

    def step_e2e(self):
        view = self.binding.evict_update_and_fetch_host(self.handle, self.kh.data_ptr(), self.vh.data_ptr(), None,
                                                        self.w["incoming"])
        self.out.fetch(self.binding, view, self.w["batch"], self.w["heads"])


class KnormSingleRun:
    l2_note = "working set (1 MB) L2-resident: latency-bound, report absolute time"

    def __init__(self, w, torch, binding, stream):
        self.w, self.torch, self.binding = w, torch, binding
        self.method = "knorm"
        k, v = synth.knorm_single_sequence(w["seq"])
        self.k, self.v = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
        self.cache = binding.EvictCache("knorm", 1, 1, budget=w["budget"], n_sink=w["n_sink"], recent=0,
                                        max_block=w["seq"], dtype="fp32", stream=stream.cuda_stream)
        self.handle = self.cache.handle
        self.handles = [self.handle]
        self.tokens_per_step = w["seq"]
        self.calls_per_step = 1
        self.rows_per_call = w["seq"]

    def step(self):
        self.binding.evict_reset(self.handle)
        self.binding.evict_update_and_fetch(self.handle, self.k.data_ptr(), self.v.data_ptr(), None, self.w["seq"])

    def setup_e2e(self):
        t = self.torch
        self.kh, self.vh = self.k.cpu().pin_memory(), self.v.cpu().pin_memory()
        self.out_h = t.empty((self.w["budget"],), dtype=t.int32).pin_memory()
        self.h2d, self.d2h = 2 * self.kh.numel() * 4, self.out_h.numel() * 4

    def step_e2e(self):
        self.binding.evict_reset(self.handle)
        view = self.binding.evict_update_and_fetch_host(self.handle, self.kh.data_ptr(), self.vh.data_ptr(), None,
                                                        self.w["seq"])
        pos = self.binding.view_tensors(view, 1, 1, "fp32")[2]
        self.out_h.copy_(pos.reshape(-1), non_blocking=True)


RUNS = {"qfilters_stack": StackRun, "decode": DecodeRun, "knorm_single": KnormSingleRun,
        "curdkv_planted": CurdkvPlantedRun}


def make_run(workload, w, torch, binding, stream, first_row=0):
    if workload == "long_context":
        if len(w["scorers"]) == 1:
            return LongContextRun(w, torch, binding, stream, w["scorers"][0], first_row=first_row)
        return LongContextSuite(w, torch, binding, stream, first_row)
    return RUNS[workload](w, torch, binding, stream)


# ----------------------------------------------------------------------------
# timing
# ----------------------------------------------------------------------------
class Timer:
    """CUDA events on the launching stream around each step; barriers (and a device synchronize)
    on both sides of a region. Anything `before` does (a state reload, an L2 flush) runs outside
    the events."""

    def __init__(self, torch, stream, barrier):
        self.torch, self.stream, self.barrier = torch, stream, barrier

    def region(self, step, steps, before=None):
        torch = self.torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        self.barrier()
        with torch.cuda.stream(self.stream):
            for a, b in evs:
                if before:
                    before()
                a.record(self.stream)
                step()
                b.record(self.stream)
        self.barrier()
        return sum(a.elapsed_time(b) for a, b in evs)


def _before(run, flush):
    reload = getattr(run, "reload", None)
    do_flush = flush is not None and getattr(run, "flush_l2", False)
    if not reload and not do_flush:
        return None

    def f():
        if reload:
            reload()
        if do_flush:
            flush.fill_(1)
    return f


def kernel_table(run, binding, timer, steps, before):
    """Per-kernel launches and times over a second region in which every launch of the run's
    handles is bracketed by events (those events serialise the launches: the region is slower,
    and its time is reported as profiled_ms_per_step)."""
    for h in run.handles[:1] if isinstance(run, StackRun) else run.handles:
        binding.evict_set_profiling(h, True)
    ms = timer.region(run.step, steps, before)
    times = {}
    for h in run.handles[:1] if isinstance(run, StackRun) else run.handles:
        for k, (n, t) in binding.evict_kernel_times(h).items():
            a, b = times.get(k, (0, 0.0))
            times[k] = (a + n, b + t)
        binding.evict_set_profiling(h, False)
    return ms, times


def roofline_of(run, ktimes, work, steps, ms_per_step, peaks, peak_kind, workload):
    """The dominant kernel against its roofline, every kernel's rate, and the whole path against
    its binding resource."""
    kernels = {}
    tot = sum(t for _, t in ktimes.values())
    for k, (n, t) in ktimes.items():
        sec = t / n / 1e3
        kernels[k] = {"launches": n, "avg_us": round(t / n * 1e3, 2), "share": round(t / tot, 4) if tot else None}
        wk = work.get(k, {})
        if "bytes" in wk:
            kernels[k]["algorithmic_bytes_per_launch"] = wk["bytes"]
            kernels[k]["achieved_gbs"] = round(wk["bytes"] / sec / 1e9, 1)
        if "flops" in wk:
            kernels[k]["algorithmic_flops_per_launch"] = wk["flops"]
            kernels[k]["achieved_tflops"] = round(wk["flops"] / sec / 1e12, 2)
        if "exps" in wk:
            kernels[k]["exp2_per_s"] = round(wk["exps"] / sec, 1)
    roof = None
    if ktimes:
        top = max(ktimes, key=lambda k: ktimes[k][1])
        n_launch, tot_ms = ktimes[top]
        per_launch_ms = tot_ms / n_launch
        wk = work.get(top, {})
        if top == "qfilters_freeze":
            achieved = wk["flops"] / (per_launch_ms / 1e3) / 1e12
            roof = {"kernel": top, "bound": "alu", "achieved": round(achieved, 2), "peak": round(FP32_FMA_TFLOPS, 1),
                    "unit": "TFLOP/s", "frac": round(achieved / FP32_FMA_TFLOPS, 4),
                    "algorithmic_flops_per_launch": wk["flops"]}
        elif top in ("curdkv_lse", "curdkv_colsum", "curdkv_gram") and "flops" in wk:
            achieved = wk["flops"] / (per_launch_ms / 1e3) / 1e12
            roof = {"kernel": top, "bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                    "algorithmic_flops_per_launch": wk["flops"]}
        elif "bytes" in wk:
            achieved = wk["bytes"] / (per_launch_ms / 1e3) / 1e9
            roof = {"kernel": top, "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "algorithmic_bytes_per_launch": wk["bytes"]}
        else:
            roof = {"kernel": top, "bound": "latency", "achieved": None, "peak": None, "unit": None, "frac": None}
        roof["peak_kind"] = peak_kind
        roof["traffic"] = _ncu_traffic(top, workload)
        roof["avg_launch_us"] = round(per_launch_ms * 1e3, 2)
    return roof, kernels, path_roofline(run, ktimes, work, steps, ms_per_step, peaks)


def path_roofline(run, ktimes, work, steps, ms_per_step, peaks):
    """The whole step against its binding resource. Byte-bound paths (KNorm, Q-Filters): every
    kernel's algorithmic bytes per step over the uninstrumented step time, against HBM. Attention
    scorers (CurDKV, H2O): the step's ideal time is the larger of its algorithmic bytes at the HBM
    peak and one pass of the proxy-attention products (2*D flops per logit) at the bf16 tensor
    peak; frac = ideal / measured."""
    if not ktimes:
        return None
    per_step = sum(work[k]["bytes"] * n / steps for k, (n, _) in ktimes.items() if "bytes" in work.get(k, {}))
    logits = getattr(run, "logits", None)
    if getattr(run, "method", None) in ("curdkv", "h2o") and logits:
        # bytes the attention scorers must move besides the byte-bound kernels: K read for every
        # row and, for CurDKV, V read for every row (Gram) with the cumulative score read/written
        units_rows = run.tokens_per_step
        extra = units_rows * (128 * 2 + (128 * 2 + 8 if run.method == "curdkv" else 8))
        hbm_us = (per_step + extra) / (peaks["hbm_gbs"] * 1e9) * 1e6
        flops = 2 * 128 * logits
        tc_us = flops / (peaks["bf16_tflops"] * 1e12) * 1e6
        ideal = max(hbm_us, tc_us)
        return {"bound": "tensor" if tc_us >= hbm_us else "hbm", "ideal_us": round(ideal, 2),
                "hbm_bytes_per_step": int(per_step + extra), "tensor_flops_per_step": int(flops),
                "measured_us": round(ms_per_step * 1e3, 2), "frac": round(ideal / (ms_per_step * 1e3), 4)}
    if not all("bytes" in work.get(k, {}) for k in ktimes):
        return None
    gbs = per_step / (ms_per_step / 1e3) / 1e9
    return {"bound": "hbm", "algorithmic_bytes_per_step": int(per_step), "achieved": round(gbs, 1), "unit": "GB/s",
            "peak": peaks["hbm_gbs"], "frac": round(gbs / peaks["hbm_gbs"], 4)}


def measure(run, workload, args, torch, binding, timer, flush, world, clocks=True, local=0, kernels=True):
    """Warm-up, the timed step region (value), the per-kernel region (roofline; skipped with
    kernels=False), the end-to-end region through the host-buffer entry point."""
    before = _before(run, flush)
    for _ in range(args.warmup):
        if before:
            before()
        run.step()
    clk = ClockSampler(local) if clocks else None
    if clk:
        clk.__enter__()
    launches0 = binding.evict_launch_count()
    ms = timer.region(run.step, args.steps, before)
    launches = binding.evict_launch_count() - launches0
    profiled_ms, ktimes = kernel_table(run, binding, timer, args.steps, before) if kernels else (None, {})
    if clk:
        clk.__exit__(None, None, None)
    for h in run.handles:
        binding.evict_sync(h)
    ms_per_step = max_over_ranks(ms) / args.steps
    peaks, peak_kind = _peaks()
    roof, ktab, path = None, {}, None
    if kernels:
        work = algorithmic_work(run, binding)
        roof, ktab, path = roofline_of(run, ktimes, work, args.steps, ms_per_step, peaks, peak_kind, workload)
    # end-to-end through the host-buffer entry point (copies in both directions inside the region)
    run.setup_e2e()
    for _ in range(min(args.warmup, 3)):
        if before:
            before()
        run.step_e2e()
    e2e_ms = max_over_ranks(timer.region(run.step_e2e, args.steps, before)) / args.steps
    rec = {
        "value": round(job_throughput(world, run.tokens_per_step, ms_per_step), 1), "unit": UNIT,
        "ms_per_step": round(ms_per_step, 5), "tokens_per_step": run.tokens_per_step,
        "calls_per_step": run.calls_per_step, "gpu_launches": int(launches),
        "l2": run.l2_note,
        "e2e": {"value": round(job_throughput(world, run.tokens_per_step, e2e_ms), 1), "unit": UNIT,
                "h2d_bytes_per_step": run.h2d, "d2h_bytes_per_step": run.d2h, "ms_per_step": round(e2e_ms, 4)},
        "roofline": roof, "kernels": ktab, "path_roofline": path,
        "profiled_ms_per_step": round(max_over_ranks(profiled_ms) / args.steps, 5) if kernels else None,
    }
    if clk:
        rec["clocks"] = clk.summary()
    return rec


def l2_copy_probe(torch, stream):
    """Copy bandwidth of a 2 x 24 MB working set that stays in L2 (read + write bytes, best of 20)."""
    a = torch.empty(24 << 20, dtype=torch.uint8, device="cuda")
    b = torch.empty_like(a)
    best = None
    with torch.cuda.stream(stream):
        for i in range(25):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            b.copy_(a)
            e1.record(stream)
            stream.synchronize()
            if i >= 5:
                t = e0.elapsed_time(e1)
                best = t if best is None else min(best, t)
    return round(2 * a.numel() / (best / 1e3) / 1e9, 1)


# ----------------------------------------------------------------------------
# algorithmic work per launch
# ----------------------------------------------------------------------------
def algorithmic_work(run, binding):
    """Work each kernel must do per launch (one launch covers every layer of a call).

    Bytes (HBM-bound kernels):
    score    : read each incoming key once, write its fp32 score.
    select   : read the n scores of every (b, h), write the budget-long source
               map, reset the chunk flags, write the 8-byte metadata.
    compact  : per incoming survivor read K and V, write K, V, position and
               score, read its score and map entry (4*D*e + 16 bytes); per kept
               row whose slot changes read and write K, V, position and score
               and read its map entry (4*D*e + 20 bytes). Rows counted from
               the last call (evict_compaction_rows).
    curdkv_leverage : read every row's value once, its attention sum, and
               read/write its score (D*2 + 12 bytes per row).
    Flops / exponentials (CurDKV attention passes): 2*D per valid logit and
    one exponential per valid logit; L = sum over (b, h) of m*k + m(m+1)/2.
    curdkv_attn_small: short blocks (m <= 8) in one kernel: every key row read
               once (D*2 bytes) and its column sum written (4 bytes); H2O adds
               the increment written and the score read and written (12 bytes).
               Rows: the call's n, or budget + 1 per launch in the per-token mode.
    curdkv_gram: 2*D*D flops per row (the bf16 hi + lo split doubles the
               tensor-core work; the algorithmic count is one product).
    evict1   : the fused single-eviction step: incoming keys, every row's
               score, and the rows behind the evicted one moved down
               (K, V, position and score read and written).
    qfilters_freeze : the key-SVD fallback's one-time freeze: every key present
               read once, 2*D*D fp32 flops per key for the centred Gram (bound
               by the fp32 FMA pipes, "alu").
    A multi-block step (the long-context stream) reports averages per launch:
    its launches see a growing kept prefix, so every figure is the step's
    total over its launches.
    """
    w = run.w
    e = 2 if w["dtype"] == "bf16" else 4
    units = w["layers"] * w["batch"] * w["heads"]
    m = w.get("seq", w.get("block", w.get("incoming", 1)))
    if isinstance(run, DecodeRun):
        m = 1
    n = run.rows_per_call
    method = getattr(run, "method", w.get("method"))
    out = {"score": {"bytes": units * m * (128 * e + 4)}}
    old, new = 0, 0
    for h in run.handles:
        a, b = binding.evict_compaction_rows(h)
        old, new = old + a, new + b
    out["compact"] = {"bytes": new * (4 * 128 * e + 16) + old * (4 * 128 * e + 20)}
    # fused single eviction: read the incoming keys and every row's score, move
    # the rows behind the evicted one (K, V, position and score read and written)
    out["evict1"] = {"bytes": units * m * 128 * e + units * 4 * n + new * (4 * 128 * e + 12) + old * (4 * 128 * e + 16)}
    flag_stride = -(-w["budget"] // (64 if e == 2 else 32)) + 1      # chunk flags + the chunk counter
    out["select"] = {"bytes": int(units * (4 * n + 4 * w["budget"] + 4 * flag_stride + 8))}
    if getattr(run, "freeze_rows", 0):
        # key-SVD freeze: read the keys present once; the centred Gram is 2*D*D flops per key
        out["qfilters_freeze"] = {"bytes": units * run.freeze_rows * 128 * e,
                                  "flops": units * run.freeze_rows * 2 * 128 * 128}
    # short blocks (m <= 8): every key row read once and its column sum written; H2O also writes
    # the increment and reads and writes the score. A per-token launch sees the budget's rows
    # plus its token.
    n_small = w["budget"] + 1 if w.get("per_token") else n
    per_row = 128 * 2 + (16 if method == "h2o" else 4)
    out["curdkv_attn_small"] = {"bytes": int(units * n_small * per_row)}
    logits = getattr(run, "logits", None)
    if logits:
        calls = run.calls_per_step
        for k in ("curdkv_lse", "curdkv_colsum"):
            out[k] = {"flops": 2 * 128 * logits / calls, "exps": logits / calls}
        out["curdkv_gram"] = {"flops": units * n * 2 * 128 * 128}
        out["h2o_mass"] = {"bytes": int(units * n * 16)}       # read the sum, write it, read/write the score
        out["curdkv_leverage"] = {"bytes": int(units * n * (128 * 2 + 12))}
    if w.get("blocks"):
        # the long-context stream: the compaction figures above are the last call's; average the
        # kept rows moved and the survivors written over the step's blocks instead (the first
        # block has no kept rows, every later one a full kept prefix of budget rows)
        B, H = w["batch"], w["heads"]
        blocks = w["blocks"]
        first_new = min(w["budget"], w["block"])
        per_unit = first_new * (4 * 128 * e + 16) + (blocks - 1) * (new * (4 * 128 * e + 16) + old * (4 * 128 * e + 20)) / (B * H)
        out["compact"] = {"bytes": int(B * H * per_unit / blocks)}
        n_first = w["block"]
        n_rest = min(w["budget"], w["block"]) + w["block"]
        n_avg = (n_first + (blocks - 1) * n_rest) / blocks
        out["select"] = {"bytes": int(units * (4 * n_avg + 4 * w["budget"] + 4 * flag_stride + 8))}
        if logits:
            out["curdkv_gram"] = {"flops": int(units * n_avg * 2 * 128 * 128)}
            out["curdkv_leverage"] = {"bytes": int(units * n_avg * (128 * 2 + 12))}
            out["h2o_mass"] = {"bytes": int(units * n_avg * 16)}
    return out


# ----------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ----------------------------------------------------------------------------
def _oracle_long_context(w, method, budget_s):
    """One (b, h) unit of the long-context stream through the oracle for as many blocks as fit
    in budget_s; returns (tokens, seconds, blocks done)."""
    from oracle import calibrate as ocal
    from oracle.cache import OracleCache
    meth, kw = _scorer_kwargs(method, w["heads"])
    if method == "qfilters":
        kw["filters"] = ocal.calibrate(synth.long_context_queries(w["heads"]), w["heads"])[:1].astype(np.float32)
    c = OracleCache(meth, 1, 1, budget=w["budget"], n_sink=w["n_sink"], recent=w["recent"], **kw)
    tokens, secs, done = 0, 0.0, 0
    for blk in range(w["blocks"]):
        k, v = synth.long_context_block(blk, 1, w["heads"], w["block"])
        t1 = time.perf_counter()
        n = c.n_kept + w["block"]
        c.update_and_fetch(k[:1, :1], v[:1, :1])
        secs += time.perf_counter() - t1
        tokens += n
        done += 1
        if secs > budget_s:
            break
    return tokens, secs, done


def _oracle_sample(workload, budget_s=10.0):
    """Run the oracle on a bounded sample of the workload; returns (tokens, seconds, description).
    For several scorers the seconds are the whole step's estimated oracle time: each scorer's
    sampled seconds per token times the tokens it handles in one step."""
    from oracle import calibrate as ocal
    from oracle.cache import OracleCache
    w = WORKLOADS[workload]
    tokens, secs, done = 0, 0.0, 0
    if workload == "long_context":
        # the step handles the same tokens with every scorer: the composite rate is the number of
        # scorers over the sum of their seconds per token; the tokens returned are what that rate
        # covers in the seconds actually spent
        parts, secs, per_token = [], 0.0, 0.0
        for method in w["scorers"]:
            t, s, done = _oracle_long_context(w, method, budget_s / len(w["scorers"]))
            parts.append(f"{method}: {done} block(s) of one (b, h) unit")
            secs += s
            per_token += s / t
        rate = len(w["scorers"]) / per_token
        return rate * secs, secs, "; ".join(parts) + " (composite rate: scorers / sum of seconds per token)"
    if workload == "qfilters_stack":
        t0 = time.perf_counter()
        for layer in range(w["layers"]):
            d = synth.qfilters_layer(layer, seq_len=w["seq"])
            f = ocal.calibrate(d["queries"], w["heads"]).astype(np.float32)
            c = OracleCache("qfilters", w["batch"], w["heads"], budget=w["budget"], n_sink=w["n_sink"],
                            recent=w["recent"], filters=f)
            t2 = time.perf_counter()                       # calibration is off the per-step path
            c.update_and_fetch(d["k"], d["v"])
            secs += time.perf_counter() - t2
            tokens += w["batch"] * w["heads"] * w["seq"]
            done += 1
            if time.perf_counter() - t0 > budget_s:
                break
        return tokens, secs, f"{done} of {w['layers']} layers (one prefill update each; calibration untimed)"
    if workload == "decode":
        k0, v0 = synth.decode_prefill(w["batch"], w["heads"], w["prefill"])
        meth, kw = _scorer_kwargs(w["method"], w["heads"])
        c = OracleCache(meth, w["batch"], w["heads"], budget=w["budget"], n_sink=w["n_sink"],
                        recent=w["recent"], **kw)
        c.update_and_fetch(k0, v0)
        ks, vs = synth.decode_steps(0, 64, w["batch"], w["heads"])
        t0 = time.perf_counter()
        for s in range(64):
            c.update_and_fetch(ks[s], vs[s])
            tokens += w["batch"] * w["heads"] * (w["budget"] + 1)
            done += 1
            if time.perf_counter() - t0 > budget_s:
                break
        return tokens, time.perf_counter() - t0, f"{done} decode steps after the 2048-token prefill"
    if workload == "curdkv_planted":
        S0, m = w["existing"], w["incoming"]
        p = synth.curdkv_planted(w["batch"], w["heads"], existing=S0, incoming=m)
        t0 = time.perf_counter()
        for b in range(w["batch"]):
            for h in range(w["heads"]):
                c = OracleCache(w["method"], 1, 1, budget=w["budget"], n_sink=w["n_sink"], rank_cap=w["rank_cap"],
                                per_token=w.get("per_token", False))
                c.set_state(p["k"][b:b + 1, h:h + 1, :S0], p["v"][b:b + 1, h:h + 1, :S0],
                            np.arange(S0, dtype=np.int32)[None, None], np.zeros((1, 1, S0)), S0)
                t1 = time.perf_counter()
                c.update_and_fetch(p["k"][b:b + 1, h:h + 1, S0:], p["v"][b:b + 1, h:h + 1, S0:])
                secs += time.perf_counter() - t1
                tokens += S0 + m
                done += 1
                if time.perf_counter() - t0 > budget_s:
                    return tokens, secs, f"{done} of {w['batch'] * w['heads']} (b, h) units (one update each)"
        return tokens, secs, f"{done} (b, h) units (one update each)"
    k, v = synth.knorm_single_sequence(w["seq"])
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < min(budget_s, 2.0):
        c = OracleCache("knorm", 1, 1, budget=w["budget"], n_sink=w["n_sink"], dtype="fp32")
        c.update_and_fetch(k, v)
        tokens += w["seq"]
        done += 1
    return tokens, time.perf_counter() - t0, f"{done} one-block prefills"


def _oracle_threads():
    """Threads the oracle's numpy can use: BLAS (the CurDKV SVDs and matrix products) runs on the
    process's cores; everything else is single-threaded numpy."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(workload, budget_s=10.0):
    tokens, secs, sample = _oracle_sample(workload, budget_s)
    return {"value": round(tokens / secs, 1), "unit": UNIT, "cores": _oracle_threads(), "kind": "oracle",
            "sample": sample + "; numpy (BLAS on the process's cores for the matrix products and SVDs, "
                               "single-threaded elsewhere)"}


# ----------------------------------------------------------------------------
# arms
# ----------------------------------------------------------------------------
def _workload_line(name, w, rec, world, extra=None):
    cfg = {"workload": name, **{k: (list(v) if isinstance(v, tuple) else v) for k, v in w.items()},
           "storage": w["dtype"], "tokens_per_step": rec["tokens_per_step"], "calls_per_step": rec["calls_per_step"],
           "l2": rec["l2"]}
    if extra:
        cfg.update(extra)
    return cfg


def run_ours(args):
    import torch
    import torch.distributed as dist
    world, rank, local = _dist()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    from kv_cache_token_bf16_gb300 import binding
    stream = torch.cuda.Stream()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    timer = Timer(torch, stream, barrier)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
    w = WORKLOADS[args.workload]
    first_row = 0
    if args.workload == "long_context":
        first_row, _ = rank_rows(rank, world, w["batch"])
    with torch.cuda.stream(stream):
        run = make_run(args.workload, w, torch, binding, stream, first_row)
    torch.cuda.synchronize()
    suite = isinstance(run, LongContextSuite)
    rec = measure(run, args.workload, args, torch, binding, timer, flush, world, local=local, kernels=not suite)

    extra = {"parallelism": (f"batch-row shards x{world} (rank r owns rows {w['batch']}r..{w['batch']}r+"
                             f"{w['batch'] - 1} of {w['batch'] * world} sequences)")
             if args.workload == "long_context" else f"replica-per-gpu x{world}"}
    line = {
        "metric": METRIC, "value": rec["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": rec["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded generators standing in for real-model activations)",
        "config": _workload_line(args.workload, w, rec, world, extra),
        "e2e": dict(rec["e2e"], readback="the kept caches (K, V, positions) return to pinned host memory "
                                         "inside the timed region" if not isinstance(run, (DecodeRun, KnormSingleRun))
                    else "kept positions only"),
        "gpu_launches": rec["gpu_launches"], "roofline": rec["roofline"], "kernels": rec["kernels"],
        "path_roofline": rec["path_roofline"], "profiled_ms_per_step": rec["profiled_ms_per_step"],
        "kernel_timing": "per-kernel CUDA events on the launching stream over a second timed region of the same "
                         "K steps (profiled_ms_per_step; per scorer for the long-context suite); the step time "
                         "comes from the first region, which has events around each step only",
        "clocks": rec.get("clocks"),
    }
    if isinstance(run, LongContextSuite):
        # every scorer's own stream: its step time, rooflines and kernels
        line["scorers"] = {}
        for sub in run.runs:
            r = measure(sub, args.workload, args, torch, binding, timer, flush, world, clocks=False, local=local)
            line["scorers"][sub.method] = {k: r[k] for k in ("value", "ms_per_step", "tokens_per_step", "roofline",
                                                             "path_roofline", "kernels", "e2e",
                                                             "profiled_ms_per_step")}
        # the headline roofline: the step's dominant kernel (most time over all scorers)
        tops = [(s["roofline"]["avg_launch_us"] * s["kernels"][s["roofline"]["kernel"]]["launches"], name)
                for name, s in line["scorers"].items() if s["roofline"]]
        if tops:
            top = max(tops)[1]
            line["roofline"] = dict(line["scorers"][top]["roofline"], scorer=top)
        ideal = 0.0
        for name, s in line["scorers"].items():
            p = s["path_roofline"]
            if p and "ideal_us" in p:
                ideal += p["ideal_us"]
            elif p:
                ideal += p["algorithmic_bytes_per_step"] / (p["peak"] * 1e9) * 1e6
        line["path_roofline"] = {"bound": "per scorer (HBM for KNorm / Q-Filters, tensor for CurDKV)",
                                 "ideal_us": round(ideal, 2), "measured_us": round(rec["ms_per_step"] * 1e3, 2),
                                 "frac": round(ideal / (rec["ms_per_step"] * 1e3), 4)}
        line.pop("kernels")
    if hasattr(run, "calib_ms"):
        line["config"]["calibration_ms_per_layer"] = round(run.calib_ms, 3)
    if hasattr(run, "class2_retention"):
        line["config"]["class2_retention"] = run.class2_retention()
    if isinstance(run, DecodeRun):
        line["stream"] = run.stream_leg(stream)
        line["stream"]["l2_copy_gbs"] = l2_copy_probe(torch, stream)
    del run
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=15.0 if args.workload == HEADLINE else 10.0)
    # the other single-GPU workloads, each with its own record (N=1 only)
    if args.workload == HEADLINE and len(w["scorers"]) > 1 and world == 1 and not args.no_configs:
        line["configs"] = {}
        for name in SUB_CONFIGS:
            sw = WORKLOADS[name]
            with torch.cuda.stream(stream):
                sub = make_run(name, sw, torch, binding, stream)
            torch.cuda.synchronize()
            r = measure(sub, name, args, torch, binding, timer, flush, world, local=local)
            r["config"] = _workload_line(name, sw, r, world)
            r.pop("l2")
            if hasattr(sub, "calib_ms"):
                r["config"]["calibration_ms_per_layer"] = round(sub.calib_ms, 3)
            if hasattr(sub, "class2_retention"):
                r["config"]["class2_retention"] = sub.class2_retention()
            if isinstance(sub, DecodeRun):
                r["stream"] = sub.stream_leg(stream)
                r["stream"]["l2_copy_gbs"] = l2_copy_probe(torch, stream)
            del sub
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
            if not args.no_cpu_baseline:
                r["cpu_baseline"] = cpu_baseline(name, budget_s=8.0)
            line["configs"][name] = r
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    for _ in range(args.warmup):
        _oracle_sample(args.workload, budget_s=1.0)
    tokens_total, secs_total, sample = 0, 0.0, ""
    for _ in range(args.steps):
        t, s, sample = _oracle_sample(args.workload, budget_s=4.0)
        tokens_total += t
        secs_total += s
    value = tokens_total / secs_total
    cfg = {"workload": args.workload, **{k: (list(v) if isinstance(v, tuple) else v) for k, v in w.items()}}
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs_total / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": _oracle_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=HEADLINE)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="headline workload only (no sub-records)")
    ap.add_argument("--method", choices=["knorm", "qfilters", "qfilters_fallback", "curdkv", "h2o"], default=None,
                    help="one scorer for the long_context and decode workloads (qfilters_fallback: Q-Filters "
                         "without calibrated filters, freezing a key-SVD filter after 128 keys) or for "
                         "curdkv_planted (curdkv or h2o)")
    ap.add_argument("--per-token", action="store_true",
                    help="curdkv_planted: absorb the incoming block one token at a time (the pages' loop)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.method:
        ok = {"long_context": {"knorm", "qfilters", "qfilters_fallback", "curdkv", "h2o"},
              "decode": {"knorm", "qfilters", "qfilters_fallback", "curdkv", "h2o"},
              "curdkv_planted": {"curdkv", "h2o"}}
        if args.method not in ok.get(args.workload, ()):
            ap.error("--method: long_context and decode take any scorer, curdkv_planted curdkv / h2o")
        if args.workload == "long_context":
            WORKLOADS["long_context"]["scorers"] = (args.method,)
        else:
            WORKLOADS[args.workload]["method"] = args.method
    if args.per_token:
        if args.workload != "curdkv_planted":
            ap.error("--per-token applies to curdkv_planted")
        WORKLOADS[args.workload]["per_token"] = True
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
