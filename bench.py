"""Throughput of block KV-cache eviction on GB300 through libevict.

Default workload: the Q-Filters calibrated Llama-3.2-3B-like layer stack —
28 layers, 8 KV heads (24 query heads, GQA 3), D=128, bf16, B=1, one
8192-token prefill block per layer, budget 1024, n_sink 4. One step = the
whole hot path over that batch: every layer's cache is reset and absorbs
the block (score, protected top-k, order-preserving compaction). Filters
come from the GPU calibration (uncentered query SVD) run once before timing.

Metric: cache tokens evicted-and-compacted per second (sum over layers and
(b, h) of the rows each call scores and selects from), with the dominant
kernel's achieved HBM GB/s against the measured copy bandwidth.

Other workloads (--workload): decode (B=32, H=8, 2048 prefill then
single-token steps, budget 512, recent 128; also timed with 64 steps
captured in one CUDA graph, the "graph" key), long_context (B=4, H=8,
16 x 8192-token blocks, budget 4096), curdkv_planted (B=H=8, 16384 kept
rows + a 512-token block, budget 2048; reports the class-2 retention),
knorm_single (B=H=1, fp32, S=1024).

Scorer (--method): knorm, qfilters (calibrated filters), qfilters_fallback
(no filters: the key-SVD fallback freezes after 128 keys), curdkv, h2o, for
the decode and long_context workloads; curdkv / h2o for curdkv_planted,
where --per-token absorbs the block one token at a time.

Arms:
  --impl ours       (default) libevict on the GPU
  --impl reference  the CPU oracle (numpy), as it stands, on a bounded sample
                    of the same workload; prints the same JSON line.

Multi-GPU (torchrun): every rank runs its own copy of the workload on its
own GPU (independent units, no collective on the data path); value is the
sum over ranks divided by the slowest rank's time ("scaling": "weak").
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


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------
WORKLOADS = {
    "qfilters_stack": dict(method="qfilters", layers=28, batch=1, heads=8, q_heads=24, seq=8192, budget=1024,
                           n_sink=4, recent=0, dtype="bf16"),
    "decode": dict(method="knorm", layers=1, batch=32, heads=8, prefill=2048, steps=256, budget=512, n_sink=4,
                   recent=128, dtype="bf16"),
    "long_context": dict(method="knorm", layers=1, batch=4, heads=8, block=8192, blocks=16, budget=4096, n_sink=4,
                         recent=0, dtype="bf16"),
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
# GPU arm
# ----------------------------------------------------------------------------
class StackRun:
    """Q-Filters layer stack: 28 caches updated by one grouped call per step."""

    def __init__(self, w, torch, binding, stream):
        self.w, self.torch, self.binding = w, torch, binding
        L, H, S = w["layers"], w["heads"], w["seq"]
        self.k, self.v, self.q = [], [], []
        self.filters = []
        for layer in range(L):
            d = synth.qfilters_layer(layer, n_q_heads=w["q_heads"], n_kv_heads=H, seq_len=S, batch=w["batch"])
            self.k.append(torch.from_numpy(d["k"].view(np.int16)).cuda().view(torch.bfloat16))
            self.v.append(torch.from_numpy(d["v"].view(np.int16)).cuda().view(torch.bfloat16))
            qd = torch.from_numpy(d["queries"].view(np.int16)).cuda()
            f = torch.empty((H, 128), dtype=torch.float32, device="cuda")
            t0 = time.perf_counter()
            binding.evict_qfilters_calibrate(qd.data_ptr(), binding.EVICT_BF16, w["q_heads"], qd.shape[1], 128, H,
                                             f.data_ptr(), stream.cuda_stream)
            self.calib_ms = (time.perf_counter() - t0) * 1e3
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

    def step(self):
        for h in self.handles:
            self.binding.evict_reset(h)
        self.binding.evict_update_and_fetch_group(self.handles, self.kp, self.vp, None, self.w["seq"])

    # end-to-end through the public host-buffer call: inputs start in pinned host memory
    def setup_e2e(self):
        torch = self.torch
        self.kh = [t.view(torch.int16).cpu().pin_memory() for t in self.k]
        self.vh = [t.view(torch.int16).cpu().pin_memory() for t in self.v]
        n = self.w["batch"] * self.w["heads"] * self.w["budget"]
        self.out_h = torch.empty((len(self.caches), n), dtype=torch.int32).pin_memory()
        self.h2d = sum(t.numel() * 2 for t in self.kh) + sum(t.numel() * 2 for t in self.vh)
        self.d2h = self.out_h.numel() * 4

    def step_e2e(self):
        torch = self.torch
        for i, h in enumerate(self.handles):
            self.binding.evict_reset(h)
            view = self.binding.evict_update_and_fetch_host(h, self.kh[i].data_ptr(), self.vh[i].data_ptr(), None,
                                                            self.w["seq"])
            pos = self.binding.view_tensors(view, self.w["batch"], self.w["heads"], "bf16")[2]
            self.out_h[i].copy_(pos.reshape(-1), non_blocking=True)

    def score_bytes_per_launch(self):
        w = self.w
        return w["layers"] * w["batch"] * w["heads"] * w["seq"] * (128 * 2 + 4)


def _scorer_kwargs(w, H, torch=None):
    """Cache arguments of a workload's scorer (w["method"]): the library method name and
    extra keywords. Q-Filters on the decode and long-context streams: seeded unit filters
    (decode) or the GPU calibration on the workload's queries (long context, done by the
    caller); qfilters_fallback: no filters, the key-SVD fallback freezing after 128 keys."""
    meth = w["method"]
    if meth == "qfilters_fallback":
        return "qfilters", {"filters": None, "calib_tokens": 128, "sign": 1}
    if meth == "qfilters":
        f = synth.decode_filters(H)
        return "qfilters", {"filters": torch.from_numpy(f).cuda() if torch else f, "sign": 1}
    if meth == "curdkv":
        return "curdkv", {"rank_cap": 16}
    return meth, {}                     # knorm, h2o


class DecodeRun:
    """Decode streaming: after a 2048-token prefill, one step = one single-token update."""

    def __init__(self, w, torch, binding, stream):
        self.w, self.torch, self.binding = w, torch, binding
        B, H = w["batch"], w["heads"]
        k0, v0 = synth.decode_prefill(B, H, w["prefill"])
        self.k0 = torch.from_numpy(k0.view(np.int16)).cuda().view(torch.bfloat16)
        self.v0 = torch.from_numpy(v0.view(np.int16)).cuda().view(torch.bfloat16)
        ks, vs = synth.decode_steps(0, w["steps"], B, H)
        self.ks = torch.from_numpy(ks.view(np.int16)).cuda().view(torch.bfloat16)
        self.vs = torch.from_numpy(vs.view(np.int16)).cuda().view(torch.bfloat16)
        meth, extra = _scorer_kwargs(w, H, torch)
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

    def score_bytes_per_launch(self):
        w = self.w
        return w["batch"] * w["heads"] * (128 * 2 + 4)

    def graph_leg(self, stream, reps, per_graph=64):
        """The same steps captured in one CUDA graph of `per_graph` decode steps and replayed;
        before each replay the cache is restored to the captured start state (evict_set_state,
        outside the timed events)."""
        torch, b = self.torch, self.binding
        per_graph = min(per_graph, self.w["steps"])
        with torch.cuda.stream(stream):
            snap = [t.contiguous().clone() for t in self.cache.view()]
        off = b.evict_stats(self.handle)["offset"]
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        launches0 = b.evict_launch_count()
        with torch.cuda.graph(g, stream=stream):
            for s in range(per_graph):
                b.evict_update_and_fetch(self.handle, self.ks[s].data_ptr(), self.vs[s].data_ptr(), None, 1)
        launches = b.evict_launch_count() - launches0
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps + 1)]
        with torch.cuda.stream(stream):
            for a, e in evs:
                b.evict_set_state(self.handle, snap[0].data_ptr(), snap[1].data_ptr(), snap[2].data_ptr(),
                                  snap[3].data_ptr(), snap[0].shape[2], off)
                a.record(stream)
                g.replay()
                e.record(stream)
        stream.synchronize()
        b.evict_sync(self.handle)
        ms = sum(a.elapsed_time(e) for a, e in evs[1:]) / reps          # the first replay is warm-up
        return {"steps_per_graph": per_graph, "replays": reps, "gpu_launches_per_graph": int(launches),
                "ms_per_step": round(ms / per_graph, 5),
                "value": round(self.tokens_per_step / (ms / per_graph / 1e3), 1), "unit": UNIT}


class LongContextRun:
    """Long-context chunked prefill: one step = 16 blocks of 8192 tokens through one cache."""

    def __init__(self, w, torch, binding, stream):
        self.w, self.torch, self.binding = w, torch, binding
        B, H = w["batch"], w["heads"]
        self.k, self.v = [], []
        for blk in range(w["blocks"]):
            k, v = synth.long_context_block(blk, B, H, w["block"])
            self.k.append(torch.from_numpy(k.view(np.int16)).cuda().view(torch.bfloat16))
            self.v.append(torch.from_numpy(v.view(np.int16)).cuda().view(torch.bfloat16))
        meth, extra = _scorer_kwargs(w, H, torch)
        if w["method"] == "qfilters":
            q = synth.long_context_queries(H)
            qd = torch.from_numpy(q.view(np.int16)).cuda()
            f = torch.empty((H, 128), dtype=torch.float32, device="cuda")
            binding.evict_qfilters_calibrate(qd.data_ptr(), binding.EVICT_BF16, H, q.shape[1], 128, H,
                                             f.data_ptr(), stream.cuda_stream)
            extra["filters"] = f
        # the fallback freezes once per sequence, on the first block (>= 128 keys)
        self.freeze_rows = w["block"] if w["method"] == "qfilters_fallback" else 0
        self.cache = binding.EvictCache(meth, B, H, budget=w["budget"], n_sink=w["n_sink"],
                                        recent=w["recent"], max_block=w["block"], stream=stream.cuda_stream, **extra)
        self.handle = self.cache.handle
        self.handles = [self.handle]
        per_bh = sum(min(blk * w["block"], w["budget"]) + w["block"] for blk in range(w["blocks"]))
        kk = [min(blk * w["block"], w["budget"]) for blk in range(w["blocks"])]
        m = w["block"]
        self.logits = B * H * sum(m * k + m * (m + 1) // 2 for k in kk)
        self.tokens_per_step = B * H * per_bh
        self.calls_per_step = w["blocks"]
        self.rows_per_call = per_bh / w["blocks"]

    def step(self):
        self.binding.evict_reset(self.handle)
        for k, v in zip(self.k, self.v):
            self.binding.evict_update_and_fetch(self.handle, k.data_ptr(), v.data_ptr(), None, self.w["block"])

    def setup_e2e(self):
        t = self.torch
        self.kh = [x.view(t.int16).cpu().pin_memory() for x in self.k]
        self.vh = [x.view(t.int16).cpu().pin_memory() for x in self.v]
        self.out_h = t.empty((self.w["batch"] * self.w["heads"] * self.w["budget"],), dtype=t.int32).pin_memory()
        self.h2d = sum(x.numel() * 2 for x in self.kh) * 2
        self.d2h = self.out_h.numel() * 4

    def step_e2e(self):
        self.binding.evict_reset(self.handle)
        view = None
        for kh, vh in zip(self.kh, self.vh):
            view = self.binding.evict_update_and_fetch_host(self.handle, kh.data_ptr(), vh.data_ptr(), None,
                                                            self.w["block"])
        pos = self.binding.view_tensors(view, self.w["batch"], self.w["heads"], "bf16")[2]
        self.out_h.copy_(pos.reshape(-1), non_blocking=True)

    def score_bytes_per_launch(self):
        w = self.w
        return w["batch"] * w["heads"] * w["block"] * (128 * 2 + 4)


class CurdkvPlantedRun:
    """CurDKV planted geometry: a 16384-row cache (reloaded before every step,
    outside the timed events) absorbs a 512-token block whose keys are the
    proxy queries; budget 2048."""

    def __init__(self, w, torch, binding, stream):
        self.w, self.torch, self.binding = w, torch, binding
        B, H, S0, m = w["batch"], w["heads"], w["existing"], w["incoming"]
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
        t = self.torch
        self.kh = self.kn.view(t.int16).cpu().pin_memory()
        self.vh = self.vn.view(t.int16).cpu().pin_memory()
        self.out_h = t.empty((self.w["batch"] * self.w["heads"] * self.w["budget"],), dtype=t.int32).pin_memory()
        self.h2d, self.d2h = 2 * self.kh.numel() * 2, self.out_h.numel() * 4

    def step_e2e(self):
        view = self.binding.evict_update_and_fetch_host(self.handle, self.kh.data_ptr(), self.vh.data_ptr(), None,
                                                        self.w["incoming"])
        pos = self.binding.view_tensors(view, self.w["batch"], self.w["heads"], "bf16")[2]
        self.out_h.copy_(pos.reshape(-1), non_blocking=True)


class KnormSingleRun:
    def __init__(self, w, torch, binding, stream):
        self.w, self.torch, self.binding = w, torch, binding
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

    def score_bytes_per_launch(self):
        return self.w["seq"] * (128 * 4 + 4)


RUNS = {"qfilters_stack": StackRun, "decode": DecodeRun, "long_context": LongContextRun,
        "knorm_single": KnormSingleRun, "curdkv_planted": CurdkvPlantedRun}


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
    w = WORKLOADS[args.workload]
    with torch.cuda.stream(stream):
        run = RUNS[args.workload](w, torch, binding, stream)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    reload = getattr(run, "reload", None)
    # warm-up, on the same shapes as the timed steps
    for _ in range(args.warmup):
        if reload:
            reload()
        run.step()
    barrier()
    # Two timed regions of K steps each, CUDA events on the launching stream. The first gives the
    # step time (value): events only around each step. The second, right after it, also brackets
    # every kernel launch of the first handle with events (per-kernel times, roofline); those
    # events make each launch wait for the previous kernel to drain, so that region's steps are
    # slower and it is reported separately (profiled_ms_per_step).
    def timed_steps():
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        barrier()
        for a, b in evs:
            if reload:
                reload()               # restores the pre-existing cache; outside the timed events
            a.record(stream)
            run.step()
            b.record(stream)
        barrier()
        return sum(a.elapsed_time(b) for a, b in evs)

    with ClockSampler(local) as clk:
        launches0 = binding.evict_launch_count()
        ms = timed_steps()
        launches = binding.evict_launch_count() - launches0
        binding.evict_set_profiling(run.handles[0], True)
        profiled_ms = timed_steps()
    ktimes = binding.evict_kernel_times(run.handles[0])
    binding.evict_set_profiling(run.handles[0], False)
    for h in run.handles:
        binding.evict_sync(h)
    ms = max_over_ranks(ms)
    ms_per_step = ms / args.steps
    value = job_throughput(world, run.tokens_per_step, ms_per_step)
    profiled_ms_per_step = max_over_ranks(profiled_ms) / args.steps

    # end-to-end through the host-buffer entry point (copies inside the region)
    run.setup_e2e()
    for _ in range(args.warmup):
        if reload:
            reload()
        run.step_e2e()
    barrier()
    e2e_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    for a, b in e2e_evs:
        if reload:
            reload()
        a.record(stream)
        run.step_e2e()
        b.record(stream)
    barrier()
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_evs) / args.steps)

    peaks, peak_kind = _peaks()
    work = algorithmic_work(run, binding)
    # the decode loop captured in a CUDA graph (one launch sequence replayed per 64 steps);
    # after the work count, which reads the last eager update's compaction metadata
    graph = run.graph_leg(stream, max(3, min(args.steps, 20))) if hasattr(run, "graph_leg") else None
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
            roof = {"kernel": top, "bound": "alu", "achieved": round(achieved, 2), "peak": FP32_FMA_TFLOPS,
                    "unit": "TFLOP/s", "frac": round(achieved / FP32_FMA_TFLOPS, 4),
                    "algorithmic_flops_per_launch": wk["flops"]}
        elif "bytes" in wk:
            achieved = wk["bytes"] / (per_launch_ms / 1e3) / 1e9
            roof = {"kernel": top, "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "algorithmic_bytes_per_launch": wk["bytes"]}
        elif "flops" in wk and top in ("curdkv_lse", "curdkv_colsum"):
            achieved = wk["flops"] / (per_launch_ms / 1e3) / 1e12
            roof = {"kernel": top, "bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                    "algorithmic_flops_per_launch": wk["flops"]}
        else:
            roof = {"kernel": top, "bound": "latency", "achieved": None, "peak": None, "unit": None, "frac": None}
        roof["peak_kind"] = peak_kind
        roof["traffic"] = _ncu_traffic(top, args.workload)
        roof["avg_launch_us"] = round(per_launch_ms * 1e3, 2)
    # the whole path: every kernel's algorithmic bytes per step over the (uninstrumented) step time,
    # when all of the step's kernels are byte-bound
    path = None
    if ktimes and all("bytes" in work.get(k, {}) for k in ktimes):
        per_step = sum(work[k]["bytes"] * n / args.steps for k, (n, _) in ktimes.items())
        gbs = per_step / (ms_per_step / 1e3) / 1e9
        path = {"algorithmic_bytes_per_step": int(per_step), "achieved": round(gbs, 1), "unit": "GB/s",
                "peak": peaks["hbm_gbs"], "frac": round(gbs / peaks["hbm_gbs"], 4)}
    cpu = cpu_baseline(args.workload) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded generators standing in for real-model activations)",
            "config": {"workload": args.workload, **{k: v for k, v in w.items()},
                       "storage": w["dtype"], "tokens_per_step": run.tokens_per_step,
                       "calls_per_step": run.calls_per_step, "l2": "inputs larger than L2" if
                       args.workload in ("qfilters_stack", "long_context") else "working set may be L2-resident",
                       "parallelism": f"replica-per-gpu x{world}"},
            "e2e": {"value": round(job_throughput(world, run.tokens_per_step, e2e_ms), 1), "unit": UNIT,
                    "h2d_bytes_per_step": run.h2d, "d2h_bytes_per_step": run.d2h, "ms_per_step": round(e2e_ms, 4)},
            "gpu_launches": int(launches),
            "roofline": roof,
            "kernels": kernels,
            "path_roofline": path,
            "profiled_ms_per_step": round(profiled_ms_per_step, 5),
            "kernel_timing": "per-kernel CUDA events on the launching stream over a second timed region "
                             "of the same K steps (profiled_ms_per_step); the step time comes from the "
                             "first region, which has events around each step only",
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
        }
        if hasattr(run, "calib_ms"):
            line["config"]["calibration_ms_per_layer"] = round(run.calib_ms, 3)
        if graph is not None:
            line["graph"] = graph
        if hasattr(run, "class2_retention"):
            line["config"]["class2_retention"] = run.class2_retention()
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


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
    """
    w = run.w
    e = 2 if w["dtype"] == "bf16" else 4
    units = w["layers"] * w["batch"] * w["heads"]
    m = w.get("seq", w.get("block", w.get("incoming", 1)))
    if isinstance(run, DecodeRun):
        m = 1
    n = run.rows_per_call
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
    per_row = 128 * 2 + (16 if w["method"] == "h2o" else 4)
    out["curdkv_attn_small"] = {"bytes": int(units * n_small * per_row)}
    logits = getattr(run, "logits", None)
    if logits:
        calls = run.calls_per_step
        for k in ("curdkv_lse", "curdkv_colsum"):
            out[k] = {"flops": 2 * 128 * logits / calls, "exps": logits / calls}
        out["curdkv_gram"] = {"flops": units * n * 2 * 128 * 128}
        out["h2o_mass"] = {"bytes": int(units * n * 16)}       # read the sum, write it, read/write the score
        out["curdkv_leverage"] = {"bytes": int(units * n * (128 * 2 + 12))}
    return out


# ----------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ----------------------------------------------------------------------------
def _oracle_sample(workload, budget_s=10.0):
    """Run the oracle on a bounded sample of the workload; returns (tokens, seconds, description)."""
    from oracle import calibrate as ocal
    from oracle.cache import OracleCache
    w = WORKLOADS[workload]
    tokens, secs, done = 0, 0.0, 0
    if workload == "qfilters_stack":
        t0 = time.perf_counter()
        for layer in range(w["layers"]):
            d = synth.qfilters_layer(layer, seq_len=w["seq"])
            t1 = time.perf_counter()
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
        meth, kw = _scorer_kwargs(w, w["heads"])
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
    if workload == "long_context":
        # one (b, h) unit followed through the stream (units are independent)
        meth, kw = _scorer_kwargs(w, w["heads"])
        if w["method"] == "qfilters":
            kw["filters"] = ocal.calibrate(synth.long_context_queries(w["heads"]), w["heads"])[:1].astype(np.float32)
        c = OracleCache(meth, 1, 1, budget=w["budget"], n_sink=w["n_sink"], recent=w["recent"], **kw)
        for blk in range(w["blocks"]):
            k, v = synth.long_context_block(blk, w["batch"], w["heads"], w["block"])
            t1 = time.perf_counter()
            n = c.n_kept + w["block"]
            c.update_and_fetch(k[:1, :1], v[:1, :1])
            secs += time.perf_counter() - t1
            tokens += n
            done += 1
            if secs > budget_s:
                break
        return tokens, secs, f"{done} of {w['blocks']} blocks of one (b, h) unit"
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


def cpu_baseline(workload):
    tokens, secs, sample = _oracle_sample(workload)
    return {"value": round(tokens / secs, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": sample + "; numpy, single thread (the oracle's array ops do not use BLAS threads)"}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    vals = []
    for _ in range(args.warmup):
        _oracle_sample(args.workload, budget_s=2.0)
    tokens_total, secs_total, sample = 0, 0.0, ""
    for _ in range(args.steps):
        t, s, sample = _oracle_sample(args.workload, budget_s=5.0)
        tokens_total += t
        secs_total += s
        vals.append(t / s)
    value = tokens_total / secs_total
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs_total / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": {"workload": args.workload, **w},
            "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="qfilters_stack")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--method", choices=["knorm", "qfilters", "qfilters_fallback", "curdkv", "h2o"], default=None,
                    help="scorer for the long_context and decode workloads (qfilters_fallback: Q-Filters "
                         "without calibrated filters, freezing a key-SVD filter after 128 keys) and for "
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
