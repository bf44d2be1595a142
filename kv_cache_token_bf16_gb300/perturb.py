"""Synthetic output-perturbation harness for the eviction scorers.

How far does an evicted cache move a layer's attention output? For probe
queries q drawn from a query cluster, the full cache gives
o_full = softmax(q K^T / sqrt(D)) V and the kept rows o_kept; the
perturbation of one trial is the mean over the probes of 1 - cos(o_kept,
o_full), and an arm's advantage is random eviction's perturbation minus its
own ("L2Norm — Intrinsic Key-Norm Eviction", §Evidence and the offline
harness paragraph: keep-low against keep-high, random and H2O-adapted,
paper-like geometry against an isotropic control; "Q-Filters —
Query-Agnostic Projection Eviction", §Evidence and its offline harness:
sign +1 / -1, best-of-sign, KNorm-adapted, H2O-adapted and random, with the
key-SVD fallback's filter cosine to the planted axis). No weights or text:
the geometries are the seeded constructions of ``synth.perturbation_geometry``.

Every arm but random evicts through the library on the GPU (one block of
the whole sequence per trial row, n_sink 4); Q-Filters arms run the key-SVD
fallback, as the pages' harness does without a calibration artifact. The
attention outputs are the harness's own measurement, computed in fp64 on the
host from the kept positions.

    python -m kv_cache_token_bf16_gb300.perturb [--lengths 256 512 1024] [--budgets 64 128]
"""
from __future__ import annotations

import argparse
import json

import numpy as np

from . import synth

ARMS = ("knorm_low", "knorm_high", "qfilters_plus", "qfilters_minus", "qfilters_best", "h2o", "random")
N_SINK = 4


def attention_output(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """softmax(q k^T / sqrt(D)) v for probes q [P, D], keys k [n, D], values v [n, D] (fp64)."""
    z = q @ k.T / np.sqrt(k.shape[1])
    z -= z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    return p @ v


def perturbation(q: np.ndarray, k: np.ndarray, v: np.ndarray, kept: np.ndarray) -> float:
    """Mean over the probes of 1 - cos(o_kept, o_full); 0 when every row is kept."""
    full = attention_output(q, k, v)
    part = attention_output(q, k[kept], v[kept])
    cos = np.sum(part * full, axis=1) / (np.linalg.norm(part, axis=1) * np.linalg.norm(full, axis=1))
    return float(np.mean(1.0 - cos))


def random_kept(seed: int, batch: int, length: int, budget: int) -> np.ndarray:
    """Random eviction: the sinks plus budget - n_sink rows drawn without replacement."""
    g = np.random.Generator(np.random.PCG64(seed))
    out = []
    for _ in range(batch):
        rest = N_SINK + g.choice(length - N_SINK, budget - N_SINK, replace=False)
        out.append(np.sort(np.r_[np.arange(N_SINK), rest]))
    return np.stack(out)


def gpu_kept(arm: str, k_bits: np.ndarray, v_bits: np.ndarray, budget: int):
    """Kept positions [B, budget] of one GPU arm, the eviction time (ms) and, for the Q-Filters
    arms, the frozen filters [B, 128]."""
    import torch

    from . import binding
    B, _, S, _ = k_bits.shape
    if arm.startswith("knorm"):
        kw = dict(method="knorm", keep_low=arm == "knorm_low")
    elif arm.startswith("qfilters"):
        kw = dict(method="qfilters", filters=None, sign=1 if arm == "qfilters_plus" else -1, calib_tokens=128)
    else:
        kw = dict(method="h2o")
    meth = kw.pop("method")
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.bfloat16)
    kd, vd = dev(k_bits), dev(v_bits)
    cache = binding.EvictCache(meth, B, 1, budget=budget, n_sink=N_SINK, max_block=S, **kw)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    view = cache.update_and_fetch(kd, vd)
    b.record()
    cache.sync()
    torch.cuda.synchronize()
    kept = view[2][:, 0].cpu().numpy().astype(np.int64)
    filt = cache.filters()[:, 0] if meth == "qfilters" else None
    cache.close()
    return kept, a.elapsed_time(b), filt


def run(geometry: str, length: int, budget: int, seed: int = 0, batch: int = 8, n_probe: int = 32) -> dict:
    """One sweep point: per arm the mean perturbation over the trial rows, its advantage over
    random eviction and the eviction time; the fallback filters' mean |cosine| to the axis."""
    k_bits, v_bits, q, u = synth.perturbation_geometry(geometry, synth.seed_for(6, seed), batch, length, n_probe)
    kf = synth.bf16_bits_to_f32(k_bits[:, 0]).astype(np.float64)
    vf = synth.bf16_bits_to_f32(v_bits[:, 0]).astype(np.float64)
    qf = q.astype(np.float64)
    per_row, ms = {}, {}
    filters = {}
    for arm in ARMS:
        if arm == "qfilters_best":
            continue
        if arm == "random":
            kept = random_kept(synth.seed_for(6, 100 + seed), batch, length, budget)
        else:
            kept, ms[arm], f = gpu_kept(arm, k_bits, v_bits, budget)
            if f is not None:
                filters[arm] = f
        per_row[arm] = np.array([perturbation(qf[r], kf[r], vf[r], kept[r]) for r in range(batch)])
    per_row["qfilters_best"] = np.minimum(per_row["qfilters_plus"], per_row["qfilters_minus"])
    rnd = per_row["random"]
    out = {"geometry": geometry, "length": length, "budget": budget, "trials": batch, "probes": n_probe,
           "perturbation": {a: round(float(per_row[a].mean()), 4) for a in ARMS},
           "advantage_vs_random": {a: round(float((rnd - per_row[a]).mean()), 4) for a in ARMS if a != "random"},
           "evict_ms": {a: round(t, 3) for a, t in ms.items()}}
    f = filters.get("qfilters_plus")
    if f is not None:
        cos = np.abs(np.sum(f.astype(np.float64) * u, axis=1)) / np.linalg.norm(f, axis=1)
        out["filter_cosine"] = round(float(cos.mean()), 4)
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--lengths", type=int, nargs="+", default=[256, 512, 1024])
    ap.add_argument("--budgets", type=int, nargs="+", default=[64, 128])
    ap.add_argument("--geometries", nargs="+", default=list(synth.PERTURB_GEOMETRIES))
    ap.add_argument("--trials", type=int, default=8)
    args = ap.parse_args(argv)
    from . import _build
    _build.ensure_built()
    for geo in args.geometries:
        for length in args.lengths:
            for budget in args.budgets:
                if budget < length:
                    print(json.dumps(run(geo, length, budget, batch=args.trials)), flush=True)


if __name__ == "__main__":
    main()
