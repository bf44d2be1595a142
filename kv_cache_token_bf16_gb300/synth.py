"""Seeded synthetic inputs for the eviction path.

This module is the ONLY code shared between the CPU oracle side (tests,
``bench.py``'s CPU baseline) and the CUDA side. It draws random numbers and
rounds them to the storage format; it holds none of the eviction method's
arithmetic (no scoring, no softmax, no SVD, no selection).

Every generator takes an explicit seed and returns numpy arrays:

* bf16 tensors are returned as ``uint16`` arrays holding the bf16 bit
  patterns (numpy has no bf16 type); the CUDA side reinterprets the same bits
  as ``torch.bfloat16`` and the oracle expands them itself.
* fp32 tensors are returned as ``float32``.

Workloads (the pages measure on real models and real text; these seeded
draws stand in for them, with the shapes and value laws each workload names):

1. KNorm single sequence, fp32 keys/values iid N(0,1).
2. Q-Filters calibrated Llama-3.2-3B-like stack: per (layer, KV head) a unit
   drift direction u shared by its GQA query heads; queries
   u*N(4, 0.5) + N(0, I); keys N(0, I) + c*u with c ~ N(0, 2) (std).
3. Decode streaming: keys s*N(0, I) with s ~ LogNormal(0, 0.3) per token,
   values N(0, 1); a seeded random unit filter per KV head.
4. CurDKV planted geometry: per (b, h) a unit common direction c; every key
   c + N(0, 0.05); half the tokens class 1 (value 3*N(0,1)), half class 2
   (value 1e-3*N(0,1)), classes in a random permutation.
5. Long-context chunked prefill: keys N(0, I) + 2*u_h, values N(0, 1),
   131072 tokens in 8192-token blocks; calibration queries u_h*N(4,0.5)+N(0,I).

Distribution parameters follow numpy's (mean, std) convention.
"""
from __future__ import annotations

import numpy as np

SEED_BASE = 20261202
HEAD_DIM = 128


def seed_for(workload: int, sub: int = 0) -> int:
    """Seed of one workload's draw: base + 1000*workload + sub-index."""
    return SEED_BASE + 1000 * workload + sub


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even); return the bits.

    NaN maps to the canonical quiet NaN 0x7FC0 (sign kept). For every other
    value the 32-bit sum below cannot wrap (the largest finite magnitude plus
    the rounding bias stays below 2^32).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    rounded = ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        sign = ((b >> np.uint32(16)) & np.uint32(0x8000)).astype(np.uint16)
        rounded = np.where(nan, sign | np.uint16(0x7FC0), rounded)
    return rounded


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (for building inputs)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def unit_vectors(g: np.random.Generator, count: int, dim: int = HEAD_DIM) -> np.ndarray:
    """`count` seeded random unit vectors (float64), one per row."""
    u = g.standard_normal((count, dim))
    return u / np.linalg.norm(u, axis=1, keepdims=True)


# --------------------------------------------------------------------------
# 1. KNorm single sequence (fp32)
# --------------------------------------------------------------------------
def knorm_single_sequence(seq_len: int = 1024, seed: int | None = None):
    """B=1, H_kv=1, D=128 fp32 keys and values iid N(0,1).

    Returns (K, V) of shape [1, 1, seq_len, 128], float32.
    """
    g = rng(seed_for(1) if seed is None else seed)
    k = g.standard_normal((1, 1, seq_len, HEAD_DIM)).astype(np.float32)
    v = g.standard_normal((1, 1, seq_len, HEAD_DIM)).astype(np.float32)
    return k, v


# --------------------------------------------------------------------------
# 2. Q-Filters calibrated layer stack (bf16)
# --------------------------------------------------------------------------
def qfilters_layer(layer: int, n_q_heads: int = 24, n_kv_heads: int = 8, n_samples: int = 3000,
                   seq_len: int = 8192, batch: int = 1, drift_mean: float = 4.0,
                   drift_std: float = 0.5, key_proj_std: float = 2.0):
    """One layer of the GQA stack.

    Returns a dict with
      ``u``       [n_kv_heads, 128] float64 unit drift directions,
      ``queries`` [n_q_heads, n_samples, 128] bf16 bits (u*N(4,0.5)+N(0,I)),
      ``k``, ``v`` [batch, n_kv_heads, seq_len, 128] bf16 bits.
    Query head h belongs to KV head h // (n_q_heads // n_kv_heads).
    """
    g = rng(seed_for(2, layer))
    group = n_q_heads // n_kv_heads
    u = unit_vectors(g, n_kv_heads)
    uq = np.repeat(u, group, axis=0)                                   # [Hq, D]
    c = g.normal(drift_mean, drift_std, size=(n_q_heads, n_samples, 1))
    q = c * uq[:, None, :] + g.standard_normal((n_q_heads, n_samples, HEAD_DIM))
    ck = g.normal(0.0, key_proj_std, size=(batch, n_kv_heads, seq_len, 1))
    k = g.standard_normal((batch, n_kv_heads, seq_len, HEAD_DIM)) + ck * u[None, :, None, :]
    v = g.standard_normal((batch, n_kv_heads, seq_len, HEAD_DIM))
    return {
        "u": u,
        "queries": f32_to_bf16_bits(q.astype(np.float32)),
        "k": f32_to_bf16_bits(k.astype(np.float32)),
        "v": f32_to_bf16_bits(v.astype(np.float32)),
    }


# --------------------------------------------------------------------------
# 3. Decode streaming (bf16)
# --------------------------------------------------------------------------
def _lognormal_keys(g, shape):
    s = g.lognormal(0.0, 0.3, size=shape[:-1] + (1,))
    return s * g.standard_normal(shape)


def decode_prefill(batch: int = 32, n_kv_heads: int = 8, prefill: int = 2048, seed: int | None = None):
    """Prefill block of the decode workload: (K, V) bf16 bits [B, H, prefill, 128]."""
    g = rng(seed_for(3, 0) if seed is None else seed)
    k = _lognormal_keys(g, (batch, n_kv_heads, prefill, HEAD_DIM))
    v = g.standard_normal((batch, n_kv_heads, prefill, HEAD_DIM))
    return f32_to_bf16_bits(k.astype(np.float32)), f32_to_bf16_bits(v.astype(np.float32))


def decode_steps(first_step: int, n_steps: int, batch: int = 32, n_kv_heads: int = 8,
                 seed: int | None = None):
    """Decode tokens ``first_step .. first_step+n_steps-1``: bf16 bits [n_steps, B, H, 1, 128].

    Each step has its own seed so any window of steps is reproducible alone.
    """
    ks, vs = [], []
    for s in range(first_step, first_step + n_steps):
        g = rng((seed_for(3, 1) if seed is None else seed) * 7919 + s)
        ks.append(_lognormal_keys(g, (batch, n_kv_heads, 1, HEAD_DIM)))
        vs.append(g.standard_normal((batch, n_kv_heads, 1, HEAD_DIM)))
    k = np.stack(ks).astype(np.float32)
    v = np.stack(vs).astype(np.float32)
    return f32_to_bf16_bits(k), f32_to_bf16_bits(v)


def decode_filters(n_kv_heads: int = 8, seed: int | None = None) -> np.ndarray:
    """Seeded random unit filter per KV head, float32 [H, 128]."""
    g = rng(seed_for(3, 2) if seed is None else seed)
    return unit_vectors(g, n_kv_heads).astype(np.float32)


# --------------------------------------------------------------------------
# 4. CurDKV planted two-class geometry (bf16)
# --------------------------------------------------------------------------
def curdkv_planted(batch: int = 8, n_kv_heads: int = 8, existing: int = 16384, incoming: int = 512,
                   key_noise: float = 0.05, v1_scale: float = 3.0, v2_scale: float = 1e-3,
                   seed: int | None = None):
    """Planted geometry over n = existing + incoming tokens per (b, h).

    Returns dict with ``k``, ``v`` bf16 bits [B, H, n, 128] (first ``existing``
    rows are the pre-existing cache, the rest the incoming block) and
    ``cls`` int8 [B, H, n] (1 = value-relevant, 2 = near-zero value).
    Exactly half of the n tokens of each (b, h) are class 1.
    """
    g = rng(seed_for(4) if seed is None else seed)
    n = existing + incoming
    c = unit_vectors(g, batch * n_kv_heads).reshape(batch, n_kv_heads, 1, HEAD_DIM)
    k = c + key_noise * g.standard_normal((batch, n_kv_heads, n, HEAD_DIM))
    cls = np.empty((batch, n_kv_heads, n), dtype=np.int8)
    base = np.concatenate([np.ones(n // 2, np.int8), np.full(n - n // 2, 2, np.int8)])
    for b in range(batch):
        for h in range(n_kv_heads):
            cls[b, h] = g.permutation(base)
    scale = np.where(cls == 1, v1_scale, v2_scale)[..., None]
    v = scale * g.standard_normal((batch, n_kv_heads, n, HEAD_DIM))
    return {"k": f32_to_bf16_bits(k.astype(np.float32)),
            "v": f32_to_bf16_bits(v.astype(np.float32)), "cls": cls}


# --------------------------------------------------------------------------
# 5. Long-context chunked prefill (bf16)
# --------------------------------------------------------------------------
def long_context_directions(n_kv_heads: int = 8, seed: int | None = None) -> np.ndarray:
    """Per-head unit drift direction u_h, float64 [H, 128]."""
    g = rng(seed_for(5, 999) if seed is None else seed)
    return unit_vectors(g, n_kv_heads)


def long_context_block(block: int, batch: int = 4, n_kv_heads: int = 8, block_len: int = 8192,
                       drift: float = 2.0, seed: int | None = None, first_row: int = 0):
    """Block ``block`` of the 131072-token stream: (K, V) bf16 bits [B, H, block_len, 128].

    Rows ``first_row .. first_row + batch - 1`` of a global batch: every batch
    row is drawn from its own stream (seeded by the block and the global row),
    so a batch split into shards draws exactly the rows of the whole batch.
    """
    u = long_context_directions(n_kv_heads)
    base = seed_for(5, block) if seed is None else seed
    k = np.empty((batch, n_kv_heads, block_len, HEAD_DIM), np.uint16)
    v = np.empty_like(k)
    for j in range(batch):
        g = np.random.Generator(np.random.PCG64([base, first_row + j]))
        kr = g.standard_normal((n_kv_heads, block_len, HEAD_DIM), dtype=np.float32)
        kr += (drift * u[:, None, :]).astype(np.float32)
        k[j] = f32_to_bf16_bits(kr)
        v[j] = f32_to_bf16_bits(g.standard_normal((n_kv_heads, block_len, HEAD_DIM), dtype=np.float32))
    return k, v


def long_context_queries(n_heads: int = 8, n_samples: int = 3000, seed: int | None = None):
    """Calibration queries for workload 5 (H_q = H_kv): bf16 bits [H, N, 128]."""
    u = long_context_directions(n_heads)
    g = rng(seed_for(5, 998) if seed is None else seed)
    c = g.normal(4.0, 0.5, size=(n_heads, n_samples, 1))
    q = c * u[:, None, :] + g.standard_normal((n_heads, n_samples, HEAD_DIM))
    return f32_to_bf16_bits(q.astype(np.float32))


# --------------------------------------------------------------------------
# Small generic draws for parity/edge-case tests
# --------------------------------------------------------------------------
def gaussian_block(seed: int, batch: int, n_kv_heads: int, length: int, dtype: str = "bf16",
                   scale: float = 1.0):
    """(K, V) iid scale*N(0,1) in the requested storage format ("bf16" bits or "fp32")."""
    g = rng(seed)
    k = (scale * g.standard_normal((batch, n_kv_heads, length, HEAD_DIM))).astype(np.float32)
    v = (scale * g.standard_normal((batch, n_kv_heads, length, HEAD_DIM))).astype(np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(k), f32_to_bf16_bits(v)
    return k, v


def planted_spectrum_values(seed: int, batch: int, n_kv_heads: int, length: int, rank: int = 16,
                            top: float = 3.0, decay: float = 0.9, floor: float = 0.05):
    """Values whose rows share a planted spectrum: V = Z diag(s) R^T (bf16 bits).

    Z ~ N(0,1) [length, 128], R a seeded random orthogonal matrix per (b, h),
    s_j = top * decay^j for j < rank and `floor` beyond: a clear gap after the
    first `rank` directions.
    """
    g = rng(seed)
    s = np.where(np.arange(HEAD_DIM) < rank, top * decay ** np.arange(HEAD_DIM), floor)
    out = np.empty((batch, n_kv_heads, length, HEAD_DIM), np.float32)
    for b in range(batch):
        for h in range(n_kv_heads):
            q, _ = np.linalg.qr(g.standard_normal((HEAD_DIM, HEAD_DIM)))
            z = g.standard_normal((length, HEAD_DIM))
            out[b, h] = (z * s) @ q.T
    return f32_to_bf16_bits(out)


def clustered_keys(seed: int, batch: int, n_kv_heads: int, length: int, spread: float = 0.5):
    """Keys = a common unit direction per (b, h) + spread * N(0, I) (bf16 bits)."""
    g = rng(seed)
    c = unit_vectors(g, batch * n_kv_heads).reshape(batch, n_kv_heads, 1, HEAD_DIM)
    k = c + spread * g.standard_normal((batch, n_kv_heads, length, HEAD_DIM))
    return f32_to_bf16_bits(k.astype(np.float32))


def dominant_axis_block(seed: int, batch: int, n_kv_heads: int, length: int, spread: float = 12.0,
                        dtype: str = "bf16"):
    """Keys with one planted dominant variance axis per (b, h), values N(0, 1).

    k = N(0, I) + spread * N(0, 1) * u_bh for a seeded unit axis u_bh, so the
    centred keys' top singular direction is u_bh up to sampling noise.
    Returns (K, V) in the storage format ("bf16" bits or "fp32") and the axes
    u [B, H, 128] (float64).
    """
    g = rng(seed)
    u = unit_vectors(g, batch * n_kv_heads).reshape(batch, n_kv_heads, 1, HEAD_DIM)
    t = g.standard_normal((batch, n_kv_heads, length, 1))
    k = (g.standard_normal((batch, n_kv_heads, length, HEAD_DIM)) + spread * t * u).astype(np.float32)
    v = g.standard_normal((batch, n_kv_heads, length, HEAD_DIM)).astype(np.float32)
    if dtype == "bf16":
        k, v = f32_to_bf16_bits(k), f32_to_bf16_bits(v)
    return k, v, u[:, :, 0]


# --------------------------------------------------------------------------
# Output-perturbation harness geometries
# --------------------------------------------------------------------------
PERTURB_GEOMETRIES = ("knorm_paper", "qfilters_paper", "isotropic")


def perturbation_geometry(kind: str, seed: int, batch: int, length: int, n_probe: int = 32):
    """Keys, values and probe queries of one harness geometry; every batch row is one trial.

    Per row a seeded unit axis u; probe queries q = 8 u + 0.3 N(0, I) (a query cluster).
      knorm_paper     half the tokens low-norm and aligned with the query cluster
                      (k = u + 0.05 N(0, I)), half high-norm and anti-aligned
                      (k = -2.5 u + 0.15 N(0, I)), in random order;
      qfilters_paper  a quarter of the tokens important: a large projection on the
                      dominant axis u and aligned with the queries (k = 3 u + 0.3 N(0, I)),
                      the rest k = 0.5 N(0, 1) u + 0.3 N(0, I);
      isotropic       k = N(0, I), no relation to the queries.
    Values N(0, I). Returns (K, V) bf16 bits [B, 1, length, 128], probes float32
    [B, n_probe, 128] and the axes u float64 [B, 128].
    """
    if kind not in PERTURB_GEOMETRIES:
        raise ValueError(f"unknown geometry {kind}")
    g = rng(seed)
    u = unit_vectors(g, batch)                                   # [B, D]
    q = 8.0 * u[:, None, :] + 0.3 * g.standard_normal((batch, n_probe, HEAD_DIM))
    noise = g.standard_normal((batch, length, HEAD_DIM))
    if kind == "knorm_paper":
        aligned = np.stack([g.permutation(length) < length // 2 for _ in range(batch)])[..., None]
        k = np.where(aligned, u[:, None, :] + 0.05 * noise, -2.5 * u[:, None, :] + 0.15 * noise)
    elif kind == "qfilters_paper":
        important = np.stack([g.permutation(length) < length // 4 for _ in range(batch)])[..., None]
        c = np.where(important, 3.0, 0.5 * g.standard_normal((batch, length, 1)))
        k = c * u[:, None, :] + 0.3 * noise
    else:
        k = noise
    v = g.standard_normal((batch, length, HEAD_DIM))
    kb = f32_to_bf16_bits(k[:, None].astype(np.float32))
    vb = f32_to_bf16_bits(v[:, None].astype(np.float32))
    return kb, vb, q.astype(np.float32), u
