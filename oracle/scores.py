"""Intrinsic scores: KNorm (key L2 norm) and Q-Filters (signed projection).

Test infrastructure only.

Sources
-------
* "L2Norm — Intrinsic Key-Norm Eviction", §How it works step 1: the L2 norm
  of each incoming key row, computed once at insertion and never updated.
* "Q-Filters — Query-Agnostic Projection Eviction", §How it works step 3:
  each stored token is scored by sign * (key . filter_dir) in float32, once
  at insertion; §Metal kernels: fp32 accumulation over the stored keys.

Two evaluations are provided:

``*_plain``      the definition in fp64 (used to check score accuracy);
``*_canonical``  fp32 in one fixed evaluation order (used to drive selection,
                 so that kept sets are reproducible bit for bit).

Reading (the pages only say "fp32"): the canonical order is
  x_d = float32(k_d)                                   (exact for bf16/fp32)
  t_d = fl(x_d * x_d)   [KNorm]   or   fl(x_d * f_d)   [Q-Filters]
        rounded to nearest even, no fused multiply-add, subnormals kept;
  a_c = (((t_{8c} + t_{8c+1}) + t_{8c+2}) + ... + t_{8c+7})   for c = 0..15
        (16 chunks of 8 consecutive elements, summed left to right);
  then a pairwise tree over chunk sums: a_c += a_{c+h} for h = 8, 4, 2, 1
        (c < h), and S = a_0;
  KNorm:  sigma = sqrt(S) rounded to nearest (IEEE square root);
  Q-Filters: sigma = sign * S (exact).
The score is a pure function of the key's bits (and the filter's), never of
the block length, batch or launch shape — the property that makes one-block
prefill and token-by-token decode select identical sets ("L2Norm",
§A third scorer class, consequence 2).
"""
import numpy as np

from .bf16 import to_f32

CHUNK = 8


def _canonical_sum(t: np.ndarray) -> np.ndarray:
    """Fixed-order float32 sum over the last axis of `t` (length 8 * 2^j)."""
    assert t.dtype == np.float32
    d = t.shape[-1]
    assert d % CHUNK == 0
    n_chunks = d // CHUNK
    assert n_chunks & (n_chunks - 1) == 0, "chunk count must be a power of two"
    chunks = t.reshape(t.shape[:-1] + (n_chunks, CHUNK))
    a = chunks[..., 0].copy()
    for j in range(1, CHUNK):
        a = a + chunks[..., j]                       # float32 + float32 -> float32 (RN)
    h = n_chunks // 2
    while h >= 1:
        a = a[..., :h] + a[..., h:2 * h]
        h //= 2
    return a[..., 0]


def key_norm_canonical(k: np.ndarray) -> np.ndarray:
    """KNorm score, canonical fp32: sqrt of the fixed-order sum of squares."""
    x = to_f32(k)
    t = x * x                                         # float32 products, RN
    with np.errstate(invalid="ignore"):
        return np.sqrt(_canonical_sum(t)).astype(np.float32)


def key_norm_plain(k: np.ndarray) -> np.ndarray:
    """KNorm score by definition, in fp64: ||k||_2."""
    x = to_f32(k).astype(np.float64)
    return np.sqrt(np.sum(x * x, axis=-1))


def projection_canonical(k: np.ndarray, filters: np.ndarray, sign: int) -> np.ndarray:
    """Q-Filters score, canonical fp32: sign * fixed-order sum of k_d * f_d.

    `k` is [B, H, T, D] (storage format), `filters` is [H, D] float32.
    """
    x = to_f32(k)
    f = np.asarray(filters, dtype=np.float32)
    t = x * f[None, :, None, :]
    s = _canonical_sum(t)
    return (np.float32(sign) * s).astype(np.float32)


def projection_plain(k: np.ndarray, filters: np.ndarray, sign: int) -> np.ndarray:
    """Q-Filters score by definition, in fp64: sign * (k . f)."""
    x = to_f32(k).astype(np.float64)
    f = np.asarray(filters, dtype=np.float32).astype(np.float64)
    return sign * np.einsum("bhtd,hd->bht", x, f)


def projection_condition(k: np.ndarray, filters: np.ndarray) -> np.ndarray:
    """sum_d |k_d f_d| in fp64: the scale against which a dot-product error is judged."""
    x = to_f32(k).astype(np.float64)
    f = np.asarray(filters, dtype=np.float32).astype(np.float64)
    return np.einsum("bhtd,hd->bht", np.abs(x), np.abs(f))
