"""CurDKV-adapted block scoring: proxy attention, weighted values, leverage.

Test infrastructure only.

Source: "CurDKV-adapted — Value-Aware Leverage-Score Eviction".
* §The honesty crux, item 1: the incoming key stands in for the query.
* §The honesty crux, item 2: weighted_values[i] = attn[i] * values[i]; the
  leverage of row i is l_i = sum_j (s_j^2 / sum s^2) * U[i, j]^2 over the
  block's leading left singular vectors (energy weighting, item 3).
* §How it works, steps 1-4: proxy softmax of the incoming key against all
  stored keys (the softmax H2O uses); the weighted value block; leverage
  over the leading min(rank_cap, n, D) left singular vectors; existing
  tokens accumulate the leverage, the new token is seeded with its own
  leverage (item 4), not with 0.

Readings (the page describes one token at a time; the cache here takes a
block of m tokens per call):
* The m incoming keys are the proxy queries. Query t (row k+t of the
  concatenation) attends rows i <= k+t (causal; it sees itself), with the
  usual 1/sqrt(D) logit scale. With m = 1 this is exactly the page's step 1.
  The alternative "every incoming key sees the whole block" is rejected
  because it does not reduce to the page's steps at m = 1.
* attn[i] = sum over the m queries of their softmax weight on row i.
* sum s^2 runs over ALL singular values (= ||W||_F^2); the numerator keeps
  the leading r = min(rank_cap, n, D) directions. With r >= D the leverage
  of row i is ||w_i||^2 / ||W||_F^2 exactly.
* All-zero weighted values (sum s^2 = 0) give l = 0, finite (§Evidence:
  a degenerate all-zero-value block produces finite scores).
* Everything in fp64; the softmax subtracts each row's maximum.
"""
import numpy as np

from .bf16 import to_f64


def proxy_attention(keys: np.ndarray, m: int) -> np.ndarray:
    """Column sums of the causal key-as-query softmax for one (b, h).

    ``keys`` [n, D] are the concatenated rows (kept then incoming); the last
    m rows are the queries. Returns attn [n] (fp64); sum(attn) == m.
    """
    x = to_f64(keys)
    n, d = x.shape
    k = n - m
    attn = np.zeros(n)
    for t in range(m):
        row = k + t
        logits = x[: row + 1] @ x[row] / np.sqrt(d)
        logits -= logits.max()
        p = np.exp(logits)
        attn[: row + 1] += p / p.sum()
    return attn


def proxy_attention_block(keys: np.ndarray, m: int) -> np.ndarray:
    """Same as ``proxy_attention`` with the m queries handled as one matrix."""
    x = to_f64(keys)
    n, d = x.shape
    k = n - m
    logits = (x[k:] @ x.T) / np.sqrt(d)                   # [m, n]
    causal = np.arange(n)[None, :] > (k + np.arange(m))[:, None]
    logits[causal] = -np.inf
    logits -= logits.max(axis=1, keepdims=True)
    p = np.exp(logits)
    p /= p.sum(axis=1, keepdims=True)
    return p.sum(axis=0)


def leverage(w: np.ndarray, rank_cap: int) -> np.ndarray:
    """Energy-weighted leverage of each row of the weighted-value block W [n, D]."""
    n, d = w.shape
    r = min(rank_cap, n, d)
    u, s, _ = np.linalg.svd(w, full_matrices=False)
    energy = float(np.sum(s * s))
    if energy == 0.0:
        return np.zeros(n)
    return np.sum((u[:, :r] ** 2) * (s[:r] ** 2)[None, :], axis=1) / energy


def block_scores(keys: np.ndarray, values: np.ndarray, m: int, rank_cap: int):
    """Leverage of every row after appending m rows, for one (b, h).

    Returns (l [n], attn [n], singular values s of W). Very large blocks use
    the query-by-query form of the attention (same values, bounded memory:
    the matrix form holds three m x n fp64 arrays).
    """
    n = keys.shape[0]
    attn = proxy_attention(keys, m) if m * n > 1.1e8 else proxy_attention_block(keys, m)
    w = attn[:, None] * to_f64(values)
    l = leverage(w, rank_cap)
    s = np.linalg.svd(w, compute_uv=False)
    return l, attn, s


def cumulative(cum_old: np.ndarray, l: np.ndarray) -> np.ndarray:
    """Existing rows accumulate their leverage; new rows are seeded with it."""
    k = cum_old.shape[-1]
    return np.concatenate([cum_old + l[:k], l[k:]])
