"""H2O-adapted block scoring: cumulative proxy-attention mass.

Test infrastructure only.

Sources: "CurDKV-adapted — Value-Aware Leverage-Score Eviction", §How it works
step 1 (each incoming key stands in for the query, and its softmax over the
stored keys is the one H2O scores with) and §The honesty crux, item 4 (under
H2O a token starts from a score of zero when it is appended and gathers mass
only from later steps); "L2Norm — Intrinsic Key-Norm Eviction" and
"Q-Filters — Query-Agnostic Projection Eviction", the method tables (H2O ranks
a token by the proxy attention it has accumulated); "Q-Filters",
§Integration (H2O runs with only a budget and sinks: its accumulated score is
already biased toward recent tokens, so no trailing window is added).

Readings (the pages describe one token at a time; the cache here takes a
block of m tokens per call, as for CurDKV):
* Query t of the block (row k+t of the concatenation) attends rows i <= k+t
  (causal, itself included in the softmax) with the 1/sqrt(D) logit scale:
  the same proxy softmax as the CurDKV oracle.
* Row i's mass increment is the sum of the weights the queries put on it,
  EXCEPT a new row's weight from its own query: at its own step a token is
  seeded with 0, so it only gathers mass from the queries after it. With
  m = 1 this is exactly the per-token step; a block equals m single-token
  calls whenever none of them would have evicted.
* Existing rows add the increment to their cumulative score; new rows start
  from the increment (0 plus what the later queries of the block gave them).
* Everything in fp64; the softmax subtracts each query's maximum.
"""
import numpy as np

from .bf16 import to_f64


def proxy_mass(keys: np.ndarray, m: int) -> np.ndarray:
    """Mass increment of every row for one (b, h); ``keys`` [n, D], the last m rows are the queries."""
    x = to_f64(keys)
    n, d = x.shape
    k = n - m
    mass = np.zeros(n)
    for t in range(m):
        row = k + t
        logits = x[: row + 1] @ x[row] / np.sqrt(d)
        logits -= logits.max()
        p = np.exp(logits)
        p /= p.sum()
        mass[:row] += p[:row]          # the query's own row is seeded with 0, not its self weight
    return mass


def cumulative(cum_old: np.ndarray, mass: np.ndarray) -> np.ndarray:
    """Existing rows accumulate their mass; new rows start from theirs."""
    k = cum_old.shape[-1]
    return np.concatenate([cum_old + mass[:k], mass[k:]])
