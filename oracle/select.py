"""Protected top-k selection and order-preserving compaction.

Test infrastructure only.

Sources
-------
* "Q-Filters — Query-Agnostic Projection Eviction", §How it works step 4:
  over budget, keep the budget highest-scoring positions in one top-k with
  the first n_sink positions and the optional trailing recent window forced
  to survive; kept tokens keep their temporal order.
* Same page, §Metal kernels (the tie trap): rows strictly above the
  threshold are always admitted, rows equal to it only while quota remains,
  lowest index first — never more than budget rows.
* "L2Norm — Intrinsic Key-Norm Eviction", §How it works step 3: keep the
  budget lowest-norm positions ("high" inverts the ranking), same
  protection, temporal order kept.
* "CurDKV-adapted", §How it works step 5: sinks protected, lowest
  cumulative score evicted (here lifted to the same block top-k).

Readings
--------
* Priority (higher = keep): Q-Filters and CurDKV use the score; KNorm
  keep-low uses -score, keep-high the score.
* -0 is treated as +0 and NaN as -inf (evicted first): the pages are silent
  and a raw bit order would split +-0 ties.
* Protected rows are always kept; they are not encoded as +inf scores, so
  a genuine +inf score never competes with a protected row.
* Ties between unprotected rows keep the LOWER index, for every scorer
  (the tie rule of the Q-Filters page; the CurDKV page's per-token argmin
  would break a tie the other way).
"""
import numpy as np


def priority(score: np.ndarray, keep_low: bool = False) -> np.ndarray:
    """Canonical priority: +-score with -0 -> +0 and NaN -> -inf."""
    p = -score if keep_low else score.copy()
    p = np.where(np.isnan(p), -np.inf, p)
    p = np.where(p == 0, 0.0, p).astype(score.dtype)   # -0 -> +0
    return p


def protected_mask(n: int, n_sink: int, recent: int) -> np.ndarray:
    """Rows i < n_sink or i >= n - recent are protected (always kept)."""
    i = np.arange(n)
    return (i < n_sink) | (i >= n - recent)


def kept_indices(prio: np.ndarray, n_sink: int, recent: int, budget: int) -> np.ndarray:
    """Indices kept from ``n`` concatenated rows, ascending (temporal order).

    ``prio`` is [..., n]. Returns an int64 array [..., min(n, budget)].
    Over budget: all protected rows, plus the q = budget - |protected|
    unprotected rows that come first when sorted by priority descending and
    then index ascending.
    """
    n = prio.shape[-1]
    lead = prio.shape[:-1]
    if n <= budget:
        return np.broadcast_to(np.arange(n), lead + (n,)).copy()
    lo, hi = n_sink, n - recent                  # the unprotected rows are [lo, hi)
    q = budget - (n - (hi - lo))
    assert q > 0
    sub = prio[..., lo:hi]
    order = np.argsort(-sub, axis=-1, kind="stable")    # stable: ties keep index order
    chosen = lo + order[..., :q]
    prot = np.broadcast_to(np.concatenate([np.arange(lo), np.arange(hi, n)]), lead + (n - (hi - lo),))
    return np.sort(np.concatenate([prot, chosen], axis=-1), axis=-1)


def kept_indices_argmin(prio: np.ndarray, n_sink: int, recent: int, budget: int) -> np.ndarray:
    """Per-token eviction ("CurDKV-adapted", §How it works step 5): when the
    rows exceed the budget by one, the unprotected row of lowest priority
    leaves; on equal priorities the first one (numpy's argmin). Protected
    rows count as +inf. Any other row count falls back to ``kept_indices``.
    """
    n = prio.shape[-1]
    if n != budget + 1:
        return kept_indices(prio, n_sink, recent, budget)
    p = np.where(protected_mask(n, n_sink, recent), np.inf, prio)
    e = np.argmin(p, axis=-1)
    idx = np.broadcast_to(np.arange(n), prio.shape)
    return idx[idx != e[..., None]].reshape(prio.shape[:-1] + (budget,))


def kept_indices_bruteforce(prio: np.ndarray, n_sink: int, recent: int, budget: int) -> np.ndarray:
    """Same selection by pairwise counting on one (b, h) row (tiny n only).

    Unprotected row i is kept iff fewer than q unprotected rows beat it,
    where j beats i when prio_j > prio_i, or prio_j == prio_i and j < i.
    """
    n = prio.shape[-1]
    if n <= budget:
        return np.arange(n)
    prot = protected_mask(n, n_sink, recent)
    q = budget - int(prot.sum())
    keep = []
    for i in range(n):
        if prot[i]:
            keep.append(i)
            continue
        beaten_by = 0
        for j in range(n):
            if prot[j] or j == i:
                continue
            if prio[j] > prio[i] or (prio[j] == prio[i] and j < i):
                beaten_by += 1
        if beaten_by < q:
            keep.append(i)
    return np.array(keep, dtype=np.int64)


def gather_rows(x: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Gather along the token axis (axis 2) per (b, h): x[b, h, idx[b, h]]."""
    if x.ndim == 4:
        return np.take_along_axis(x, idx[..., None], axis=2)
    return np.take_along_axis(x, idx, axis=2)
