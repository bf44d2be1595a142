"""CPU oracle for per-block KV-cache token eviction — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct numpy restatement of what the eviction path
computes, written from three documentation pages:

* "Q-Filters — Query-Agnostic Projection Eviction" (§How it works,
  §Calibrated — the paper's actual mechanism, §Metal kernels),
* "L2Norm — Intrinsic Key-Norm Eviction" (§How it works),
* "CurDKV-adapted — Value-Aware Leverage-Score Eviction" (§The honesty
  crux, §How it works).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package. The product
path (the C-ABI library and its Python binding) never imports it and shares
no code with it; the seeded input generators live in a module of their own.

Modules
-------
``bf16``       bf16 bit patterns -> float32 (exact widening).
``scores``     KNorm and Q-Filters scores: plain fp64 definitions and the
               canonical fp32 evaluation order.
``select``     priority, protection, protected top-k with lower-index tie
               break, order-preserving compaction.
``curdkv``     key-as-query proxy attention, weighted values, energy-weighted
               leverage by explicit SVD, cumulative update.
``calibrate``  uncentered query SVD filter, sign fix, GQA averaging.
``cache``      the per-layer cache: update_and_fetch, offset, byte stats.

Readings of the pages taken where they are silent or ambiguous are listed in
each function's docstring. Every function is pinned by ``tests/`` against
closed forms, invariants, brute force on tiny inputs or values the pages
print; none is "parity unpinned".
"""
from . import bf16, scores, select, curdkv, calibrate, cache  # noqa: F401
