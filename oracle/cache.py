"""The per-layer eviction cache: update_and_fetch, offset and byte stats.

Test infrastructure only.

One ``OracleCache`` stands for one attention layer's cache ("single-layer,
no coordinator" on all three pages). Per call (block of m tokens):

1. Concatenate the incoming K/V after the kept rows (all pages,
   §How it works); assign absolute positions offset + [0, m) unless given.
2. Score: KNorm norm / Q-Filters projection of the incoming keys, once;
   CurDKV proxy attention + leverage over the whole concatenation,
   accumulated into the kept rows' cumulative score; H2O the proxy
   attention mass (new rows seeded with 0, ``h2o.py``), accumulated alike.
3. If the concatenation exceeds the budget, keep the protected top-k
   (``select.kept_indices``); otherwise keep everything.
4. Compact in temporal order: K/V bits, positions (never renumbered —
   "Q-Filters", §Adaptation notes) and scores are gathered unchanged.
5. offset += m: the true absolute position, not the retained row count
   ("Q-Filters", §RoPE positions had to be fixed first; "L2Norm",
   §RoPE positions had to be fixed too).

Byte accounting ("L2Norm", §How it works; "Q-Filters", §How it works;
"CurDKV-adapted", §Byte accounting): kept_bytes counts the retained K+V in
their storage format (plus, for Q-Filters, the frozen filter: D * 4 bytes
per KV head); full_seq_bytes is the cost had every token been kept;
compression_ratio = full_seq_bytes / kept_bytes.

Key-SVD fallback ("Q-Filters", §How it works step 2, §Key-SVD fallback,
§Path dependence): Q-Filters without calibrated filters keeps every row
(no filter, so no eviction, even over budget) while the keys seen stay below
calib_tokens. The call whose block reaches calib_tokens estimates, per
(b, h), the filter from all keys present then (calibrate.key_svd_filter),
freezes it, scores every stored row once with it, and evicts as usual.
Which keys are present at that call depends on the chunking, which is the
path dependence the page describes. Reading: each (b, h) freezes its own
filter (the page's per-group filter freezing) and the byte accounting
counts those filters (D * 4 bytes per (b, h)) once frozen.

Build-time validation ("Q-Filters", §Evidence: n_sink + recent >= budget
and an invalid sign raise; filters whose head layout disagrees with the
layer raise).
"""
import numpy as np

from . import calibrate as _calibrate
from . import curdkv as _curdkv
from . import h2o as _h2o
from . import scores as _scores
from .bf16 import to_f64
from .select import gather_rows, kept_indices, kept_indices_argmin, priority

KNORM, QFILTERS, CURDKV, H2O = "knorm", "qfilters", "curdkv", "h2o"


class OracleCache:
    def __init__(self, method, batch, n_kv_heads, budget, n_sink=4, recent=0, keep_low=True,
                 sign=1, filters=None, rank_cap=16, head_dim=128, dtype="bf16", score_mode="canonical",
                 calib_tokens=128, per_token=False):
        if method not in (KNORM, QFILTERS, CURDKV, H2O):
            raise ValueError(f"unknown method {method}")
        if n_sink < 0 or recent < 0 or budget <= 0:
            raise ValueError("budget must be positive, n_sink and recent non-negative")
        if n_sink + recent >= budget:
            raise ValueError("n_sink + recent must be below the budget")
        if sign not in (1, -1):
            raise ValueError("sign must be +1 or -1")
        self.fallback = method == QFILTERS and filters is None
        if method == QFILTERS and not self.fallback:
            filters = np.asarray(filters, dtype=np.float32)
            if filters.shape != (n_kv_heads, head_dim):
                raise ValueError("filter head layout does not match the layer")
        if self.fallback and calib_tokens < 1:
            raise ValueError("calib_tokens must be >= 1")
        if method == CURDKV and rank_cap <= 0:
            raise ValueError("rank_cap must be positive")
        if per_token and method not in (CURDKV, H2O):
            raise ValueError("per-token mode is for CurDKV and H2O")
        self.per_token = per_token
        self.method, self.batch, self.heads, self.d = method, batch, n_kv_heads, head_dim
        self.budget, self.n_sink, self.recent = budget, n_sink, recent
        self.keep_low, self.sign, self.filters, self.rank_cap = keep_low, sign, filters, rank_cap
        self.dtype, self.score_mode = dtype, score_mode
        sdt = np.uint16 if dtype == "bf16" else np.float32
        self.k = np.zeros((batch, n_kv_heads, 0, head_dim), sdt)
        self.v = np.zeros((batch, n_kv_heads, 0, head_dim), sdt)
        self.pos = np.zeros((batch, n_kv_heads, 0), np.int32)
        sc = np.float64 if method in (CURDKV, H2O) else (np.float32 if score_mode == "canonical" else np.float64)
        self.score = np.zeros((batch, n_kv_heads, 0), sc)
        self.offset = 0
        self.last_kept = None          # indices kept by the last call, [B, H, n_kept]
        self.last_leverage = None      # CurDKV: leverage of the last call's rows
        self.calib_tokens = calib_tokens
        self.filters_bh = None         # fallback: frozen per-(b, h) filters [B, H, D] fp32

    # ------------------------------------------------------------------
    def set_state(self, k, v, pos, score, offset):
        """Load a pre-existing kept set (same layout as the kept arrays)."""
        self.k, self.v = np.array(k), np.array(v)
        self.pos = np.array(pos, dtype=np.int32)
        self.score = np.array(score, dtype=self.score.dtype)
        self.offset = int(offset)

    @property
    def n_kept(self) -> int:
        return self.k.shape[2]

    def _project(self, k, filters_bh):
        """Canonical fp32 projection of k [B, H, n, D] onto per-(b, h) filters."""
        return np.concatenate([_scores.projection_canonical(k[b:b + 1], filters_bh[b], self.sign)
                               for b in range(self.batch)], axis=0)

    def _freeze(self, k_all):
        """Fallback: estimate and freeze every (b, h)'s filter from the keys present."""
        f = np.empty((self.batch, self.heads, self.d), np.float32)
        for b in range(self.batch):
            for h in range(self.heads):
                f[b, h] = _calibrate.key_svd_filter(k_all[b, h]).astype(np.float32)
        self.filters_bh = f

    def _score_new(self, k_new):
        if self.fallback:
            return self._project(k_new, self.filters_bh)
        if self.method == KNORM:
            if self.score_mode == "canonical":
                return _scores.key_norm_canonical(k_new)
            return _scores.key_norm_plain(k_new)
        if self.score_mode == "canonical":
            return _scores.projection_canonical(k_new, self.filters, self.sign)
        return _scores.projection_plain(k_new, self.filters, self.sign)

    def update_and_fetch(self, k_new, v_new, pos=None):
        """Absorb one block [B, H, m, D]; return (K, V, pos, score) kept arrays.

        Per-token mode (CurDKV, H2O): the block is absorbed one token at a
        time, each an m = 1 call whose single eviction takes the argmin rule
        ("CurDKV-adapted", §How it works: every incoming token goes through
        steps 1-5, prefill and decode alike).
        """
        m = k_new.shape[2]
        if m == 0:
            return self.k, self.v, self.pos, self.score
        if self.per_token and m > 1:
            for t in range(m):
                self.update_and_fetch(k_new[:, :, t:t + 1], v_new[:, :, t:t + 1],
                                      None if pos is None else np.asarray(pos)[:, t:t + 1])
            return self.k, self.v, self.pos, self.score
        if pos is None:
            pos_new = np.broadcast_to(self.offset + np.arange(m, dtype=np.int64),
                                      (self.batch, self.heads, m)).astype(np.int32)
        else:
            pos_new = np.broadcast_to(np.asarray(pos, np.int32)[:, None, :], (self.batch, self.heads, m))
        k_all = np.concatenate([self.k, k_new], axis=2)
        v_all = np.concatenate([self.v, v_new], axis=2)
        pos_all = np.concatenate([self.pos, pos_new], axis=2)
        if self.method == CURDKV:
            score_all = np.empty(k_all.shape[:3])
            self.last_leverage = np.empty(k_all.shape[:3])
            for b in range(self.batch):
                for h in range(self.heads):
                    l, _, _ = _curdkv.block_scores(k_all[b, h], v_all[b, h], m, self.rank_cap)
                    self.last_leverage[b, h] = l
                    score_all[b, h] = _curdkv.cumulative(self.score[b, h], l)
            prio = priority(score_all, keep_low=False)
        elif self.method == H2O:
            score_all = np.empty(k_all.shape[:3])
            self.last_mass = np.empty(k_all.shape[:3])
            for b in range(self.batch):
                for h in range(self.heads):
                    mass = _h2o.proxy_mass(k_all[b, h], m)
                    self.last_mass[b, h] = mass
                    score_all[b, h] = _h2o.cumulative(self.score[b, h], mass)
            prio = priority(score_all, keep_low=False)
        elif self.fallback and self.filters_bh is None:
            if self.offset + m < self.calib_tokens:
                # no filter yet: keep everything (placeholder scores, replaced at the freeze)
                self.k, self.v, self.pos = k_all, v_all, pos_all
                self.score = np.zeros(k_all.shape[:3], np.float32)
                self.last_kept = np.broadcast_to(np.arange(k_all.shape[2]), k_all.shape[:3])
                self.offset += m
                return self.k, self.v, self.pos, self.score
            self._freeze(k_all)
            score_all = self._project(k_all, self.filters_bh)
            prio = priority(score_all, keep_low=False)
        else:
            score_all = np.concatenate([self.score, self._score_new(k_new).astype(self.score.dtype)], axis=2)
            prio = priority(score_all, keep_low=(self.method == KNORM and self.keep_low))
        self.last_scores = score_all           # every row's score before this call's selection
        self.last_rows = (k_all, v_all, pos_all)   # the concatenation this call selected from
        select = kept_indices_argmin if self.per_token else kept_indices
        idx = select(prio, self.n_sink, self.recent, self.budget)
        self.last_kept = idx
        self.k, self.v = gather_rows(k_all, idx), gather_rows(v_all, idx)
        self.pos, self.score = gather_rows(pos_all, idx), gather_rows(score_all, idx)
        self.offset += m
        return self.k, self.v, self.pos, self.score

    # ------------------------------------------------------------------
    def stats(self):
        e = self.k.dtype.itemsize
        per_token = self.batch * self.heads * 2 * self.d * e
        kept = per_token * self.n_kept
        if self.method == QFILTERS and not self.fallback:
            kept += self.heads * self.d * 4
        elif self.fallback and self.filters_bh is not None:
            kept += self.batch * self.heads * self.d * 4
        full = per_token * self.offset
        return {
            "tokens_seen": self.offset,
            "tokens_kept": self.n_kept,
            "kept_bytes": kept,
            "full_seq_bytes": full,
            "compression_ratio": (full / kept) if kept else 0.0,
            "offset": self.offset,
        }


def keys_f64(x):
    """Convenience for tests: storage array -> fp64."""
    return to_f64(x)
