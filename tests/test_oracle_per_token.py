"""Pins of the oracle's per-token mode for CurDKV and H2O.

"CurDKV-adapted — Value-Aware Leverage-Score Eviction", §How it works: every
incoming token goes through steps 1-5; step 5 evicts the lowest-cumulative
non-sink token (argmin: on equal scores the first one) with the sinks
protected as +inf. The brute-force loops below restate those steps directly
(one token at a time, a full SVD per step, an explicit argmin).
"""
import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import synth
from oracle.bf16 import to_f64
from oracle.cache import OracleCache


def _softmax_row(x, q):
    z = x @ q / np.sqrt(x.shape[1])
    z = np.exp(z - z.max())
    return z / z.sum()


def _bruteforce(method, keys, vals, budget, n_sink, rank):
    """The pages' loop for one (b, h): returns (kept token indices, cumulative scores)."""
    K, V = to_f64(keys), to_f64(vals)
    kept, cum = [], []
    for t in range(len(K)):
        kept.append(t)
        rows = np.array(kept)
        a = _softmax_row(K[rows], K[t])                   # the new key against every stored key
        if method == "curdkv":
            w = a[:, None] * V[rows]
            u, s, _ = np.linalg.svd(w, full_matrices=False)
            r = min(rank, len(rows), w.shape[1])
            energy = np.sum(s ** 2)
            gain = np.zeros(len(rows)) if energy == 0 else (u[:, :r] ** 2 @ s[:r] ** 2) / energy
            cum = [c + g for c, g in zip(cum, gain[:-1])] + [gain[-1]]   # the new token seeded with its own
        else:
            cum = [c + g for c, g in zip(cum, a[:-1])] + [0.0]           # H2O: the new token starts at 0
        if len(kept) > budget:
            guarded = np.array(cum, dtype=float)
            guarded[:n_sink] = np.inf
            e = int(np.argmin(guarded))
            del kept[e], cum[e]
    return np.array(kept), np.array(cum)


@pytest.mark.parametrize("method", ["curdkv", "h2o"])
@pytest.mark.parametrize("seed", range(3))
def test_per_token_mode_is_the_pages_loop(method, seed):
    B, H, S, budget = 1, 2, 40, 12
    keys = synth.clustered_keys(500 + seed, B, H, S, spread=0.8)
    vals = synth.planted_spectrum_values(600 + seed, B, H, S, rank=4)
    c = OracleCache(method, B, H, budget=budget, n_sink=2, rank_cap=4, per_token=True)
    c.update_and_fetch(keys[:, :, :25], vals[:, :, :25])          # one call, absorbed token by token
    c.update_and_fetch(keys[:, :, 25:], vals[:, :, 25:])
    for h in range(H):
        kept, cum = _bruteforce(method, keys[0, h], vals[0, h], budget, 2, 4)
        assert np.array_equal(c.pos[0, h], kept)
        assert np.allclose(c.score[0, h], cum, rtol=1e-9, atol=1e-15)


def test_tie_rules_on_zero_values():
    # zero values: every leverage is 0. The per-token argmin evicts the oldest non-sink each
    # step; the block rule keeps the lower index, so a full cache evicts the newcomer.
    B, H, S, budget, sinks = 1, 1, 30, 10, 3
    keys = synth.gaussian_block(7, B, H, S)[0]
    vals = np.zeros_like(keys)
    per = OracleCache("curdkv", B, H, budget=budget, n_sink=sinks, per_token=True)
    per.update_and_fetch(keys, vals)
    assert per.pos[0, 0].tolist() == list(range(sinks)) + list(range(S - (budget - sinks), S))
    blk = OracleCache("curdkv", B, H, budget=budget, n_sink=sinks)
    for t in range(S):
        blk.update_and_fetch(keys[:, :, t:t + 1], vals[:, :, t:t + 1])
    assert blk.pos[0, 0].tolist() == list(range(budget))


def test_h2o_per_token_equals_block_without_eviction():
    # H2O's mass adds up query by query; CurDKV's block leverage takes one SVD of the whole block,
    # so only H2O's block form equals its token-by-token loop when nothing is evicted
    keys, vals = synth.gaussian_block(8, 1, 2, 50)
    per = OracleCache("h2o", 1, 2, budget=64, n_sink=4, per_token=True)
    blk = OracleCache("h2o", 1, 2, budget=64, n_sink=4)
    per.update_and_fetch(keys, vals)
    blk.update_and_fetch(keys, vals)
    assert np.array_equal(per.pos, blk.pos)
    assert np.allclose(per.score, blk.score, rtol=1e-10, atol=1e-15)


def test_per_token_only_for_attention_scorers():
    with pytest.raises(ValueError):
        OracleCache("knorm", 1, 1, budget=8, per_token=True)
