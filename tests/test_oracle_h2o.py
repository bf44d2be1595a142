"""Pins of the oracle's H2O-adapted scorer (cumulative proxy-attention mass).

"CurDKV-adapted — Value-Aware Leverage-Score Eviction", §How it works step 1
(the proxy softmax H2O uses), §The honesty crux item 4 (a new token starts
from exactly 0), §The planted-geometry observable (H2O, given identical keys,
cannot tell value-relevant from negligible-value tokens).
"""
import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import synth
from oracle import h2o
from oracle.cache import OracleCache


def _harmonic(a, b):
    """sum_{j=a+1}^{b} 1/j"""
    return sum(1.0 / j for j in range(a + 1, b + 1))


@pytest.mark.parametrize("k,m", [(0, 1), (0, 7), (5, 1), (9, 6), (30, 30)])
def test_identical_keys_harmonic_mass(k, m):
    # equal logits: query t spreads 1/(k+t+1) over rows <= k+t; its own weight is not kept
    key = synth.f32_to_bf16_bits(np.linspace(-1, 1, 128).astype(np.float32))
    keys = np.tile(key, (k + m, 1))
    mass = h2o.proxy_mass(keys, m)
    for i in range(k):
        assert mass[i] == pytest.approx(_harmonic(k, k + m), rel=1e-12)
    for s in range(m):
        assert mass[k + s] == pytest.approx(_harmonic(k + s + 1, k + m), rel=1e-12, abs=1e-15)
    assert mass[-1] == 0.0                          # the last token is seeded with exactly 0


def test_orthogonal_keys_closed_form():
    # one-hot keys a_i e_i: a query's logit is a^2/sqrt(D) on itself and 0 elsewhere
    n, m, d = 12, 5, 128
    a = np.linspace(0.5, 3.0, n)
    keys = synth.f32_to_bf16_bits((np.eye(n, d) * a[:, None]).astype(np.float32))
    a = synth.bf16_bits_to_f32(keys).astype(np.float64).sum(axis=1)      # the bf16-rounded scales
    mass = h2o.proxy_mass(keys, m)
    k = n - m
    want = np.zeros(n)
    for t in range(m):
        row = k + t
        z = np.exp(a[row] ** 2 / np.sqrt(d)) + row                       # self weight plus `row` others of logit 0
        want[:row] += 1.0 / z
    assert np.allclose(mass, want, rtol=1e-12, atol=0)


def test_block_equals_single_token_calls_without_eviction():
    k_all, v_all = synth.gaussian_block(5, 1, 2, 90)
    one = OracleCache("h2o", 1, 2, budget=200, n_sink=4)
    one.update_and_fetch(k_all[:, :, :40], v_all[:, :, :40])
    one.update_and_fetch(k_all[:, :, 40:], v_all[:, :, 40:])
    seq = OracleCache("h2o", 1, 2, budget=200, n_sink=4)
    for t in range(90):
        seq.update_and_fetch(k_all[:, :, t:t + 1], v_all[:, :, t:t + 1])
    # the first block's queries see each other causally, as the single-token calls do
    assert np.allclose(one.score, seq.score, rtol=1e-12, atol=1e-15)


def test_mass_budget_and_scores():
    k_all, v_all = synth.gaussian_block(6, 2, 2, 150)
    c = OracleCache("h2o", 2, 2, budget=48, n_sink=4)
    for a in range(0, 150, 25):
        before = c.n_kept
        c.update_and_fetch(k_all[:, :, a:a + 25], v_all[:, :, a:a + 25])
        m = c.last_mass
        # each query's weights sum to 1: the mass handed out is m minus the self weights
        assert np.all(m >= 0) and np.all(m.sum(axis=-1) < 25 + 1e-9)
        assert np.all(m[..., -1] == 0.0)
        assert c.n_kept == min(before + 25, 48)
    assert c.offset == 150 and np.all(c.pos[..., :4] == np.arange(4))


def test_h2o_is_blind_to_values_on_the_planted_geometry():
    rates_h2o, rates_cd = [], []
    for seed in range(8):
        p = synth.curdkv_planted(batch=1, n_kv_heads=1, existing=240, incoming=16, seed=1000 + seed)
        kept = {}
        for method, vals in (("h2o", p["v"]), ("h2o_swapped", p["v"][:, :, ::-1].copy()), ("curdkv", p["v"])):
            c = OracleCache("h2o" if method.startswith("h2o") else "curdkv", 1, 1, budget=24, n_sink=4,
                            rank_cap=16)
            c.set_state(p["k"][:, :, :240], vals[:, :, :240], np.arange(240, dtype=np.int32)[None, None],
                        np.zeros((1, 1, 240)), 240)
            c.update_and_fetch(p["k"][:, :, 240:], vals[:, :, 240:])
            kept[method] = c.last_kept[0, 0]
        # H2O scores keys only: any values give the same kept set
        assert np.array_equal(kept["h2o"], kept["h2o_swapped"])
        rates_h2o.append(np.mean(p["cls"][0, 0, kept["h2o"][4:]] == 2))
        rates_cd.append(np.mean(p["cls"][0, 0, kept["curdkv"][4:]] == 2))
    assert max(rates_cd) == 0.0                           # CurDKV keeps only value-relevant tokens
    assert 0.2 < np.mean(rates_h2o) < 0.8                 # H2O keeps both classes
