"""Pins of the oracle's Q-Filters key-SVD fallback.

"Q-Filters — Query-Agnostic Projection Eviction": §Calibrated vs key-SVD
fallback (the filter comes from the SVD of observed keys), §Key-SVD fallback
(it recovers a dominant axis, loses a pure-drift direction: cosine below 0.3),
§How it works step 2 (before calib_tokens keys nothing is evicted; once
enough keys are seen the filter is estimated and frozen), §Path dependence
(the filter depends on which keys are present when the threshold is
crossed; the budget and offset hold at every chunk size), §Evidence
(estimate_filter_dir recovers a planted dominant direction with cosine above
0.99; the kept set is the budget highest projections against the frozen
direction, in temporal order; a stored score never changes once the filter
is set).
"""
import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import synth
from oracle import calibrate as ocal
from oracle import scores as oscores
from oracle import select as osel
from oracle.bf16 import to_f64
from oracle.cache import OracleCache


def _dominant_axis_keys(seed, n, spread=6.0):
    g = synth.rng(seed)
    u = synth.unit_vectors(g, 1)[0]
    k = g.standard_normal((n, 128)) + np.outer(g.normal(0.0, spread, n), u)
    return synth.f32_to_bf16_bits(k.astype(np.float32)), u


def test_key_svd_recovers_a_planted_dominant_axis():
    for seed in range(4):
        k, u = _dominant_axis_keys(seed, 512)
        f = ocal.key_svd_filter(k)
        assert abs(np.linalg.norm(f) - 1.0) < 1e-12
        assert abs(f @ u) > 0.99


def test_key_svd_loses_a_pure_drift_direction_that_query_svd_keeps():
    # drift along u (mean 4, sd 0.5) plus isotropic N(0, 1): centring removes the drift
    g = synth.rng(11)
    u = synth.unit_vectors(g, 1)[0]
    x = g.standard_normal((2000, 128)) + np.outer(g.normal(4.0, 0.5, 2000), u)
    bits = synth.f32_to_bf16_bits(x.astype(np.float32))
    assert abs(ocal.key_svd_filter(bits) @ u) < 0.3
    assert ocal.compute_qfilter(bits) @ u > 0.99          # the uncentred query-side estimator


def test_sign_rule_makes_the_largest_component_positive():
    k, _ = _dominant_axis_keys(5, 300)
    f = ocal.key_svd_filter(k)
    j = int(np.argmax(np.abs(f)))
    assert f[j] > 0
    # the estimate is invariant to negating every key up to that rule
    neg = synth.f32_to_bf16_bits(-to_f64(k).astype(np.float32))
    assert np.allclose(ocal.key_svd_filter(neg), f, atol=1e-9)


def test_passthrough_below_calib_tokens_then_freeze_on_the_present_keys():
    B, H, budget, calib = 1, 2, 16, 100
    k, v = synth.gaussian_block(3, B, H, 200)
    c = OracleCache("qfilters", B, H, budget=budget, n_sink=2, filters=None, calib_tokens=calib)
    c.update_and_fetch(k[:, :, :64], v[:, :, :64])
    assert c.n_kept == 64 and c.filters_bh is None          # over budget, nothing evicted
    c.update_and_fetch(k[:, :, 64:128], v[:, :, 64:128])      # 128 >= 100 keys: freeze on all 128
    assert c.n_kept == budget and c.offset == 128
    for h in range(H):
        f = ocal.key_svd_filter(k[0, h, :128]).astype(np.float32)
        assert np.array_equal(c.filters_bh[0, h], f)
        # kept set = protected rows + budget - 2 highest projections, temporal order
        s = oscores.projection_canonical(k[:, h:h + 1, :128], f[None], 1)[0, 0]
        want = osel.kept_indices(osel.priority(s[None, None]), 2, 0, budget)[0, 0]
        assert np.array_equal(c.last_kept[0, h], want)
    assert c.stats()["kept_bytes"] == B * H * budget * 2 * 128 * 2 + B * H * 128 * 4


def test_stored_scores_never_change_after_the_freeze():
    B, H = 1, 1
    k, v = synth.gaussian_block(4, B, H, 400)
    c = OracleCache("qfilters", B, H, budget=32, n_sink=1, recent=2, filters=None, calib_tokens=50)
    seen = {}
    for a in range(0, 400, 7):
        c.update_and_fetch(k[:, :, a:a + 7], v[:, :, a:a + 7])
        if c.filters_bh is None:
            continue
        for p, s in zip(c.pos[0, 0], c.score[0, 0]):
            assert seen.setdefault(int(p), s.tobytes()) == s.tobytes()


@pytest.mark.parametrize("chunk", [1, 7, 64, 256, 300])
def test_budget_offset_and_unit_filters_at_every_chunk_size(chunk):
    B, H, budget = 2, 2, 40
    k, v = synth.gaussian_block(6, B, H, 300)
    for sign in (1, -1):
        c = OracleCache("qfilters", B, H, budget=budget, n_sink=4, recent=3, filters=None, sign=sign,
                        calib_tokens=128)
        for a in range(0, 300, chunk):
            c.update_and_fetch(k[:, :, a:a + chunk], v[:, :, a:a + chunk])
            assert c.n_kept <= max(budget, min(c.offset, 127))
        assert c.n_kept == budget and c.offset == 300
        assert np.allclose(np.linalg.norm(c.filters_bh.astype(np.float64), axis=-1), 1.0, atol=1e-6)


def test_degenerate_freezes():
    same = np.tile(synth.f32_to_bf16_bits(np.linspace(-1, 1, 128).astype(np.float32)), (5, 1))
    f = ocal.key_svd_filter(same)                       # no variance: the first coordinate axis
    assert f[0] == 1.0 and not np.any(f[1:])
    assert np.array_equal(ocal.key_svd_filter(same[:1]), f)   # a single key is the same case
    bad = same.copy()
    bad[2, 7] = 0x7FC0                                  # bf16 NaN
    with pytest.raises(ValueError):
        ocal.key_svd_filter(bad)
    # two distinct keys: the direction is their difference, normalised and sign-fixed
    two = synth.f32_to_bf16_bits(np.stack([np.eye(128)[3] * 2 - np.eye(128)[9], np.zeros(128)]).astype(np.float32))
    d = np.zeros(128)
    d[3], d[9] = 2.0, -1.0
    assert np.allclose(ocal.key_svd_filter(two), d / np.linalg.norm(d), atol=1e-12)
