"""Pins for the oracle's scores and protected top-k (CPU only).

Each test checks the oracle against something other than itself: a value
derived by hand from the stated evaluation order, a closed form, brute force
on tiny inputs, or a property the pages fix.
"""
import itertools
import json
import os

import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import synth
from oracle import scores, select

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _key_from(nonzero):
    k = np.zeros((1, 1, 1, 128), np.float32)
    for d, x in nonzero.items():
        k[0, 0, 0, int(d)] = x
    return k


# --------------------------------------------------------------------- scores
def test_canonical_order_pins_golden():
    g = json.load(open(os.path.join(GOLDEN, "canonical_sum.json")))
    k = _key_from(g["within_chunk"]["nonzero"])
    s = scores._canonical_sum(k * k)
    assert s.item() == g["within_chunk"]["expected_sum"]
    assert scores.key_norm_canonical(k).item() == g["within_chunk"]["expected_norm"]
    # the fp64 definition differs (sqrt(2^24 + 7)): the order is what is pinned
    assert scores.key_norm_plain(k).item() > 4096.0
    k2 = _key_from(g["across_chunks"]["nonzero"])
    assert scores._canonical_sum(k2 ** 2).item() == g["across_chunks"]["expected_sum"]


def test_knorm_onehot_is_exact():
    # a one-hot key has norm |x| exactly, for every coordinate and sign
    g = synth.rng(11)
    vals = synth.f32_to_bf16_bits(g.standard_normal(128).astype(np.float32))
    k = np.zeros((1, 1, 128, 128), np.uint16)
    for d in range(128):
        k[0, 0, d, d] = vals[d]
    got = scores.key_norm_canonical(k)[0, 0]
    want = np.abs(synth.bf16_bits_to_f32(vals))
    assert np.array_equal(got, want)


def test_knorm_canonical_close_to_definition():
    k, _ = synth.gaussian_block(5, 2, 3, 257, dtype="bf16", scale=3.0)
    c = scores.key_norm_canonical(k).astype(np.float64)
    p = scores.key_norm_plain(k)
    assert np.all(np.abs(c - p) <= 4e-6 * p)


def test_knorm_constant_key_closed_form():
    # all 128 entries equal c: ||k|| = |c| * sqrt(128) = |c| * 8 * sqrt(2)
    for c in (0.5, -1.25, 3.0):
        k = np.full((1, 1, 1, 128), c, np.float32)
        got = scores.key_norm_canonical(k).item()
        assert abs(got - abs(c) * 8 * np.sqrt(2.0)) <= 1e-6 * abs(c) * 11.4


def test_knorm_subnormal_squares_kept():
    # squares of 2^-70 are 2^-140 (subnormal in fp32); flushing would give 0
    k = np.full((1, 1, 1, 128), 2.0 ** -70, np.float32)
    got = scores.key_norm_canonical(k).item()
    assert got > 0
    assert abs(got - 2.0 ** -70 * np.sqrt(128)) <= 0.05 * 2.0 ** -70 * np.sqrt(128)


def test_projection_axis_filter_is_exact():
    # filter = e_d: the score is sign * k_d exactly
    k, _ = synth.gaussian_block(7, 1, 2, 64, dtype="bf16")
    for sign in (1, -1):
        for d in (0, 77, 127):
            f = np.zeros((2, 128), np.float32)
            f[:, d] = 1.0
            got = scores.projection_canonical(k, f, sign)
            want = sign * synth.bf16_bits_to_f32(k[..., d])
            assert np.array_equal(got, want)


def test_projection_close_to_definition():
    k, _ = synth.gaussian_block(8, 2, 4, 300, dtype="bf16")
    f = synth.unit_vectors(synth.rng(3), 4).astype(np.float32)
    c = scores.projection_canonical(k, f, 1).astype(np.float64)
    p = scores.projection_plain(k, f, 1)
    cond = scores.projection_condition(k, f)
    assert np.all(np.abs(c - p) <= 1e-5 * np.maximum(np.abs(p), cond))
    assert np.array_equal(scores.projection_canonical(k, f, -1), -scores.projection_canonical(k, f, 1))


def test_score_depends_only_on_the_key():
    # the same key in different blocks / batches / positions gets the same bits
    k, _ = synth.gaussian_block(9, 2, 2, 50, dtype="bf16")
    full = scores.key_norm_canonical(k)
    part = scores.key_norm_canonical(k[:, :, 17:18])
    assert np.array_equal(full[:, :, 17:18], part)
    swapped = scores.key_norm_canonical(k[::-1, ::-1])
    assert np.array_equal(swapped[::-1, ::-1], full)


# ------------------------------------------------------------------ selection
_TIE_VALUES = np.array([0.0, -0.0, 1.0, 1.0, -1.0, 2.0, np.inf, -np.inf, np.nan], np.float32)


def test_selection_matches_bruteforce_on_tiny_inputs():
    g = synth.rng(21)
    checked = 0
    for n in range(1, 11):
        for budget in range(1, n + 2):
            for n_sink, recent in itertools.product(range(0, 3), range(0, 3)):
                if n_sink + recent >= budget:
                    continue
                for _ in range(6):
                    s = g.choice(_TIE_VALUES, size=n)
                    for keep_low in (False, True):
                        p = select.priority(s, keep_low)
                        got = select.kept_indices(p[None, None], n_sink, recent, budget)[0, 0]
                        want = select.kept_indices_bruteforce(p, n_sink, recent, budget)
                        assert np.array_equal(got, want), (s, n_sink, recent, budget, keep_low)
                        checked += 1
    assert checked > 1000


def test_kept_set_is_budget_lowest_norms_in_temporal_order():
    # L2Norm page, Evidence: kept set = budget lowest-norm positions, temporal order
    k, _ = synth.gaussian_block(31, 1, 1, 300, dtype="fp32")
    norms = scores.key_norm_canonical(k)[0, 0]
    budget = 40
    idx = select.kept_indices(select.priority(norms, keep_low=True)[None, None], 0, 0, budget)[0, 0]
    thresh = np.sort(norms)[budget - 1]
    assert len(idx) == budget and np.all(np.diff(idx) > 0)
    assert np.all(norms[idx] <= thresh)
    assert np.sum(norms < thresh) < budget
    # keep="high" mirrors it
    hi = select.kept_indices(select.priority(norms, keep_low=False)[None, None], 0, 0, budget)[0, 0]
    assert np.all(norms[hi] >= np.sort(norms)[-budget])


def test_sinks_survive_with_the_highest_norms():
    k, _ = synth.gaussian_block(32, 1, 1, 100, dtype="fp32")
    k[0, 0, :4] *= 50.0                       # sinks get the largest norms
    norms = scores.key_norm_canonical(k)[0, 0]
    idx = select.kept_indices(select.priority(norms, True)[None, None], 4, 0, 20)[0, 0]
    assert set(range(4)) <= set(idx.tolist()) and len(idx) == 20


def test_recent_window_survives():
    # keep-low on increasing scores prefers the oldest rows; the trailing
    # window must survive anyway
    s = np.arange(30, dtype=np.float32)
    idx = select.kept_indices(select.priority(s, True)[None, None], 2, 5, 10)[0, 0]
    assert idx.tolist() == [0, 1, 2, 3, 4, 25, 26, 27, 28, 29]


def test_all_equal_scores_keep_exactly_budget_lowest_indices():
    # Q-Filters page, Metal kernels: ties never overflow the budget
    for val in (1.5, np.inf, -np.inf, 0.0):
        s = np.full(50, val, np.float32)
        idx = select.kept_indices(select.priority(s)[None, None], 3, 4, 20)[0, 0]
        assert len(idx) == 20
        assert idx.tolist() == list(range(16)) + list(range(46, 50))


def test_nan_is_evicted_first_and_signed_zeros_tie():
    s = np.array([np.nan, -0.0, 0.0, np.nan, -0.0, 1.0], np.float32)
    idx = select.kept_indices(select.priority(s)[None, None], 0, 0, 3)[0, 0]
    assert idx.tolist() == [1, 2, 5]


def test_bf16_rounding_of_inputs_is_nearest_even():
    # input generation sanity: ties round to even, NaN stays NaN
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, np.nan, np.inf], np.float32)
    b = synth.f32_to_bf16_bits(x)
    back = synth.bf16_bits_to_f32(b)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.0 + 2 ** -6
    assert back[3] == -2.5 and np.isnan(back[4]) and back[5] == np.inf
