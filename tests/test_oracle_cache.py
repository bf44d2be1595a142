"""Pins for the oracle cache: path independence, immutability, offset, stats."""
import json
import os

import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import synth
from oracle import scores
from oracle.cache import OracleCache

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _feed(cache, k, v, chunk):
    s = k.shape[2]
    for a in range(0, s, chunk):
        cache.update_and_fetch(k[:, :, a:a + chunk], v[:, :, a:a + chunk])
    return cache


@pytest.mark.parametrize("chunk", [1, 64, 256])
def test_knorm_one_block_equals_chunked_feed(chunk):
    # L2Norm page, consequence 2 + Evidence: block vs token-by-token bit-identical (recent=0)
    k, v = synth.knorm_single_sequence(1024)
    a = OracleCache("knorm", 1, 1, budget=512, n_sink=4, recent=0, keep_low=True, dtype="fp32")
    a.update_and_fetch(k, v)
    b = _feed(OracleCache("knorm", 1, 1, budget=512, n_sink=4, recent=0, keep_low=True, dtype="fp32"),
              k, v, chunk)
    for x, y in ((a.k, b.k), (a.v, b.v), (a.pos, b.pos), (a.score, b.score)):
        assert x.tobytes() == y.tobytes()
    assert a.offset == b.offset == 1024


@pytest.mark.parametrize("chunk", [1, 256])
def test_calibrated_qfilters_one_block_equals_chunked_feed(chunk):
    # Q-Filters page, one-shot vs incremental: identical K/V and offset
    k, v = synth.gaussian_block(41, 2, 3, 700, dtype="bf16")
    f = synth.unit_vectors(synth.rng(4), 3).astype(np.float32)
    kw = dict(budget=200, n_sink=4, recent=0, sign=1, filters=f)
    a = OracleCache("qfilters", 2, 3, **kw)
    a.update_and_fetch(k, v)
    b = _feed(OracleCache("qfilters", 2, 3, **kw), k, v, chunk)
    assert a.k.tobytes() == b.k.tobytes() and a.v.tobytes() == b.v.tobytes()
    assert np.array_equal(a.pos, b.pos) and a.offset == b.offset


def test_kept_rows_are_original_rows_at_original_positions():
    k, v = synth.gaussian_block(42, 1, 2, 300, dtype="bf16")
    c = OracleCache("knorm", 1, 2, budget=50, n_sink=4, recent=8)
    _feed(c, k, v, 37)
    for h in range(2):
        p = c.pos[0, h]
        assert np.all(np.diff(p) > 0)                     # temporal order
        assert np.array_equal(c.k[0, h], k[0, h, p])      # bit copies, positions not renumbered
        assert np.array_equal(c.v[0, h], v[0, h, p])
        assert list(p[:4]) == [0, 1, 2, 3] and list(p[-8:]) == list(range(292, 300))


def test_stored_scores_never_change():
    # L2Norm page: norm immutability
    k, v = synth.gaussian_block(43, 1, 1, 400, dtype="bf16")
    c = OracleCache("knorm", 1, 1, budget=64, n_sink=4)
    first = {}
    for a in range(0, 400, 25):
        c.update_and_fetch(k[:, :, a:a + 25], v[:, :, a:a + 25])
        for p, s in zip(c.pos[0, 0], c.score[0, 0]):
            first.setdefault(int(p), s.tobytes())
            assert first[int(p)] == s.tobytes()
    want = scores.key_norm_canonical(k)[0, 0]
    assert np.array_equal(c.score[0, 0], want[c.pos[0, 0]])


def test_offset_contract_golden():
    g = json.load(open(os.path.join(GOLDEN, "offset_contract.json")))
    n = g["prefill"] + g["decode_steps"]
    k, v = synth.gaussian_block(44, 1, 1, n, dtype="bf16")
    for method, kw in (("knorm", {}), ("qfilters", {"filters": synth.decode_filters(1)})):
        c = OracleCache(method, 1, 1, budget=g["budget"], n_sink=4, recent=16, **kw)
        c.update_and_fetch(k[:, :, :g["prefill"]], v[:, :, :g["prefill"]])
        assert c.offset == g["prefill"]
        for t in range(g["prefill"], n):
            c.update_and_fetch(k[:, :, t:t + 1], v[:, :, t:t + 1])
            assert c.offset == t + 1                          # zero drift at every step
            assert c.pos[0, 0, -1] == t                       # newest row sits at its true position
        assert c.offset == g["expected_offset"] and c.n_kept == g["expected_kept"]


def test_budget_verification_golden():
    g = json.load(open(os.path.join(GOLDEN, "budget_verification.json")))
    k, v = synth.gaussian_block(45, 1, 2, g["prompt_tokens"], dtype="bf16")
    c = OracleCache("knorm", 1, 2, budget=g["budget"], n_sink=4)
    c.update_and_fetch(k, v)
    assert c.n_kept == g["expected_kept"] and c.offset == g["expected_offset"]


def test_byte_accounting_closed_form():
    k, v = synth.gaussian_block(46, 2, 3, 100, dtype="bf16")
    f = synth.unit_vectors(synth.rng(1), 3).astype(np.float32)
    c = OracleCache("qfilters", 2, 3, budget=40, n_sink=2, filters=f)
    c.update_and_fetch(k, v)
    st = c.stats()
    assert st["tokens_seen"] == 100 and st["tokens_kept"] == 40
    assert st["kept_bytes"] == 2 * 3 * 40 * 2 * 128 * 2 + 3 * 128 * 4
    assert st["full_seq_bytes"] == 2 * 3 * 100 * 2 * 128 * 2
    assert st["compression_ratio"] == pytest.approx(st["full_seq_bytes"] / st["kept_bytes"])


def test_under_budget_appends_everything():
    k, v = synth.gaussian_block(47, 1, 1, 30, dtype="bf16")
    c = OracleCache("knorm", 1, 1, budget=64, n_sink=4)
    c.update_and_fetch(k[:, :, :10], v[:, :, :10])
    c.update_and_fetch(k[:, :, 10:10], v[:, :, 10:10])       # m = 0 is a no-op
    c.update_and_fetch(k[:, :, 10:], v[:, :, 10:])
    assert np.array_equal(c.k, k) and c.pos[0, 0].tolist() == list(range(30))


def test_explicit_positions_are_kept_verbatim():
    k, v = synth.gaussian_block(48, 2, 1, 20, dtype="bf16")
    c = OracleCache("knorm", 2, 1, budget=8, n_sink=1)
    pos = np.stack([np.arange(20) * 3 + 5, np.arange(20) * 7]).astype(np.int32)
    c.update_and_fetch(k, v, pos=pos)
    for b in range(2):
        kept = c.last_kept[b, 0]
        assert np.array_equal(c.pos[b, 0], pos[b, kept])


@pytest.mark.parametrize("kw", [
    dict(n_sink=4, recent=60, budget=64),            # n_sink + recent >= budget
    dict(n_sink=64, recent=0, budget=64),
    dict(n_sink=4, recent=0, budget=64, sign=0),     # invalid sign
    dict(n_sink=4, recent=0, budget=64, sign=2),
])
def test_invalid_configs_raise(kw):
    with pytest.raises(ValueError):
        OracleCache("knorm", 1, 1, **kw)


def test_filter_head_layout_mismatch_raises():
    with pytest.raises(ValueError):
        OracleCache("qfilters", 1, 8, budget=64, filters=np.zeros((4, 128), np.float32))
    with pytest.raises(ValueError):      # filters=None is the key-SVD fallback; it needs calib_tokens >= 1
        OracleCache("qfilters", 1, 8, budget=64, filters=None, calib_tokens=0)
