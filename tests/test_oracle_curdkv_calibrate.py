"""Pins for the oracle's CurDKV leverage and Q-Filters calibration (CPU only)."""
import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import synth
from oracle import calibrate, curdkv
from oracle.cache import OracleCache


def _orthonormal(g, n, r):
    q, _ = np.linalg.qr(g.standard_normal((n, r)))
    return q


# ------------------------------------------------------------------ leverage
def test_leverage_on_a_known_decomposition():
    # W = U diag(s) V^T with known factors: l_i = sum_{j<r} s_j^2 U_ij^2 / sum s^2
    g = synth.rng(51)
    n, d = 300, 128
    u, v = _orthonormal(g, n, d), _orthonormal(g, d, d)
    s = np.sort(g.uniform(0.1, 5.0, d))[::-1]
    w = (u * s) @ v.T
    for r in (1, 5, 16, 40):
        want = np.sum(u[:, :r] ** 2 * s[:r] ** 2, axis=1) / np.sum(s ** 2)
        assert np.allclose(curdkv.leverage(w, r), want, rtol=1e-9, atol=1e-15)


def test_full_rank_leverage_is_row_energy_share():
    # summed over every singular direction the leverage of row i is ||w_i||^2 / ||W||_F^2
    g = synth.rng(52)
    w = g.standard_normal((500, 128)) * g.uniform(0, 3, (500, 1))
    l = curdkv.leverage(w, 128)
    assert np.allclose(l, np.sum(w * w, 1) / np.sum(w * w), rtol=1e-10)
    # fewer rows than D: r = min(cap, n, D) = n covers every direction too
    w2 = g.standard_normal((20, 128))
    assert np.allclose(curdkv.leverage(w2, 64), np.sum(w2 * w2, 1) / np.sum(w2 * w2))


def test_leverage_total_is_captured_energy_fraction():
    g = synth.rng(53)
    w = g.standard_normal((400, 128)) @ np.diag(np.linspace(3, 0.1, 128))
    lam = np.sort(np.linalg.eigvalsh(w.T @ w))[::-1]
    for r in (1, 16, 100):
        assert curdkv.leverage(w, r).sum() == pytest.approx(lam[:r].sum() / lam.sum(), rel=1e-9)


def test_leverage_invariant_to_scaling_attention_or_values():
    g = synth.rng(54)
    keys = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(g.standard_normal((90, 128)).astype(np.float32)))
    vals = g.standard_normal((90, 128))
    l1, a, _ = curdkv.block_scores(keys, vals, 10, 16)
    l2, _, _ = curdkv.block_scores(keys, 7.5 * vals, 10, 16)
    assert np.allclose(l1, l2, rtol=1e-10)
    w = a[:, None] * vals
    assert np.allclose(curdkv.leverage(3.0 * w, 16), curdkv.leverage(w, 16), rtol=1e-10)


def test_all_zero_values_give_finite_zero_leverage():
    g = synth.rng(55)
    keys = g.standard_normal((40, 128)).astype(np.float32)
    l, _, _ = curdkv.block_scores(keys, np.zeros((40, 128), np.float32), 8, 16)
    assert np.all(np.isfinite(l)) and np.all(l == 0)


def test_identical_keys_different_values_diverge():
    g = synth.rng(56)
    keys = g.standard_normal((30, 128)).astype(np.float32)
    keys[12] = keys[11]
    vals = g.standard_normal((30, 128))
    vals[12] = 0.01 * vals[11]
    l, a, _ = curdkv.block_scores(keys, vals, 5, 16)
    assert a[11] == a[12]                                 # same keys -> same attention
    assert l[11] > 100 * l[12]                            # different values -> different leverage


# -------------------------------------------------------------- attention
def test_attention_mass_sums_to_block_length_and_is_causal():
    g = synth.rng(57)
    keys = g.standard_normal((50, 128)).astype(np.float32)
    a = curdkv.proxy_attention_block(keys, 12)
    assert a.sum() == pytest.approx(12.0, rel=1e-12)
    assert np.allclose(a, curdkv.proxy_attention(keys, 12), rtol=1e-12)


def test_attention_with_identical_keys_is_harmonic():
    # all keys equal: query t spreads mass uniformly over the k+t+1 rows it sees
    keys = np.tile(np.linspace(-1, 1, 128, dtype=np.float32), (20, 1))
    k, m = 14, 6
    a = curdkv.proxy_attention_block(keys, m)
    want = np.array([sum(1.0 / (k + t + 1) for t in range(m) if k + t >= i) for i in range(k + m)])
    assert np.allclose(a, want, rtol=1e-12)


def _per_token_bruteforce(keys, vals, cum_old, rank_cap):
    """CurDKV page, How it works steps 1-4 for ONE incoming token, written out
    with explicit loops; leverage from the eigen-decomposition of W W^T."""
    n, d = keys.shape
    q = keys[-1]
    logits = [sum(float(keys[i, j]) * float(q[j]) for j in range(d)) / np.sqrt(d) for i in range(n)]
    mx = max(logits)
    e = [np.exp(x - mx) for x in logits]
    z = sum(e)
    attn = [x / z for x in e]
    w = np.array([[attn[i] * float(vals[i, j]) for j in range(d)] for i in range(n)])
    mu, vec = np.linalg.eigh(w @ w.T)                  # mu_j = s_j^2, vec = U
    order = np.argsort(mu)[::-1]
    mu, vec = mu[order], vec[:, order]
    r = min(rank_cap, n, d)
    lev = [sum(mu[j] * vec[i, j] ** 2 for j in range(r)) / sum(mu) for i in range(n)]
    return [cum_old[i] + lev[i] for i in range(n - 1)] + [lev[n - 1]]


def test_block_of_one_equals_per_token_steps():
    g = synth.rng(58)
    for trial in range(4):
        n = 6 + 2 * trial
        keys = g.standard_normal((n, 128)).astype(np.float32)
        vals = g.standard_normal((n, 128))
        cum_old = g.uniform(0, 1, n - 1)
        l, _, _ = curdkv.block_scores(keys, vals, 1, rank_cap=3)
        got = curdkv.cumulative(cum_old, l)
        want = _per_token_bruteforce(keys, vals, cum_old, 3)
        assert np.allclose(got, want, rtol=1e-9, atol=1e-14)


@pytest.mark.parametrize("seed", range(8))
def test_planted_class1_tokens_fill_the_budget(seed):
    # CurDKV page, planted-geometry observable: every non-sink budget slot is class 1
    p = synth.curdkv_planted(batch=1, n_kv_heads=1, existing=240, incoming=16, seed=1000 + seed)
    c = OracleCache("curdkv", 1, 1, budget=24, n_sink=4, rank_cap=16)
    c.set_state(p["k"][:, :, :240], p["v"][:, :, :240],
                np.arange(240, dtype=np.int32)[None, None], np.zeros((1, 1, 240)), 240)
    c.update_and_fetch(p["k"][:, :, 240:], p["v"][:, :, 240:])
    kept = c.last_kept[0, 0]
    cls = p["cls"][0, 0, kept]
    assert c.n_kept == 24 and np.all(cls[4:] == 1)


def test_sink_with_negligible_value_survives():
    p = synth.curdkv_planted(batch=1, n_kv_heads=1, existing=100, incoming=8, seed=77)
    v = p["v"].copy()
    v[0, 0, :2] = 0                                          # sinks with zero value
    c = OracleCache("curdkv", 1, 1, budget=10, n_sink=2, rank_cap=16)
    c.update_and_fetch(p["k"], v)
    assert c.last_kept[0, 0, :2].tolist() == [0, 1]


# -------------------------------------------------------------- calibration
def _planted_queries(g, u, mean, n=3000):
    c = g.normal(mean, 0.5, size=(n, 1))
    return c * u[None, :] + g.standard_normal((n, 128))


def test_calibration_recovers_planted_drift_with_sign():
    g = synth.rng(61)
    u = synth.unit_vectors(g, 1)[0]
    f = calibrate.compute_qfilter(_planted_queries(g, u, 4.0))
    assert f @ u > 0.99
    f_neg = calibrate.compute_qfilter(_planted_queries(g, u, -4.0))
    assert f_neg @ u < -0.99                                   # tracks the negated drift


def test_calibration_of_rank_one_queries_is_exact():
    g = synth.rng(62)
    u = synth.unit_vectors(g, 1)[0]
    c = g.uniform(0.5, 2.0, (200, 1))
    assert np.allclose(calibrate.compute_qfilter(c * u[None, :]), u, atol=1e-12)
    assert np.allclose(calibrate.compute_qfilter(-c * u[None, :]), -u, atol=1e-12)


def test_calibration_matches_power_iteration():
    # independent method: power iteration on Q^T Q, sign by the mean projection
    g = synth.rng(63)
    u = synth.unit_vectors(g, 1)[0]
    q = _planted_queries(g, u, 1.5)
    c = q.T @ q
    x = np.ones(128)
    for _ in range(2000):
        x = c @ x
        x /= np.linalg.norm(x)
    if q.mean(0) @ x < 0:
        x = -x
    assert np.allclose(calibrate.compute_qfilter(q), x, atol=1e-8)


def test_centering_picks_the_wrong_axis():
    # drift along u (mean 4, sd 0.5) and a zero-mean high-variance axis w (sd 2)
    g = synth.rng(64)
    u, w = _orthonormal(g, 128, 2).T
    n = 3000
    q = (g.normal(4.0, 0.5, (n, 1)) * u + g.normal(0.0, 2.0, (n, 1)) * w
         + 0.1 * g.standard_normal((n, 128)))
    assert abs(calibrate.compute_qfilter(q) @ u) > 0.99        # uncentered: the drift axis
    assert abs(calibrate.centered_top_direction(q) @ w) > 0.99  # centered: the variance axis
    assert abs(calibrate.centered_top_direction(q) @ u) < 0.1


def test_gqa_average_is_unit_norm_and_grouped():
    g = synth.rng(65)
    f = synth.unit_vectors(g, 6)
    out = calibrate.average_gqa(f, 2)
    assert np.allclose(np.linalg.norm(out, axis=1), 1.0)
    want0 = f[:3].mean(0) / np.linalg.norm(f[:3].mean(0))
    assert np.allclose(out[0], want0)


def test_degenerate_gqa_average_raises():
    u = np.zeros(128)
    u[3] = 1.0
    with pytest.raises(ValueError):
        calibrate.average_gqa(np.stack([u, -u]), 1)


def test_calibrate_on_the_layer_stack_workload_shape():
    layer = synth.qfilters_layer(0, n_samples=400, seq_len=8)
    f = calibrate.calibrate(layer["queries"], 8)
    assert f.shape == (8, 128)
    assert np.all(np.einsum("hd,hd->h", f, layer["u"]) > 0.99)
