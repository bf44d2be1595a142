"""The output-perturbation harness on the host: the attention output and the
metric against closed forms, and the pages' qualitative findings with the
oracle's eviction ("L2Norm — Intrinsic Key-Norm Eviction", offline harness:
keep-low wins on paper-like geometry and loses to random on the isotropic
control; "Q-Filters — Query-Agnostic Projection Eviction", offline harness:
best-of-sign beats random on paper-like geometry, the key-SVD direction
recovers the planted axis)."""
import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import perturb, synth
from oracle.bf16 import to_f64
from oracle.cache import OracleCache


def test_attention_output_closed_forms():
    g = np.random.default_rng(0)
    v = g.standard_normal((3, 128))
    q = g.standard_normal((2, 128))
    # one key: the output is its value
    assert np.allclose(perturb.attention_output(q, g.standard_normal((1, 128)), v[:1]), v[:1])
    # keys orthogonal to every probe: equal logits, the plain average
    k = np.zeros((3, 128))
    k[:, 5] = [1.0, 2.0, 3.0]
    qo = q.copy()
    qo[:, 5] = 0.0
    assert np.allclose(perturb.attention_output(qo, k, v), v.mean(axis=0))
    # two keys: weights e^a / (e^a + e^b) with a, b the scaled logits
    k2 = np.stack([np.eye(128)[0] * 2.0, np.eye(128)[1] * 1.0])
    q2 = np.eye(128)[[0]] * 3.0 + np.eye(128)[[1]] * 1.5
    a, b = 6.0 / np.sqrt(128), 1.5 / np.sqrt(128)
    w = np.exp(a) / (np.exp(a) + np.exp(b))
    assert np.allclose(perturb.attention_output(q2, k2, v[:2]), w * v[0] + (1 - w) * v[1])


def test_perturbation_fixed_points():
    g = np.random.default_rng(1)
    k, v, q = g.standard_normal((40, 128)), g.standard_normal((40, 128)), g.standard_normal((4, 128))
    assert perturb.perturbation(q, k, v, np.arange(40)) == pytest.approx(0.0, abs=1e-12)
    p = perturb.perturbation(q, k, v, np.arange(10))
    assert 0.0 < p <= 2.0
    assert perturb.perturbation(q, k, 3.0 * v, np.arange(10)) == pytest.approx(p, rel=1e-12)   # scale-free


def test_random_arm():
    kept = perturb.random_kept(5, 3, 100, 20)
    assert kept.shape == (3, 20)
    for row in kept:
        assert list(row[:4]) == [0, 1, 2, 3] and np.all(np.diff(row) > 0) and row[-1] < 100


def _oracle_arm(method, k, v, budget, **kw):
    c = OracleCache(method, k.shape[0], 1, budget=budget, n_sink=4, **kw)
    c.update_and_fetch(k, v)
    return c.last_kept[:, 0], c


def _arms(geometry, S=512, budget=64, B=8):
    k, v, q, u = synth.perturbation_geometry(geometry, synth.seed_for(6, 0), B, S)
    kf, vf, qf = to_f64(k[:, 0]), to_f64(v[:, 0]), q.astype(np.float64)
    kept = {"knorm_low": _oracle_arm("knorm", k, v, budget, keep_low=True)[0],
            "knorm_high": _oracle_arm("knorm", k, v, budget, keep_low=False)[0],
            "random": perturb.random_kept(synth.seed_for(6, 100), B, S, budget)}
    plus, cache = _oracle_arm("qfilters", k, v, budget, filters=None, sign=1)
    kept["qfilters_plus"] = plus
    kept["qfilters_minus"] = _oracle_arm("qfilters", k, v, budget, filters=None, sign=-1)[0]
    per = {a: np.array([perturb.perturbation(qf[r], kf[r], vf[r], kept[a][r]) for r in range(B)]) for a in kept}
    per["qfilters_best"] = np.minimum(per["qfilters_plus"], per["qfilters_minus"])
    cos = np.abs(np.sum(cache.filters_bh[:, 0].astype(np.float64) * u, axis=1))
    return {a: x.mean() for a, x in per.items()}, cos


def test_knorm_paper_geometry_keep_low_wins():
    m, _ = _arms("knorm_paper")
    assert m["knorm_low"] < m["random"] - 0.05 and m["knorm_low"] < m["knorm_high"] - 0.2


def test_isotropic_control_keep_low_loses_to_random():
    m, _ = _arms("isotropic")
    assert m["knorm_low"] > m["random"]


def test_qfilters_paper_geometry_best_of_sign_wins_and_axis_recovered():
    m, cos = _arms("qfilters_paper")
    assert m["qfilters_best"] < m["random"] - 0.2
    assert cos.mean() > 0.9
