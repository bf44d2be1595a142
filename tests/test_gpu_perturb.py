"""The output-perturbation harness on the GPU path: the kept sets it measures
are the oracle's (KNorm bit for bit; the key-SVD fallback against an oracle
that freezes its own filter, outside the band the two filters' distance
sets), and the pages' findings hold on its numbers."""
import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import perturb, synth
from oracle.cache import OracleCache
from tests.gpu_util import kept_sets_agree_outside_band, projection_tolerance

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("geometry", synth.PERTURB_GEOMETRIES)
def test_harness_kept_sets_are_the_oracles(geometry):
    B, S, budget = 8, 512, 64
    k, v, _, _ = synth.perturbation_geometry(geometry, synth.seed_for(6, 0), B, S)
    for arm in ("knorm_low", "knorm_high", "qfilters_plus", "qfilters_minus"):
        kept, ms, filt = perturb.gpu_kept(arm, k, v, budget)
        if arm.startswith("knorm"):
            ref = OracleCache("knorm", B, 1, budget=budget, n_sink=4, keep_low=arm == "knorm_low")
            ref.update_and_fetch(k, v)
            assert np.array_equal(kept, ref.last_kept[:, 0]), (geometry, arm)
        else:
            ref = OracleCache("qfilters", B, 1, budget=budget, n_sink=4, filters=None,
                              sign=1 if arm == "qfilters_plus" else -1)
            ref.update_and_fetch(k, v)
            for b in range(B):
                tol = projection_tolerance(k[b, 0], filt[b], ref.filters_bh[b, 0])
                assert kept_sets_agree_outside_band(ref.last_scores[b, 0], ref.last_kept[b, 0], kept[b], tol, 4, 0,
                                                    budget), (geometry, arm, b)
        assert ms > 0


def test_harness_findings_on_the_gpu():
    paper = perturb.run("knorm_paper", 512, 64)
    iso = perturb.run("isotropic", 512, 64)
    qf = perturb.run("qfilters_paper", 512, 64)
    assert paper["advantage_vs_random"]["knorm_low"] > 0.05
    assert paper["perturbation"]["knorm_low"] < paper["perturbation"]["knorm_high"] - 0.2
    assert iso["advantage_vs_random"]["knorm_low"] < 0
    assert qf["advantage_vs_random"]["qfilters_best"] > 0.2 and qf["filter_cosine"] > 0.9
    for r in (paper, iso, qf):
        assert set(r["evict_ms"]) == {"knorm_low", "knorm_high", "qfilters_plus", "qfilters_minus", "h2o"}
