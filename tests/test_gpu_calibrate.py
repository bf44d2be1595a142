"""GPU Q-Filters calibration against the oracle's uncentered query SVD."""
import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import synth
from oracle import calibrate as ocal
from tests.gpu_util import to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _gpu_calibrate(q, n_kv, dtype="bf16"):
    from kv_cache_token_bf16_gb300 import binding
    qd = to_dev(q, torch)
    out = torch.empty((n_kv, 128), dtype=torch.float32, device="cuda")
    binding.evict_qfilters_calibrate(qd.data_ptr(), binding.DTYPES[dtype], q.shape[0], q.shape[1], 128, n_kv,
                                     out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return out.cpu().numpy().astype(np.float64)


def _eigengap(q_heads):
    x = synth.bf16_bits_to_f32(q_heads).astype(np.float64) if q_heads.dtype == np.uint16 else q_heads
    s = np.linalg.svd(x, compute_uv=False)
    lam = s ** 2
    return (lam[0] - lam[1]) / lam[0]


@pytest.mark.parametrize("layer", [0, 13, 27])
def test_layer_stack_calibration_matches_oracle(layer):
    L = synth.qfilters_layer(layer, seq_len=8)
    got = _gpu_calibrate(L["queries"], 8)
    want = ocal.calibrate(L["queries"], 8)
    cos = np.einsum("hd,hd->h", got, want)
    assert np.all(cos >= 1 - 1e-6), cos
    assert np.allclose(np.linalg.norm(got, axis=1), 1.0, atol=1e-6)
    assert np.all(np.einsum("hd,hd->h", got, L["u"]) > 0.99)


def test_fp32_queries_and_no_gqa():
    q = synth.bf16_bits_to_f32(synth.long_context_queries(8))
    assert all(_eigengap(q[h]) > 1e-2 for h in range(8))
    got = _gpu_calibrate(q, 8, dtype="fp32")
    want = ocal.calibrate(q, 8)
    assert np.all(np.einsum("hd,hd->h", got, want) >= 1 - 1e-6)


def test_negated_drift_flips_the_filter():
    L = synth.qfilters_layer(3, n_q_heads=4, n_kv_heads=2, seq_len=8)
    q = synth.bf16_bits_to_f32(L["queries"])
    a = _gpu_calibrate(q, 2, dtype="fp32")
    b = _gpu_calibrate(-q, 2, dtype="fp32")
    assert np.allclose(a, -b, atol=1e-6)


def test_degenerate_inputs_raise():
    from kv_cache_token_bf16_gb300 import binding
    g = synth.rng(5)
    u = synth.unit_vectors(g, 1)[0]
    c = g.normal(4.0, 0.5, (500, 1))
    q = np.stack([c * u, -c * u]).astype(np.float32)          # opposite filters in one group
    with pytest.raises(binding.EvictError) as e:
        _gpu_calibrate(q, 1, dtype="fp32")
    assert e.value.code == binding.EVICT_ENUM
    with pytest.raises(binding.EvictError) as e:
        _gpu_calibrate(np.zeros((2, 300, 128), np.float32), 2, dtype="fp32")
    assert e.value.code == binding.EVICT_ENUM
    with pytest.raises(binding.EvictError) as e:
        _gpu_calibrate(np.zeros((3, 300, 128), np.float32), 2, dtype="fp32")   # 3 not a multiple of 2
    assert e.value.code == binding.EVICT_EINVAL
