"""evict_prefill_noalloc against the regular cache path.

The no-allocation entry point serves callers that cannot call cudaMalloc
(graph capture, fixed memory pools, plug-ins inside another framework's
allocator). It keeps its intermediate data in a fixed array inside the
library, so this test also checks that a second call in a row, which finds
the previous call's leftovers in that array, still gives the right answer.
This file is collected last on purpose.
"""
import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import synth
from tests.gpu_util import to_bits, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _config(binding, method, B, H, budget, filters=None):
    return binding.EvictConfig(
        method=binding.METHODS[method], dtype=binding.EVICT_BF16, batch=B, n_kv_heads=H, head_dim=128,
        budget=budget, n_sink=4, recent=16, max_block=0, max_kept=0, keep_low=1, sign=1,
        filters=filters.data_ptr() if filters is not None else None, n_filter_heads=0, rank_cap=0,
        stream=torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("method", ["knorm", "qfilters"])
def test_no_alloc_matches_the_cache_path_on_two_calls_in_a_row(method):
    from kv_cache_token_bf16_gb300 import binding
    B, H, budget = 2, 4, 512
    filters = None
    if method == "qfilters":
        filters = torch.from_numpy(synth.unit_vectors(synth.rng(8), H).astype(np.float32)).cuda()
    cfg = _config(binding, method, B, H, budget, filters)
    k_out = torch.empty((B, H, budget, 128), dtype=torch.bfloat16, device="cuda")
    v_out = torch.empty_like(k_out)
    pos_out = torch.empty((B, H, budget), dtype=torch.int32, device="cuda")
    score_out = torch.empty((B, H, budget), dtype=torch.float32, device="cuda")
    for call, (seed, n) in enumerate([(31, 3000), (32, 2500)]):
        k, v = synth.gaussian_block(seed, B, H, n)
        kd, vd = to_dev(k, torch), to_dev(v, torch)
        binding.evict_prefill_noalloc(cfg, kd.data_ptr(), vd.data_ptr(), None, n, k_out.data_ptr(),
                                      v_out.data_ptr(), pos_out.data_ptr(), score_out.data_ptr())
        ref = binding.EvictCache(method, B, H, budget=budget, n_sink=4, recent=16, max_block=n,
                                 filters=filters, sign=1)
        rk, rv, rp, rs = ref.update_and_fetch(kd, vd)
        ref.sync()
        torch.cuda.synchronize()
        assert np.array_equal(to_bits(pos_out), to_bits(rp)), f"call {call}: positions differ"
        assert np.array_equal(to_bits(k_out), to_bits(rk)), f"call {call}: keys differ"
        assert np.array_equal(to_bits(v_out), to_bits(rv)), f"call {call}: values differ"
        assert to_bits(score_out).tobytes() == to_bits(rs).tobytes(), f"call {call}: scores differ"
        ref.close()


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    from kv_cache_token_bf16_gb300 import binding
    B, H, budget, n = 32, 8, 4096, 8192       # needs ~12.6 MB of scratch, more than the 8 MiB array
    cfg = _config(binding, "knorm", B, H, budget)
    dummy = torch.empty(1, device="cuda")
    with pytest.raises(binding.EvictError) as e:
        binding.evict_prefill_noalloc(cfg, dummy.data_ptr(), dummy.data_ptr(), None, n, dummy.data_ptr(),
                                      dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr())
    assert e.value.code == binding.EVICT_ELIMIT
