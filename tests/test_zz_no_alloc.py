"""evict_prefill_noalloc against the regular cache path and the oracle.

The no-allocation entry point serves callers that cannot call cudaMalloc
(graph capture, fixed memory pools, plug-ins inside another framework's
allocator). It keeps its intermediate data in a fixed array inside the
library, so this file also checks that a second call in a row, which finds
the previous call's leftovers in that array, still gives the right answer,
and that the array's error word reads clean after the calls.
This file is collected last on purpose.
"""
import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import synth
from oracle.cache import OracleCache
from tests.gpu_util import to_bits, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _config(binding, method, B, H, budget, filters=None, dtype="bf16", recent=16, keep_low=1, sign=1):
    return binding.EvictConfig(
        method=binding.METHODS[method], dtype=binding.EVICT_BF16 if dtype == "bf16" else binding.EVICT_FP32,
        batch=B, n_kv_heads=H, head_dim=128, budget=budget, n_sink=4, recent=recent, max_block=0, max_kept=0,
        keep_low=keep_low, sign=sign, filters=filters.data_ptr() if filters is not None else None, n_filter_heads=0,
        rank_cap=0, stream=torch.cuda.current_stream().cuda_stream)


def _outputs(B, H, budget, dtype):
    t = torch.bfloat16 if dtype == "bf16" else torch.float32
    k_out = torch.empty((B, H, budget, 128), dtype=t, device="cuda")
    return (k_out, torch.empty_like(k_out), torch.empty((B, H, budget), dtype=torch.int32, device="cuda"),
            torch.empty((B, H, budget), dtype=torch.float32, device="cuda"))


@pytest.mark.parametrize("method", ["knorm", "qfilters"])
def test_no_alloc_matches_the_cache_path_on_two_calls_in_a_row(method):
    from kv_cache_token_bf16_gb300 import binding
    B, H, budget = 2, 4, 512
    filters = None
    if method == "qfilters":
        filters = torch.from_numpy(synth.unit_vectors(synth.rng(8), H).astype(np.float32)).cuda()
    cfg = _config(binding, method, B, H, budget, filters)
    k_out, v_out, pos_out, score_out = _outputs(B, H, budget, "bf16")
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
    binding.evict_noalloc_status(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("method,dtype,n,budget,explicit_pos", [
    ("knorm", "bf16", 3000, 512, False),
    ("knorm", "fp32", 1500, 256, True),        # fp32 storage, caller positions
    ("qfilters", "bf16", 300, 512, True),      # n <= budget: an append, no eviction
    ("qfilters", "fp32", 2000, 700, False),
    ("knorm", "bf16", 30000, 4096, False),     # more rows than the register selection holds
    ("qfilters", "bf16", 26000, 1024, True),
])
def test_no_alloc_matches_the_oracle(method, dtype, n, budget, explicit_pos):
    from kv_cache_token_bf16_gb300 import binding
    B, H = (1, 2) if n > 24576 else (2, 3)
    k, v = synth.gaussian_block(40 + n, B, H, n, dtype=dtype)
    kw = dict(n_sink=4, recent=16, dtype=dtype)
    filters = None
    if method == "qfilters":
        f = synth.unit_vectors(synth.rng(9), H).astype(np.float32)
        filters = torch.from_numpy(f).cuda()
        kw.update(filters=f, sign=-1)
    else:
        kw.update(keep_low=False)
    pos = (1000 + 3 * np.arange(n, dtype=np.int32))[None].repeat(B, 0) if explicit_pos else None
    cfg = _config(binding, method, B, H, budget, filters, dtype, keep_low=0, sign=-1)
    outs = _outputs(B, H, budget, dtype)
    kd, vd = to_dev(k, torch), to_dev(v, torch)
    pd = torch.from_numpy(pos).cuda() if explicit_pos else None
    for _ in range(2):                             # the second call finds the first one's leftovers
        for t in outs:
            t.fill_(0)
        binding.evict_prefill_noalloc(cfg, kd.data_ptr(), vd.data_ptr(), pd.data_ptr() if pd is not None else None,
                                      n, *[t.data_ptr() for t in outs])
        binding.evict_noalloc_status(torch.cuda.current_stream().cuda_stream)
        ref = OracleCache(method, B, H, budget=budget, **kw)
        ref.update_and_fetch(k, v, pos)
        rows = min(n, budget)
        gk, gv, gp, gs = [to_bits(t)[:, :, :rows] for t in outs]
        assert np.array_equal(gp, ref.pos), "positions differ from the oracle"
        assert np.array_equal(gk, ref.k) and np.array_equal(gv, ref.v), "kept K/V differ from the oracle"
        assert gs.tobytes() == ref.score.astype(np.float32).tobytes(), "stored scores differ from the oracle"


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    from kv_cache_token_bf16_gb300 import binding
    B, H, budget, n = 32, 8, 4096, 8192       # needs ~12.6 MB of scratch, more than the 8 MiB array
    cfg = _config(binding, "knorm", B, H, budget)
    dummy = torch.empty(1, device="cuda")
    with pytest.raises(binding.EvictError) as e:
        binding.evict_prefill_noalloc(cfg, dummy.data_ptr(), dummy.data_ptr(), None, n, dummy.data_ptr(),
                                      dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr())
    assert e.value.code == binding.EVICT_ELIMIT


def test_no_alloc_rejects_misaligned_buffers_before_any_work():
    from kv_cache_token_bf16_gb300 import binding
    B, H, budget, n = 1, 2, 64, 100
    cfg = _config(binding, "knorm", B, H, budget)
    buf = torch.zeros((4 * B * H * n * 128 + 64,), dtype=torch.bfloat16, device="cuda")
    p = buf.data_ptr()
    outs = _outputs(B, H, budget, "bf16")
    ptrs = [t.data_ptr() for t in outs]
    with pytest.raises(binding.EvictError, match="16-byte aligned") as e:
        binding.evict_prefill_noalloc(cfg, p + 2, p, None, n, *ptrs)
    assert e.value.code == binding.EVICT_EINVAL
    with pytest.raises(binding.EvictError, match="4-byte aligned"):
        binding.evict_prefill_noalloc(cfg, p, p, None, n, ptrs[0], ptrs[1], ptrs[2] + 2, ptrs[3])
    binding.evict_noalloc_status(torch.cuda.current_stream().cuda_stream)
