"""Update calls captured in a CUDA graph.

The update path never allocates, synchronises or reads device memory back
(the cache keeps n_kept and offset on the host), so a whole decode loop can
be captured once and replayed. A replay runs the captured steps exactly:
their positions and row counts are fixed at capture, so each replay must
start from the device state the capture started from. Checked bit for bit
against the oracle and against a second replay after restoring that state.
"""
import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import synth
from oracle.cache import OracleCache
from tests.gpu_util import assert_cache_equal, to_bits, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _scorer(method, H):
    if method == "knorm":
        return dict(keep_low=True)
    return dict(filters=synth.decode_filters(H), sign=1)


@pytest.mark.parametrize("method", ["knorm", "qfilters"])
@pytest.mark.parametrize("m", [1, 16])
def test_captured_decode_loop(method, m):
    from kv_cache_token_bf16_gb300 import binding
    B, H, budget, prefill, steps = 4, 2, 96, 200, 24
    kw = dict(n_sink=4, recent=16, **_scorer(method, H))
    k0, v0 = synth.decode_prefill(B, H, prefill)
    ks, vs = synth.decode_steps(0, steps * m, B, H)                 # [steps*m, B, H, 1, D]
    ks = np.ascontiguousarray(np.concatenate(list(ks), axis=2))     # [B, H, steps*m, D]
    vs = np.ascontiguousarray(np.concatenate(list(vs), axis=2))
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        cache = binding.EvictCache(method, B, H, budget=budget, max_block=prefill, stream=stream.cuda_stream, **kw)
        cache.update_and_fetch(to_dev(k0, torch), to_dev(v0, torch))
        # the blocks of every step, resident before the capture
        kd = [to_dev(ks[:, :, s * m:(s + 1) * m], torch) for s in range(steps)]
        vd = [to_dev(vs[:, :, s * m:(s + 1) * m], torch) for s in range(steps)]
        snap = [t.clone() for t in cache.view()]
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for s in range(steps):
            binding.evict_update_and_fetch(cache.handle, kd[s].data_ptr(), vd[s].data_ptr(), None, m)
    # nothing ran during the capture; the host already counts the captured steps
    assert cache.stats()["offset"] == prefill + steps * m
    g.replay()
    stream.synchronize()
    cache.sync()
    ref = OracleCache(method, B, H, budget=budget, **kw)
    ref.update_and_fetch(k0, v0)
    for s in range(steps):
        ref.update_and_fetch(ks[:, :, s * m:(s + 1) * m], vs[:, :, s * m:(s + 1) * m])
    assert_cache_equal(cache.view(), ref, f"{method} m={m} captured loop")
    first = [to_bits(t).copy() for t in cache.view()]
    # restore the pre-capture state and replay again: identical bits
    with torch.cuda.stream(stream):
        cache.set_state(*[t.contiguous() for t in snap[:3]], score=snap[3].contiguous(), offset=prefill)
    g.replay()
    stream.synchronize()
    cache.sync()
    for a, b in zip(first, cache.view()):
        assert np.array_equal(a, to_bits(b))


def test_captured_grouped_layers():
    from kv_cache_token_bf16_gb300 import binding
    B, H, L, budget, steps = 2, 2, 3, 64, 12
    kw = dict(n_sink=4, recent=8, keep_low=True)
    data = [synth.gaussian_block(90 + l, B, H, 100 + steps) for l in range(L)]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        caches = [binding.EvictCache("knorm", B, H, budget=budget, max_block=100, stream=stream.cuda_stream, **kw)
                  for _ in range(L)]
        for c, (k, v) in zip(caches, data):
            c.update_and_fetch(to_dev(k[:, :, :100], torch), to_dev(v[:, :, :100], torch))
        kd = [[to_dev(k[:, :, 100 + s:101 + s], torch) for (k, _) in data] for s in range(steps)]
        vd = [[to_dev(v[:, :, 100 + s:101 + s], torch) for (_, v) in data] for s in range(steps)]
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for s in range(steps):
            binding.evict_update_and_fetch_group([c.handle for c in caches], [t.data_ptr() for t in kd[s]],
                                                 [t.data_ptr() for t in vd[s]], None, 1)
    g.replay()
    stream.synchronize()
    for c, (k, v) in zip(caches, data):
        c.sync()
        ref = OracleCache("knorm", B, H, budget=budget, **kw)
        ref.update_and_fetch(k[:, :, :100], v[:, :, :100])
        for s in range(steps):
            ref.update_and_fetch(k[:, :, 100 + s:101 + s], v[:, :, 100 + s:101 + s])
        assert_cache_equal(c.view(), ref, "captured grouped step")


@pytest.mark.parametrize("method,kw,m", [
    ("curdkv", {}, 1),                               # decode steps: the fused single-eviction kernel
    ("curdkv", {}, 8),                               # 8-token blocks: proxy attention, Gram, eig, leverage
    ("h2o", {}, 1),
    ("h2o", {}, 8),
    ("curdkv", {"per_token": True}, 4),              # the token-by-token loop inside each call
    ("h2o", {"per_token": True}, 4),
    ("qfilters", {"filters": None, "calib_tokens": 96}, 4),   # the key-SVD freeze falls inside the capture
])
def test_captured_loop_equals_eager(method, kw, m):
    # a captured loop and the same calls issued one by one give the same bits: no kernel of these
    # scorers reduces in a run-dependent order, and nothing on the path reads device state back
    from kv_cache_token_bf16_gb300 import binding
    B, H, budget, prefill, steps = 2, 2, 64, 80, 12
    keys = synth.clustered_keys(70, B, H, prefill + steps * m, spread=0.8)
    vals = synth.planted_spectrum_values(71, B, H, prefill + steps * m, rank=4)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        pair = [binding.EvictCache(method, B, H, budget=budget, max_block=prefill, rank_cap=4,
                                   stream=stream.cuda_stream, **kw) for _ in range(2)]
        for c in pair:
            c.update_and_fetch(to_dev(keys[:, :, :prefill], torch), to_dev(vals[:, :, :prefill], torch))
        sl = [slice(prefill + s * m, prefill + (s + 1) * m) for s in range(steps)]
        kd = [to_dev(keys[:, :, x], torch) for x in sl]
        vd = [to_dev(vals[:, :, x], torch) for x in sl]
    stream.synchronize()
    eager, captured = pair
    with torch.cuda.stream(stream):
        for s in range(steps):
            eager.update_and_fetch(kd[s], vd[s])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for s in range(steps):
            binding.evict_update_and_fetch(captured.handle, kd[s].data_ptr(), vd[s].data_ptr(), None, m)
    g.replay()
    stream.synchronize()
    for c in pair:
        c.sync()
    assert eager.stats() == captured.stats()
    for a, b in zip(eager.view(), captured.view()):
        assert np.array_equal(to_bits(a), to_bits(b)), f"{method} {kw} m={m}"
    if method == "qfilters":
        assert np.array_equal(eager.filters(), captured.filters())
        assert eager.view()[0].shape[2] == budget
