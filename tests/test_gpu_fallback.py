"""GPU parity of the Q-Filters key-SVD fallback against the CPU oracle.

"Q-Filters — Query-Agnostic Projection Eviction", §How it works step 2
(before calib_tokens keys nothing is evicted; then the filter is estimated
from the key SVD and frozen), §Key-SVD fallback, §Path dependence.

The freeze estimates a direction by an iteration on each side (power
iteration in fp32 on the GPU, LAPACK's SVD in fp64 in the oracle), so the two
filters agree to rounding, not bit for bit. Each side freezes its own filter
and parity is checked in two parts: (1) the GPU filter against the oracle's
estimate on the same keys (signed cosine, planted-axis inputs with a wide
eigengap); (2) everything downstream — pass-through rows bit for bit, then the
freeze step's eviction and every later update against the oracle's own
filter: kept sets equal outside a band set by the measured distance between
the two filters (tests/gpu_util.check_own_filter_update), K / V bit-exact
copies, stored scores within the same bound. No GPU value enters the oracle.
"""
import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import synth
from oracle import calibrate as ocal
from oracle.cache import OracleCache
from tests.gpu_util import check_own_filter_update, to_bits, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _pair(B, H, budget, calib, dtype="bf16", max_block=512, **kw):
    from kv_cache_token_bf16_gb300 import binding
    gpu = binding.EvictCache("qfilters", B, H, budget=budget, max_block=max_block, dtype=dtype, filters=None,
                             calib_tokens=calib, **kw)
    ref = OracleCache("qfilters", B, H, budget=budget, dtype=dtype, filters=None, calib_tokens=calib, **kw)
    return gpu, ref


def _feed(gpu, ref, k, v, cuts, what, max_resyncs=0):
    """Feed the same blocks to both sides; each freezes its own filter. Returns the end of the
    block at which the GPU froze. On planted-axis keys the two filters agree to ~1e-6, so the
    kept sets must agree exactly (no cutoff pair of these seeds lies within the band)."""
    frozen_at = None
    resyncs = 0
    for a, b in zip(cuts[:-1], cuts[1:]):
        was = gpu.filters() is not None
        view = gpu.update_and_fetch(to_dev(k[:, :, a:b], torch), to_dev(v[:, :, a:b], torch))
        gpu.sync()
        ref.update_and_fetch(k[:, :, a:b], v[:, :, a:b])
        f = gpu.filters()
        if f is not None and not was:
            frozen_at = b
        resyncs += check_own_filter_update(view, ref, f, f"{what} after [{a},{b})")
        assert gpu.stats() == ref.stats(), f"{what}: stats after [{a},{b})"
    assert resyncs <= max_resyncs, f"{what}: {resyncs} in-band kept-set differences"
    return frozen_at


def _check_filters(gpu, k, n, axes=None, tol=2e-5):
    """GPU filters vs the oracle's key-SVD estimate over the first n keys (signed cosine)."""
    gf = gpu.filters().astype(np.float64)
    B, H = gf.shape[:2]
    for b in range(B):
        for h in range(H):
            want = ocal.key_svd_filter(k[b, h, :n])
            assert abs(np.linalg.norm(gf[b, h]) - 1.0) < 1e-5
            assert gf[b, h] @ want > 1.0 - tol, (b, h, gf[b, h] @ want)
            if axes is not None:                 # the planted axis is recovered (page: cosine > 0.99)
                assert abs(gf[b, h] @ axes[b, h]) > 0.99


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("chunk", [1, 7, 64, 300])
def test_fallback_chunked_prefill_then_decode(dtype, chunk):
    B, H, budget, calib, S = 2, 3, 40, 128, 300
    k, v, axes = synth.dominant_axis_block(71, B, H, S + 40, dtype=dtype)
    gpu, ref = _pair(B, H, budget, calib, dtype=dtype, n_sink=4, recent=3)
    cuts = list(range(0, S, chunk)) + [S]
    frozen_at = _feed(gpu, ref, k, v, cuts, f"{dtype} chunk {chunk}")
    # the freeze happens at the first call whose block reaches calib_tokens
    assert frozen_at == min(c for c in cuts if c >= calib)
    _check_filters(gpu, k, frozen_at, axes)
    # decode: single-row evictions against the frozen filters
    _feed(gpu, ref, k, v, list(range(S, S + 40)), f"{dtype} decode")
    assert gpu.stats()["kept_bytes"] == B * H * budget * 2 * 128 * (2 if dtype == "bf16" else 4) + B * H * 128 * 4


def test_fallback_passthrough_keeps_everything_over_budget():
    B, H, budget, calib = 1, 2, 16, 100
    k, v, _ = synth.dominant_axis_block(72, B, H, 160)
    gpu, ref = _pair(B, H, budget, calib, n_sink=2)
    _feed(gpu, ref, k, v, [0, 30, 60, 99], "pass-through")
    assert gpu.filters() is None
    kk, _, pos, score = gpu.view()
    assert kk.shape[2] == 99 and not torch.any(score != 0)
    assert np.array_equal(pos.cpu().numpy()[0, 0], np.arange(99))
    frozen_at = _feed(gpu, ref, k, v, [99, 100, 160], "freeze")          # 99 + 1 reaches 100
    assert frozen_at == 100
    _check_filters(gpu, k, 100)


@pytest.mark.parametrize("sign", [1, -1])
def test_fallback_one_block_freeze_and_sign(sign):
    B, H, budget = 2, 2, 64
    k, v, axes = synth.dominant_axis_block(73, B, H, 600)
    gpu, ref = _pair(B, H, budget, 128, n_sink=4, sign=sign)
    assert _feed(gpu, ref, k, v, [0, 512, 520, 600], "one block") == 512
    _check_filters(gpu, k, 512, axes)


def test_fallback_calib_tokens_one_and_reset():
    B, H = 1, 2
    k, v, _ = synth.dominant_axis_block(74, B, H, 200)
    gpu, ref = _pair(B, H, 32, 1, n_sink=1)
    # a single key has no variance: the filter is e_0
    assert _feed(gpu, ref, k, v, [0, 1], "first token") == 1
    f = gpu.filters()
    assert np.all(f[..., 0] == 1.0) and not np.any(f[..., 1:])
    _feed(gpu, ref, k, v, [1, 50, 120], "after e_0 freeze")
    # reset unfreezes: the next sequence estimates its own filters
    gpu.reset()
    assert gpu.filters() is None and gpu.stats()["offset"] == 0
    ref2 = OracleCache("qfilters", B, H, budget=32, n_sink=1, filters=None, calib_tokens=1)
    assert _feed(gpu, ref2, k, v, [120, 180, 200], "second sequence") == 180
    _check_filters(gpu, k[:, :, 120:], 60)


def test_fallback_grouped_update():
    from kv_cache_token_bf16_gb300 import binding
    B, H, L = 1, 4, 3
    data = [synth.dominant_axis_block(80 + l, B, H, 256) for l in range(L)]
    kw = dict(n_sink=4, recent=0)
    caches = [binding.EvictCache("qfilters", B, H, budget=48, max_block=256, filters=None, calib_tokens=100, **kw)
              for _ in range(L)]
    refs = [OracleCache("qfilters", B, H, budget=48, filters=None, calib_tokens=100, **kw) for _ in range(L)]
    for a, b in ((0, 60), (60, 130), (130, 256)):
        ks = [to_dev(d[0][:, :, a:b], torch) for d in data]
        vs = [to_dev(d[1][:, :, a:b], torch) for d in data]
        views = binding.evict_update_and_fetch_group([c.handle for c in caches], [t.data_ptr() for t in ks],
                                                     [t.data_ptr() for t in vs], None, b - a)
        caches[0].sync()
        for c, ref, d, vw in zip(caches, refs, data, views):
            ref.update_and_fetch(d[0][:, :, a:b], d[1][:, :, a:b])
            assert check_own_filter_update(binding.view_tensors(vw, B, H, "bf16"), ref, c.filters(),
                                           f"grouped [{a},{b})") == 0
    for c, d in zip(caches, data):
        _check_filters(c, d[0], 130)


def test_fallback_degenerate_keys():
    from kv_cache_token_bf16_gb300 import binding
    B, H = 1, 1
    row = synth.f32_to_bf16_bits(np.linspace(-2, 2, 128).astype(np.float32))
    k = np.tile(row, (B, H, 20, 1))
    v = synth.gaussian_block(75, B, H, 20)[1]
    gpu, ref = _pair(B, H, 8, 10, n_sink=1)
    _feed(gpu, ref, k, v, [0, 5, 12, 20], "equal keys")                # no variance: e_0
    f = gpu.filters()
    assert f[0, 0, 0] == 1.0 and not np.any(f[0, 0, 1:])
    # a NaN key at the freeze: reported by sync, the cache stays usable
    bad = k.copy()
    bad[0, 0, 3, 17] = 0x7FC0
    gpu2 = binding.EvictCache("qfilters", B, H, budget=8, max_block=64, filters=None, calib_tokens=10, n_sink=1)
    gpu2.update_and_fetch(to_dev(bad[:, :, :12], torch), to_dev(v[:, :, :12], torch))
    with pytest.raises(binding.EvictError) as e:
        gpu2.sync()
    assert e.value.code == binding.EVICT_EDEVICE
    gpu2.update_and_fetch(to_dev(k[:, :, 12:20], torch), to_dev(v[:, :, 12:20], torch))
    gpu2.sync()


@pytest.mark.parametrize("n,dtype", [(4096, "bf16"), (1000, "bf16"), (1500, "fp32")])
def test_fallback_freeze_across_a_cluster(n, dtype):
    # few units and many keys: the freeze splits each unit's rows over a cluster of CTAs
    # (8 for 4096 keys, 3 for 1000, 5 for 1500 with 2 units) and sums the slices in rank order
    B, H = 1, 2
    k, v, axes = synth.dominant_axis_block(90 + n, B, H, n + 16, dtype=dtype)
    gpu, ref = _pair(B, H, 256, 128, dtype=dtype, max_block=n, n_sink=4, recent=2)
    assert _feed(gpu, ref, k, v, [0, n, n + 16], f"cluster freeze n={n}") == n
    _check_filters(gpu, k, n, axes)
    # the kept rows were re-scored with the frozen filter: _feed compared every stored score with
    # the oracle's own projection, within the bound the two filters' distance sets


def test_fallback_long_context_full_size_sampled_units():
    # the long-context stream at full size (4 x 8 heads, 16 blocks of 8192, budget 4096): the
    # freeze at the first block, then every block; three sampled units are followed by oracles
    # that freeze their own filters. These keys are the pages' pure-drift case: the centred keys
    # are isotropic, the top direction is a sampling accident and the two sides' filters need
    # not agree, so the comparison is band-tolerant at whatever distance the filters lie.
    from kv_cache_token_bf16_gb300 import binding
    B, H, blocks = 4, 8, 16
    gpu = binding.EvictCache("qfilters", B, H, budget=4096, max_block=8192, filters=None, calib_tokens=128, n_sink=4)
    units = [(0, 0), (1, 5), (3, 7)]
    refs = {u: OracleCache("qfilters", 1, 1, budget=4096, n_sink=4, filters=None, calib_tokens=128) for u in units}
    resyncs = 0
    for blk in range(blocks):
        k, v = synth.long_context_block(blk, B, H)
        view = gpu.update_and_fetch(to_dev(k, torch), to_dev(v, torch))
        gpu.sync()
        f = gpu.filters()
        assert f is not None and np.allclose(np.linalg.norm(f, axis=-1), 1.0, atol=1e-5)
        gk, gv, gp, gs = [to_bits(t) for t in view]
        assert gp.shape[2] == min(4096, 8192 * (blk + 1))
        for (b, h), ref in refs.items():
            ref.update_and_fetch(k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1])
            unit = [x[b:b + 1, h:h + 1] for x in (gk, gv, gp, gs)]
            resyncs += check_own_filter_update(unit, ref, f[b:b + 1, h:h + 1], f"block {blk} unit {(b, h)}")
    print(f"long-context fallback: {resyncs} in-band resyncs over {blocks * len(units)} unit updates")
    assert gpu.stats()["offset"] == blocks * 8192
