"""GPU parity of the KNorm and Q-Filters path against the CPU oracle.

Kept index sets, positions, compacted K/V and stored scores must be
bit-exact (the canonical fp32 score order makes the score a pure function of
the key bits on both sides). Inputs are the seeded workloads' generators at
sizes the oracle finishes quickly, plus full-size runs checked on sampled
(b, h) units and by invariants.
"""
import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import synth
from oracle import calibrate as ocal
from oracle import scores as oscores
from oracle import select as osel
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


def _pair(method, batch, heads, budget, dtype="bf16", max_block=8192, **kw):
    from kv_cache_token_bf16_gb300 import binding
    gpu = binding.EvictCache(method, batch, heads, budget=budget, max_block=max_block, dtype=dtype,
                             max_kept=kw.pop("max_kept", 0), **kw)
    ref = OracleCache(method, batch, heads, budget=budget, dtype=dtype, **kw)
    return gpu, ref


def _feed(gpu, ref, k, v, cuts, check_each=False, what=""):
    view = None
    for a, b in zip(cuts[:-1], cuts[1:]):
        view = gpu.update_and_fetch(to_dev(k[:, :, a:b], torch), to_dev(v[:, :, a:b], torch))
        ref.update_and_fetch(k[:, :, a:b], v[:, :, a:b])
        if check_each:
            gpu.sync()
            assert_cache_equal(view, ref, f"{what} after [{a},{b})")
    gpu.sync()
    return view


# ---------------------------------------------------------------------------
# KNorm single sequence (fp32, B=H=1, S=1024, budget 512, n_sink 4, keep low)
# ---------------------------------------------------------------------------
def test_knorm_single_sequence_one_block_and_token_by_token():
    k, v = synth.knorm_single_sequence(1024)
    kw = dict(n_sink=4, recent=0, keep_low=True)
    gpu, ref = _pair("knorm", 1, 1, 512, dtype="fp32", max_block=1024, **kw)
    one = _feed(gpu, ref, k, v, [0, 1024])
    assert_cache_equal(one, ref, "one block")
    one_bits = [to_bits(t).copy() for t in one]
    # the same tokens one at a time: bit-identical cache (path independence)
    gpu2, ref2 = _pair("knorm", 1, 1, 512, dtype="fp32", max_block=1024, **kw)
    tok = _feed(gpu2, ref2, k, v, list(range(1025)))
    for a, b in zip(one_bits, [to_bits(t) for t in tok]):
        assert a.tobytes() == b.tobytes()
    assert gpu2.stats()["offset"] == 1024
    # an independent check on the plain fp64 norms: same kept set unless the
    # two cutoff-adjacent norms are within twice the score tolerance
    plain = oscores.key_norm_plain(k)[0, 0]
    keep_plain = osel.kept_indices(osel.priority(plain, True)[None, None], 4, 0, 512)[0, 0]
    srt = np.sort(plain[4:])
    gap = srt[508] - srt[507]
    if gap > 2e-5 * srt[508]:
        assert np.array_equal(to_bits(one[2])[0, 0], keep_plain)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("method,extra", [("knorm", {"keep_low": True}), ("knorm", {"keep_low": False}),
                                          ("qfilters", {"sign": 1}), ("qfilters", {"sign": -1})])
@pytest.mark.parametrize("shape", [
    # (B, H, budget, n_sink, recent, cuts)
    (2, 3, 64, 4, 0, [0, 300]),                  # one block, ragged tail (300 = 4*64 + 44)
    (1, 2, 64, 4, 8, [0, 30, 70, 71, 200, 201]), # append, cross, single-token steps, recent window
    (3, 1, 100, 0, 5, [0, 99, 100, 101, 400]),   # exact boundary, n_sink 0
    (1, 1, 33, 1, 1, [0, 1, 2, 40, 41, 42, 1000]),
])
def test_parity_small_shapes(dtype, method, extra, shape):
    B, H, budget, n_sink, recent, cuts = shape
    k, v = synth.gaussian_block(100 + budget + B + H, B, H, cuts[-1], dtype=dtype, scale=2.0)
    kw = dict(n_sink=n_sink, recent=recent, **extra)
    if method == "qfilters":
        kw["filters"] = synth.unit_vectors(synth.rng(9), H).astype(np.float32)
    gpu, ref = _pair(method, B, H, budget, dtype=dtype, max_block=1024, **kw)
    _feed(gpu, ref, k, v, cuts, check_each=True, what=f"{method} {dtype} {shape}")
    assert gpu.stats() == ref.stats()


@pytest.mark.parametrize("method", ["knorm", "qfilters"])
def test_ties_nan_signed_zero_and_infinity(method):
    # rows from a tiny pool of keys: many exact ties; a few special rows
    B, H, S = 2, 2, 700
    g = synth.rng(77)
    pool = synth.f32_to_bf16_bits(g.standard_normal((5, 128)).astype(np.float32))
    idx = g.integers(0, 5, size=(B, H, S))
    k = pool[idx]
    k[0, 0, 10] = 0                                   # zero key: norm 0, projection +0
    k[0, 0, 11] = 0x8000                              # -0 entries: projection may be -0
    k[0, 1, 50, 3] = 0x7FC0                           # NaN -> evicted first
    k[1, 0, 60, 7] = 0x7F80                           # +inf entry
    k[1, 1, 70, 7] = 0xFF80                           # -inf entry
    v = synth.f32_to_bf16_bits(g.standard_normal((B, H, S, 128)).astype(np.float32))
    kw = dict(n_sink=3, recent=2)
    if method == "qfilters":
        kw.update(filters=synth.unit_vectors(synth.rng(5), H).astype(np.float32), sign=1)
    gpu, ref = _pair(method, B, H, 128, max_block=1024, **kw)
    _feed(gpu, ref, k, v, [0, 400, 401, 700], check_each=True, what="ties")


@pytest.mark.parametrize("method", ["knorm", "qfilters"])
@pytest.mark.parametrize("B,H,S,budget", [(1, 3, 9000, 3000), (1, 3, 14000, 700), (1, 3, 30000, 5000),
                                          (1, 3, 70000, 4000), (8, 6, 10000, 2000)])
def test_ties_in_large_selections(method, B, H, S, budget):
    # more than 4096 rows per unit: the register selection with 8 to 24 keys per thread and, past
    # 24576 rows, the shared-memory one; tie pools, NaN, +-0 and +-inf rows lie on both sides of
    # thread-segment boundaries, and a second block makes the kept rows move
    g = synth.rng(78 + S)
    pool = synth.f32_to_bf16_bits(g.standard_normal((7, 128)).astype(np.float32))
    k = pool[g.integers(0, 7, size=(B, H, S))]
    for r in (4095, 4096, 4097, 8191, 8192, S - 3):
        k[0, 0, r] = 0                                # zero keys at CTA boundaries
    k[0, 1, 4096, 5] = 0x7FC0                         # NaN
    k[0, 1, 4095, 5] = 0x7F80                         # +inf entry
    k[0, 2, 8192, 9] = 0xFF80                         # -inf entry
    k[0, 2, 100:140, :] = 0x8000                      # -0 keys
    v = synth.f32_to_bf16_bits(g.standard_normal((B, H, S, 128)).astype(np.float32))
    kw = dict(n_sink=5, recent=7)
    if method == "qfilters":
        kw.update(filters=synth.unit_vectors(synth.rng(6), H).astype(np.float32), sign=-1)
    cut = S // 2
    gpu, ref = _pair(method, B, H, budget, max_block=S - cut, **kw)
    _feed(gpu, ref, k, v, [0, cut, S], check_each=True, what=f"large-selection ties S={S}")


@pytest.mark.parametrize("method,extra", [("knorm", {"keep_low": True}), ("knorm", {"keep_low": False}),
                                          ("qfilters", {"sign": 1}), ("qfilters", {"sign": -1})])
def test_large_selections_odd_sizes_and_equal_units(method, extra):
    # register selections of 8000 and 9002 rows with an odd budget, storage and kept count (scalar
    # score loads; compaction chunks that start inside a thread's rows): continuous scores end
    # the radix passes once the whole bin is admitted (two-signed projections take up to three
    # passes); head 1 holds one key repeated (every candidate equal: no pass at all); NaN and
    # +-inf rows sit at thread boundaries
    B, H, S, budget = 2, 3, 14001, 3001
    g = synth.rng(4242)
    k = synth.f32_to_bf16_bits((g.standard_normal((B, H, S, 128)) * 1.5).astype(np.float32))
    k[:, 1] = k[0, 1, 17]                             # every row of head 1 equal
    k[0, 0, 2999, 3] = 0x7FC0                         # NaN in the first kept block's last row
    k[0, 2, 8191, 7] = 0x7F80                         # +inf entry
    k[1, 2, 8192, 7] = 0xFF80                         # -inf entry
    k[1, 0, 4000:4016, :] = 0x8000                    # -0 keys
    v = synth.f32_to_bf16_bits(g.standard_normal((B, H, S, 128)).astype(np.float32))
    kw = dict(n_sink=3, recent=5, **extra)
    if method == "qfilters":
        kw["filters"] = synth.unit_vectors(synth.rng(8), H).astype(np.float32)
    gpu, ref = _pair(method, B, H, budget, max_block=6001, **kw)
    _feed(gpu, ref, k, v, [0, 2999, 8000, 14001], check_each=True, what=f"odd sizes {method} {extra}")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("method,extra", [("knorm", {"keep_low": True}), ("knorm", {"keep_low": False}),
                                          ("qfilters", {"sign": -1})])
def test_single_eviction_blocks(dtype, method, extra):
    """Blocks that overshoot the budget by exactly one row take the fused
    single-eviction kernel (m <= 64); m = 65 takes the general path. Both
    must give the oracle's cache bit for bit."""
    from kv_cache_token_bf16_gb300 import binding
    B, H, budget = 2, 3, 96
    k, v = synth.gaussian_block(501, B, H, 400, dtype=dtype, scale=2.0)
    kw = dict(n_sink=4, recent=6, **extra)
    if method == "qfilters":
        kw["filters"] = synth.unit_vectors(synth.rng(19), H).astype(np.float32)
    for cuts in ([0, 90, 97, 98, 99, 163, 164], [0, 33, 97, 98], [0, 32, 97, 98]):
        gpu, ref = _pair(method, B, H, budget, dtype=dtype, max_block=128, **kw)
        binding.evict_set_profiling(gpu.handle, True)
        _feed(gpu, ref, k, v, cuts, check_each=True, what=f"{method} {dtype} {cuts}")
        used = binding.evict_kernel_times(gpu.handle)
        assert "evict1" in used                           # the m <= 64 single evictions
        assert gpu.stats() == ref.stats()
        gpu.close()


@pytest.mark.parametrize("method", ["knorm", "qfilters"])
def test_single_eviction_ties_and_nan(method):
    """All-equal keys evict the highest unprotected index; a NaN score is evicted first."""
    B, H, budget = 1, 2, 40
    g = synth.rng(31)
    key = synth.f32_to_bf16_bits(g.standard_normal(128).astype(np.float32))
    k = np.broadcast_to(key, (B, H, 60, 128)).copy()
    k[0, 1, 45, 9] = 0x7FC0                               # NaN in the row that arrives at step 45
    v = synth.f32_to_bf16_bits(g.standard_normal((B, H, 60, 128)).astype(np.float32))
    kw = dict(n_sink=2, recent=3)
    if method == "qfilters":
        kw.update(filters=synth.unit_vectors(synth.rng(3), H).astype(np.float32), sign=1)
    gpu, ref = _pair(method, B, H, budget, max_block=64, **kw)
    _feed(gpu, ref, k, v, [0] + list(range(budget, 61)), check_each=True, what="single-eviction ties")


def test_all_scores_equal_keeps_exactly_budget_lowest_indices():
    B, H, S = 1, 4, 500
    row = synth.f32_to_bf16_bits(np.linspace(-1, 1, 128, dtype=np.float32))
    k = np.broadcast_to(row, (B, H, S, 128)).copy()
    v = synth.gaussian_block(3, B, H, S)[1]
    gpu, ref = _pair("knorm", B, H, 100, n_sink=4, recent=6)
    view = _feed(gpu, ref, k, v, [0, 500])
    assert_cache_equal(view, ref, "all equal")
    pos = to_bits(view[2])
    assert np.array_equal(pos[0, 0], np.r_[np.arange(94), np.arange(494, 500)])


def test_explicit_positions_and_host_inputs():
    from kv_cache_token_bf16_gb300 import binding
    B, H = 2, 2
    k, v = synth.gaussian_block(12, B, H, 300)
    pos = (np.arange(300)[None, :] * np.array([[3], [5]]) + 7).astype(np.int32)
    gpu, ref = _pair("knorm", B, H, 64, n_sink=2, recent=3)
    view = gpu.update_and_fetch(to_dev(k, torch), to_dev(v, torch), torch.from_numpy(pos).cuda())
    ref.update_and_fetch(k, v, pos=pos)
    gpu.sync()
    assert_cache_equal(view, ref, "explicit positions")
    # same block through the host-buffer entry point
    gpu2 = binding.EvictCache("knorm", B, H, budget=64, n_sink=2, recent=3, max_block=8192)
    kh = torch.from_numpy(k.view(np.int16)).pin_memory()
    vh = torch.from_numpy(v.view(np.int16)).pin_memory()
    ph = torch.from_numpy(pos).pin_memory()
    vw = binding.evict_update_and_fetch_host(gpu2.handle, kh.data_ptr(), vh.data_ptr(), ph.data_ptr(), 300)
    gpu2.sync()
    assert_cache_equal(binding.view_tensors(vw, B, H, "bf16"), ref, "host inputs")


def test_set_state_then_evict_from_an_oversized_cache():
    # a pre-existing cache larger than the budget (max_kept) is cut to budget
    B, H, S0, m = 2, 2, 1500, 100
    k, v = synth.gaussian_block(13, B, H, S0 + m)
    pos0 = np.broadcast_to(np.arange(S0, dtype=np.int32), (B, H, S0)).copy()
    score0 = oscores.key_norm_canonical(k[:, :, :S0])
    gpu, ref = _pair("knorm", B, H, 256, n_sink=4, recent=0, max_kept=S0)
    gpu.set_state(to_dev(k[:, :, :S0], torch), to_dev(v[:, :, :S0], torch), torch.from_numpy(pos0).cuda(),
                  torch.from_numpy(score0).cuda(), S0)
    ref.set_state(k[:, :, :S0], v[:, :, :S0], pos0, score0, S0)
    view = _feed(gpu, ref, k[:, :, S0:], v[:, :, S0:], [0, m])
    assert_cache_equal(view, ref, "set_state")


def test_update_errors_are_reported():
    from kv_cache_token_bf16_gb300 import binding
    gpu = binding.EvictCache("knorm", 1, 1, budget=16, max_block=8)
    k, v = synth.gaussian_block(1, 1, 1, 9)
    with pytest.raises(binding.EvictError) as e:
        gpu.update_and_fetch(to_dev(k, torch), to_dev(v, torch))
    assert e.value.code == binding.EVICT_EINVAL
    view = gpu.update_and_fetch(to_dev(k[:, :, :0], torch), to_dev(v[:, :, :0], torch))   # m = 0
    assert view[2].shape[2] == 0 and gpu.stats()["offset"] == 0


def test_two_runs_are_bit_identical():
    k, v = synth.gaussian_block(14, 4, 4, 3000)
    outs = []
    for _ in range(2):
        gpu, ref = _pair("knorm", 4, 4, 512, n_sink=4, recent=16)
        view = None
        for a in range(0, 3000, 700):
            view = gpu.update_and_fetch(to_dev(k[:, :, a:a + 700], torch), to_dev(v[:, :, a:a + 700], torch))
        gpu.sync()
        outs.append([to_bits(t).copy() for t in view])
    for a, b in zip(*outs):
        assert a.tobytes() == b.tobytes()


# ---------------------------------------------------------------------------
# Q-Filters calibrated layer stack (B=1, H_kv=8, S=8192, budget 1024, n_sink 4)
# ---------------------------------------------------------------------------
def _layer_filters(layer):
    # filters come from the ORACLE's calibration (fp64 -> fp32), never from the GPU
    return ocal.calibrate(layer["queries"], 8).astype(np.float32)


def test_qfilters_layer_full_size_single_and_grouped():
    from kv_cache_token_bf16_gb300 import binding
    layers = [synth.qfilters_layer(l) for l in range(3)]
    filts = [_layer_filters(L) for L in layers]
    kw = dict(n_sink=4, recent=0, sign=1)
    # single-layer calls
    refs = []
    for L, f in zip(layers, filts):
        gpu, ref = _pair("qfilters", 1, 8, 1024, filters=f, **kw)
        view = _feed(gpu, ref, L["k"], L["v"], [0, 8192])
        assert_cache_equal(view, ref, "qfilters layer")
        refs.append(ref)
        # the plain fp64 projection selects the same set unless the cutoff pair is within tolerance
        plain = oscores.projection_plain(L["k"], f, 1)[0]
        cond = oscores.projection_condition(L["k"], f)[0]
        for h in range(8):
            p = plain[h, 4:]
            order = np.argsort(-p, kind="stable")
            a, b = order[1019], order[1020]
            tol = 1e-5 * max(abs(p[a]), cond[h, 4 + a])
            if p[a] - p[b] > 2 * tol:
                kept_plain = np.sort(np.r_[np.arange(4), 4 + order[:1020]])
                assert np.array_equal(to_bits(view[2])[0, h], kept_plain)
    # grouped: one set of launches for the three layers
    caches = [binding.EvictCache("qfilters", 1, 8, budget=1024, max_block=8192, filters=f, **kw) for f in filts]
    ks = [to_dev(L["k"], torch) for L in layers]
    vs = [to_dev(L["v"], torch) for L in layers]
    views = binding.evict_update_and_fetch_group([c.handle for c in caches], [t.data_ptr() for t in ks],
                                                 [t.data_ptr() for t in vs], None, 8192)
    caches[0].sync()
    for vw, ref in zip(views, refs):
        assert_cache_equal(binding.view_tensors(vw, 1, 8, "bf16"), ref, "grouped")


# ---------------------------------------------------------------------------
# Decode streaming (B=32, H=8, prefill 2048 then 4096 single-token steps,
# budget 512, n_sink 4, recent 128): full shape. The first 300 steps are
# checked against a full-width oracle every 50 steps; from there three
# sampled (b, h) units are followed by their own oracles to the end of the
# stream, checked every 256 steps and at the last one.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("method", ["knorm", "qfilters"])
def test_decode_stream(method):
    B, H, steps, full_width = 32, 8, 4096, 300
    k0, v0 = synth.decode_prefill(B, H, 2048)
    ks, vs = synth.decode_steps(0, steps, B, H)
    kw = dict(n_sink=4, recent=128)
    filt = synth.decode_filters(H)
    kw.update({"keep_low": True} if method == "knorm" else {"filters": filt, "sign": 1})
    gpu, ref = _pair(method, B, H, 512, max_block=2048, **kw)
    _feed(gpu, ref, k0, v0, [0, 2048], check_each=True, what="prefill")
    kd, vd = to_dev(ks, torch), to_dev(vs, torch)
    units = [(0, 0), (17, 3), (31, 7)]
    subs = {}
    for s in range(steps):
        view = gpu.update_and_fetch(kd[s], vd[s])
        if s < full_width:
            ref.update_and_fetch(ks[s], vs[s])
            if (s + 1) % 50 == 0:
                gpu.sync()
                assert_cache_equal(view, ref, f"decode step {s}")
            if s + 1 == full_width:
                for (b, h) in units:      # the sampled units continue on oracles of their own
                    ukw = dict(kw)
                    if method == "qfilters":
                        ukw["filters"] = filt[h:h + 1]
                    sub = OracleCache(method, 1, 1, budget=512, **ukw)
                    sub.set_state(ref.k[b:b + 1, h:h + 1], ref.v[b:b + 1, h:h + 1], ref.pos[b:b + 1, h:h + 1],
                                  ref.score[b:b + 1, h:h + 1], ref.offset)
                    subs[(b, h)] = sub
            continue
        for (b, h), sub in subs.items():
            sub.update_and_fetch(ks[s][b:b + 1, h:h + 1], vs[s][b:b + 1, h:h + 1])
        if (s + 1) % 256 == 0 or s + 1 == steps:
            gpu.sync()
            gk, gv, gp, gs = [to_bits(t) for t in view]
            assert gp.shape == (B, H, 512) and np.all(np.diff(gp, axis=2) > 0)
            assert np.all(gp[:, :, :4] == np.arange(4))
            assert np.all(gp[:, :, -128:] == 2048 + s - 127 + np.arange(128))     # the recent window
            for (b, h), sub in subs.items():
                what = f"decode step {s} unit {(b, h)}"
                assert np.array_equal(gp[b, h], sub.pos[0, 0]), what
                assert np.array_equal(gk[b, h], sub.k[0, 0]) and np.array_equal(gv[b, h], sub.v[0, 0]), what
                assert gs[b, h].tobytes() == sub.score[0, 0].astype(np.float32).tobytes(), what
    assert gpu.stats()["offset"] == 2048 + steps


# ---------------------------------------------------------------------------
# Long-context chunked prefill (B=4, H=8, 8192-token blocks, budget 4096):
# full size; the oracle follows 3 sampled (b, h) units through 16 blocks.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("method", ["knorm", "qfilters"])
def test_long_context_full_size_sampled_units(method):
    B, H, blocks = 4, 8, 16
    kw = dict(n_sink=4, recent=0)
    if method == "qfilters":
        filt = ocal.calibrate(synth.long_context_queries(H), H).astype(np.float32)
        kw.update(filters=filt, sign=1)
    else:
        kw.update(keep_low=True)
    from kv_cache_token_bf16_gb300 import binding
    gpu = binding.EvictCache(method, B, H, budget=4096, max_block=8192, **kw)
    units = [(0, 0), (1, 5), (3, 7)]
    refs = {}
    for (b, h) in units:
        ukw = dict(kw)
        if method == "qfilters":
            ukw["filters"] = filt[h:h + 1]
        refs[(b, h)] = OracleCache(method, 1, 1, budget=4096, **ukw)
    for blk in range(blocks):
        k, v = synth.long_context_block(blk, B, H)
        view = gpu.update_and_fetch(to_dev(k, torch), to_dev(v, torch))
        for (b, h), ref in refs.items():
            ref.update_and_fetch(k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1])
        gpu.sync()
        gk, gv, gp, gs = [to_bits(t) for t in view]
        assert gp.shape[2] == min(4096, 8192 * (blk + 1))
        assert np.all(np.diff(gp, axis=2) > 0)                      # temporal order everywhere
        assert np.all(gp[:, :, :4] == np.arange(4))                 # sinks everywhere
        for (b, h), ref in refs.items():
            assert np.array_equal(gp[b, h], ref.pos[0, 0]), (blk, b, h)
            assert np.array_equal(gk[b, h], ref.k[0, 0]) and np.array_equal(gv[b, h], ref.v[0, 0])
            assert gs[b, h].tobytes() == ref.score[0, 0].tobytes()
    assert gpu.stats()["offset"] == blocks * 8192


def test_small_cache_created_after_a_large_one_does_not_break_it():
    # the select kernel's shared-memory limit is per function, not per cache
    from kv_cache_token_bf16_gb300 import binding
    k, v = synth.gaussian_block(15, 1, 2, 8192)
    gpu, ref = _pair("knorm", 1, 2, 4096, n_sink=4)
    small = binding.EvictCache("knorm", 1, 1, budget=16, n_sink=1, max_block=16)
    view = _feed(gpu, ref, k, v, [0, 8192])
    assert_cache_equal(view, ref, "large after small")
    small.close()


@pytest.mark.parametrize("method", ["knorm", "qfilters"])
def test_more_units_than_sms_uses_two_ctas_per_sm(method):
    # 160 (b, h) units (more than the 152 SMs) with 2048 < n <= 8192 take the 512-thread
    # selection variant; a prefill and a second block with kept rows
    B, H = 20, 8
    k, v = synth.gaussian_block(61, B, H, 5000)
    kw = dict(n_sink=4, recent=8)
    kw.update({"keep_low": True} if method == "knorm" else {"filters": synth.decode_filters(H), "sign": -1})
    gpu, ref = _pair(method, B, H, 700, max_block=3000, **kw)
    view = _feed(gpu, ref, k, v, [0, 3000, 5000], check_each=True, what="160 units")
    assert_cache_equal(view, ref, "160 units")


def test_host_inputs_back_to_back_calls_and_layers():
    # successive host-buffer calls reuse each handle's staging buffers; the copy stream must wait
    # for the previous call's kernels, and one layer's kernels overlap the next layer's copies
    from kv_cache_token_bf16_gb300 import binding
    B, H, L = 2, 4, 3
    data = [synth.gaussian_block(70 + l, B, H, 900) for l in range(L)]
    cuts = [0, 400, 700, 900]
    kw = dict(n_sink=4, recent=8, keep_low=True)
    caches = [binding.EvictCache("knorm", B, H, budget=256, max_block=400, **kw) for _ in range(L)]
    refs = [OracleCache("knorm", B, H, budget=256, **kw) for _ in range(L)]
    hosts = []
    views = [None] * L
    for a, b in zip(cuts[:-1], cuts[1:]):
        for l, (k, v) in enumerate(data):
            kh = torch.from_numpy(np.ascontiguousarray(k[:, :, a:b]).view(np.int16)).pin_memory()
            vh = torch.from_numpy(np.ascontiguousarray(v[:, :, a:b]).view(np.int16)).pin_memory()
            hosts.append((kh, vh))                       # kept alive until the stream passes the call
            views[l] = binding.evict_update_and_fetch_host(caches[l].handle, kh.data_ptr(), vh.data_ptr(), None,
                                                           b - a)
            refs[l].update_and_fetch(k[:, :, a:b], v[:, :, a:b])
    for c, ref, vw in zip(caches, refs, views):
        c.sync()
        assert_cache_equal(binding.view_tensors(vw, B, H, "bf16"), ref, "host calls")
