"""GPU parity of the CurDKV-adapted path against the CPU oracle.

Compared per (b, h):
* proxy-attention column sums: relative 1e-4 (fp32 tensor-core logits,
  fp32 sums of ex2 terms);
* captured energy (sum of the leverage = the top-r eigenvalues' share of
  tr G, well-conditioned at any gap): relative 1e-4;
* leverage, wherever the oracle's rank-r eigengap
  g = (lambda_{r-1} - lambda_r) / lambda_0 is at least 1e-2: relative 1e-3
  (+ 1e-9 * sum l);
* leverage below that gap, where the top-r subspace is ill-conditioned: a
  Davis-Kahan bound. The GPU's Gram is built from its own attention sums,
  which differ from the oracle's by the measured relative delta; so
  |G_gpu - G| <= eps * |G| with eps = 2 delta + 2e-5 (the split-bf16 Gram
  and the eigensolver's backward error), the subspace turns by at most
  sin(theta) <= eps / g, and row i's leverage w_i^T P w_i / E moves by at
  most sin(theta) |w_i|^2 / E plus the row's own rescaling (4 delta + 1e-4)
  l_i; the bound never exceeds |w_i|^2 / E, the largest any leverage can be;
* kept sets: equal counts, and every row whose oracle priority lies more
  than twice its tolerance (plus the cutoff row's) from the cutoff is kept
  by both or by neither; the compacted K/V/positions are the original rows
  of the kept positions.
The oracle never receives GPU output: multi-block cases start every block
from the oracle's own state (loaded into the GPU cache with evict_set_state).
"""
import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import synth
from oracle import curdkv as ocd
from oracle.bf16 import to_f64
from oracle import select as osel
from oracle.cache import OracleCache
from tests.gpu_util import to_bits, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

RANK = 16


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _gpu_cache(B, H, budget, max_block, max_kept=0, n_sink=4, recent=0, rank=RANK):
    from kv_cache_token_bf16_gb300 import binding
    return binding.EvictCache("curdkv", B, H, budget=budget, n_sink=n_sink, recent=recent, max_block=max_block,
                              max_kept=max_kept, rank_cap=rank)


def _gpu_scores(cache, B, H):
    from kv_cache_token_bf16_gb300 import binding
    n = binding.evict_curdkv_scores(cache.handle, None, None)
    attn = torch.empty((B, H, n), dtype=torch.float32, device="cuda")
    lev = torch.empty_like(attn)
    binding.evict_curdkv_scores(cache.handle, attn.data_ptr(), lev.data_ptr())
    cache.sync()
    return attn.cpu().numpy().astype(np.float64), lev.cpu().numpy().astype(np.float64)


def leverage_tolerance(attn_g, a_or, v_all, l_or, s, rank):
    """Per-row bound on |l_gpu - l_oracle| and the rank-r relative gap (module docstring)."""
    n = len(l_or)
    lam = s ** 2
    r = min(rank, n, 128)
    gap = (lam[r - 1] - lam[r]) / lam[0] if lam[0] > 0 and r < len(lam) else 1.0
    if gap >= 1e-2:
        return 1e-3 * l_or + 1e-9 * l_or.sum(), gap
    x = to_f64(v_all)
    w2 = a_or ** 2 * np.sum(x * x, axis=1)
    e = w2.sum()
    if e == 0:
        return np.full(n, 1e-12), gap
    pos = a_or > 0
    delta = float(np.max(np.abs(attn_g[pos] / a_or[pos] - 1.0))) if pos.any() else 0.0
    eps = 2 * delta + 2e-5
    sin_t = min(1.0, eps / gap) if gap > 0 else 1.0
    tol = (4 * delta + 1e-4) * l_or + sin_t * w2 / e + 1e-9 * l_or.sum()
    return np.minimum(tol, w2 / e + 1e-9 * l_or.sum()), gap


def _check_unit(k_all, v_all, m, attn_g, lev_g, cum_old, cum_g_all, kept_g, n_sink, recent, budget, what,
                rank=RANK, oracle=None):
    """Compare one (b, h) unit with the oracle. ``oracle`` may hold block_scores' result for these rows.
    Returns (rank-r relative gap, the oracle's cumulative scores, the oracle's kept indices)."""
    l_or, a_or, s = oracle if oracle is not None else ocd.block_scores(k_all, v_all, m, rank)
    n = len(l_or)
    assert np.allclose(attn_g, a_or, rtol=1e-4, atol=1e-7 * m), f"{what}: attention sums"
    assert abs(lev_g.sum() - l_or.sum()) <= 1e-4 * l_or.sum() + 1e-12, f"{what}: captured energy"
    tol, gap = leverage_tolerance(attn_g, a_or, v_all, l_or, s, rank)
    bad = np.abs(lev_g - l_or) > tol
    assert not bad.any(), f"{what}: leverage off at {np.flatnonzero(bad)[:5]} (gap {gap:.3g})"
    # kept set, band-tolerant around the oracle's cutoff (stored cumulative scores are fp32)
    cum_or = ocd.cumulative(cum_old, l_or)
    ctol = tol + 2.4e-7 * np.abs(cum_or)
    kept_or = np.arange(n)
    if n > budget:
        kept_or = osel.kept_indices(osel.priority(cum_or)[None, None], n_sink, recent, budget)[0, 0]
        assert len(kept_g) == budget
        prot = osel.protected_mask(n, n_sink, recent)
        unp = np.flatnonzero(~prot)
        q = budget - prot.sum()
        order = unp[np.argsort(-cum_or[unp], kind="stable")]
        cut = order[q - 1]
        clear = np.abs(cum_or - cum_or[cut]) > 2 * (ctol + ctol[cut])
        in_or = np.isin(np.arange(n), kept_or)
        in_g = np.isin(np.arange(n), kept_g)
        assert np.array_equal(in_or[clear], in_g[clear]), f"{what}: kept set differs outside the band"
    return gap, cum_or, kept_or


def _run_block(B, H, budget, k_old, v_old, cum_old, k_new, v_new, n_sink=4, recent=0, units=None, rank=RANK):
    """One GPU update starting from the oracle-provided state; checks every (or the listed) unit."""
    k0 = k_old.shape[2]
    m = k_new.shape[2]
    gpu = _gpu_cache(B, H, budget, max_block=m, max_kept=max(k0, budget), n_sink=n_sink, recent=recent, rank=rank)
    if k0:
        pos0 = np.broadcast_to(np.arange(k0, dtype=np.int32), (B, H, k0)).copy()
        gpu.set_state(to_dev(k_old, torch), to_dev(v_old, torch), torch.from_numpy(pos0).cuda(),
                      torch.from_numpy(cum_old.astype(np.float32)).cuda(), k0)
    view = gpu.update_and_fetch(to_dev(k_new, torch), to_dev(v_new, torch))
    gpu.sync()
    attn, lev = _gpu_scores(gpu, B, H)
    gk, gv, gp, gs = [to_bits(t) for t in view]
    k_all = np.concatenate([k_old, k_new], axis=2)
    v_all = np.concatenate([v_old, v_new], axis=2)
    gaps = []
    for b in range(B):
        for h in range(H):
            if units is not None and (b, h) not in units:
                continue
            kept = gp[b, h]
            assert np.all(np.diff(kept) > 0)
            assert np.array_equal(gk[b, h], k_all[b, h, kept]) and np.array_equal(gv[b, h], v_all[b, h, kept])
            gaps.append(_check_unit(k_all[b, h], v_all[b, h], m, attn[b, h], lev[b, h],
                                    cum_old[b, h].astype(np.float32).astype(np.float64), None, kept, n_sink,
                                    recent, budget, f"unit {(b, h)}", rank)[0])
    return gpu, view, attn, lev, gaps


@pytest.mark.parametrize("k0,m,budget", [(0, 300, 64), (0, 129, 200), (500, 257, 128), (1000, 1, 64),
                                         (127, 128, 100), (0, 513, 100), (300, 1100, 256), (129, 640, 700),
                                         # short blocks: the fused one-CTA-per-unit attention (m <= 8 and
                                         # m * n <= 16384), its boundary, and the tensor-core path just past it
                                         (0, 1, 64), (600, 5, 128), (2040, 8, 512), (2041, 8, 512), (3, 8, 6),
                                         (700, 9, 128)])
def test_planted_spectrum_block(k0, m, budget):
    B, H = 1, 2
    n = k0 + m
    k_all = synth.clustered_keys(100 + n, B, H, n, spread=0.5)
    v_all = synth.planted_spectrum_values(200 + n, B, H, n)
    cum_old = synth.rng(3).uniform(0, 0.01, (B, H, k0))
    gpu, view, attn, lev, gaps = _run_block(B, H, budget, k_all[:, :, :k0], v_all[:, :, :k0], cum_old,
                                            k_all[:, :, k0:], v_all[:, :, k0:])
    assert min(gaps) >= 1e-2           # the planted spectrum keeps the leverage well-conditioned


@pytest.mark.parametrize("rank", [1, 8, 16, 17, 24, 32])
def test_rank_caps_on_both_eigensolver_layouts(rank):
    # ranks up to 16 run the eigensolver's small layout (two CTAs per SM), larger ranks the
    # 32-vector one; a slower spectral decay keeps a clear gap after the r-th direction
    B, H, k0, m, budget = 1, 3, 200, 180, 128
    n = k0 + m
    k_all = synth.clustered_keys(600 + rank, B, H, n, spread=0.5)
    v_all = synth.planted_spectrum_values(700 + rank, B, H, n, rank=rank, decay=0.95)
    cum_old = synth.rng(7).uniform(0, 0.01, (B, H, k0))
    *_, gaps = _run_block(B, H, budget, k_all[:, :, :k0], v_all[:, :, :k0], cum_old, k_all[:, :, k0:],
                          v_all[:, :, k0:], rank=rank)
    assert min(gaps) >= 1e-2


def test_append_then_evict_accumulates_leverage():
    # blocks of 60 into budget 200: three appends then an eviction, cumulative scores tracked
    B, H, blk = 1, 2, 60
    k_all = synth.clustered_keys(7, B, H, 4 * blk, spread=0.5)
    v_all = synth.planted_spectrum_values(8, B, H, 4 * blk)
    gpu = _gpu_cache(B, H, 200, max_block=blk)
    ref = OracleCache("curdkv", B, H, budget=200, n_sink=4, rank_cap=RANK)
    for c in range(4):
        sl = slice(c * blk, (c + 1) * blk)
        view = gpu.update_and_fetch(to_dev(k_all[:, :, sl], torch), to_dev(v_all[:, :, sl], torch))
        ref.update_and_fetch(k_all[:, :, sl], v_all[:, :, sl])
        gpu.sync()
        gp, gs = to_bits(view[2]), to_bits(view[3]).astype(np.float64)
        assert gp.shape == ref.pos.shape
        if c < 3:
            assert np.array_equal(gp, ref.pos)
            assert np.allclose(gs, ref.score, rtol=2e-3, atol=1e-9), f"cumulative scores after block {c}"
    assert gpu.stats()["offset"] == 4 * blk and gpu.stats()["tokens_kept"] == 200


def test_zero_values_give_zero_leverage_and_index_ties():
    B, H, n = 1, 1, 300
    k = synth.clustered_keys(9, B, H, n)
    v = np.zeros((B, H, n, 128), np.uint16)
    gpu = _gpu_cache(B, H, 50, max_block=n)
    view = gpu.update_and_fetch(to_dev(k, torch), to_dev(v, torch))
    gpu.sync()
    attn, lev = _gpu_scores(gpu, B, H)
    assert np.all(lev == 0) and np.all(np.isfinite(attn))
    assert to_bits(view[2])[0, 0].tolist() == list(range(50))     # all tie: lowest indices kept


def test_identical_keys_different_values_diverge():
    # rows 30 and 31 are kept rows (seen by every query) with equal keys
    B, H, k0, m = 1, 1, 48, 16
    k = synth.clustered_keys(10, B, H, k0 + m)
    v = synth.planted_spectrum_values(11, B, H, k0 + m)
    k[0, 0, 31] = k[0, 0, 30]
    v[0, 0, 31] = synth.f32_to_bf16_bits(0.01 * synth.bf16_bits_to_f32(v[0, 0, 30]))
    gpu, view, attn, lev, gaps = _run_block(B, H, 128, k[:, :, :k0], v[:, :, :k0], np.zeros((B, H, k0)),
                                            k[:, :, k0:], v[:, :, k0:])
    assert attn[0, 0, 30] == attn[0, 0, 31]
    assert lev[0, 0, 30] > 100 * lev[0, 0, 31]


def test_planted_geometry_class1_fills_the_budget_small():
    B, H, S0, m = 2, 2, 3000, 128
    p = synth.curdkv_planted(B, H, existing=S0, incoming=m, seed=5)
    cum0 = np.zeros((B, H, S0))
    gpu, view, attn, lev, gaps = _run_block(B, H, 256, p["k"][:, :, :S0], p["v"][:, :, :S0], cum0,
                                            p["k"][:, :, S0:], p["v"][:, :, S0:])
    gp = to_bits(view[2])
    for b in range(B):
        for h in range(H):
            assert np.all(p["cls"][b, h, gp[b, h, 4:]] == 1)


def test_planted_geometry_full_size_sampled_units():
    # 8 x 8 heads, 16384 existing rows + a 512-token block, budget 2048, n_sink 4
    B, H, S0, m = 8, 8, 16384, 512
    p = synth.curdkv_planted(B, H, existing=S0, incoming=m)
    cum0 = np.zeros((B, H, S0))
    gpu, view, attn, lev, gaps = _run_block(B, H, 2048, p["k"][:, :, :S0], p["v"][:, :, :S0], cum0,
                                            p["k"][:, :, S0:], p["v"][:, :, S0:], units={(0, 0), (5, 3), (7, 7)})
    gp = to_bits(view[2])
    assert gp.shape == (B, H, 2048)
    for b in range(B):
        for h in range(H):
            assert np.all(p["cls"][b, h, gp[b, h, 4:]] == 1), (b, h)


def test_single_token_steps_after_prefill():
    B, H = 1, 2
    k_all = synth.clustered_keys(12, B, H, 140)
    v_all = synth.planted_spectrum_values(13, B, H, 140)
    ref = OracleCache("curdkv", B, H, budget=64, n_sink=4, rank_cap=RANK)
    ref.update_and_fetch(k_all[:, :, :128], v_all[:, :, :128])
    for t in range(128, 140):
        # every step starts from the oracle's state
        _run_block(B, H, 64, ref.k, ref.v, ref.score, k_all[:, :, t:t + 1], v_all[:, :, t:t + 1])
        ref.update_and_fetch(k_all[:, :, t:t + 1], v_all[:, :, t:t + 1])


def test_two_runs_are_bit_identical():
    B, H, n = 2, 2, 700
    k = synth.clustered_keys(14, B, H, n)
    v = synth.planted_spectrum_values(15, B, H, n)
    outs = []
    for _ in range(2):
        gpu = _gpu_cache(B, H, 128, max_block=n)
        view = gpu.update_and_fetch(to_dev(k, torch), to_dev(v, torch))
        gpu.sync()
        outs.append([to_bits(t).copy() for t in view] + list(_gpu_scores(gpu, B, H)))
    for a, b in zip(*outs):
        assert a.tobytes() == b.tobytes()


def test_units_shared_by_several_ctas():
    """Many (b, h) units with long kept prefixes: the attention passes split
    units across CTAs (several pass-1 partials per query) and, with m > 512,
    across query quads (merged column sums)."""
    B, H, k0, m, budget = 2, 4, 3000, 600, 1024
    n = k0 + m
    k_all = synth.clustered_keys(11, B, H, n, spread=0.5)
    v_all = synth.planted_spectrum_values(12, B, H, n)
    cum_old = synth.rng(13).uniform(0, 0.01, (B, H, k0))
    _run_block(B, H, budget, k_all[:, :, :k0], v_all[:, :, :k0], cum_old, k_all[:, :, k0:], v_all[:, :, k0:],
               units={(0, 0), (1, 3)})


def test_misaligned_inputs_are_rejected():
    from kv_cache_token_bf16_gb300 import binding
    B, H, m = 1, 2, 16
    cache = _gpu_cache(B, H, budget=64, max_block=m)
    buf = torch.zeros((B * H * m * 128 + 8,), dtype=torch.bfloat16, device="cuda")
    k_ok = buf.data_ptr()
    with pytest.raises(binding.EvictError, match="16-byte aligned"):
        binding.evict_update_and_fetch(cache.handle, k_ok + 2, k_ok, None, m)
    assert binding.evict_stats(cache.handle)["offset"] == 0


def test_single_token_steps_stay_finite():
    # a proxy query that attends almost only to itself leaves G nearly rank-deficient (the
    # other rows' weights ~1e-4); the eigensolver must skip the noise-level reflections
    # instead of overflowing beta^2 into NaN leverage
    B, H = 2, 2
    keys = synth.clustered_keys(41, B, H, 60, spread=0.8)
    vals = synth.planted_spectrum_values(42, B, H, 60, rank=4)
    gpu = _gpu_cache(B, H, 24, max_block=1)
    for t in range(60):
        view = gpu.update_and_fetch(to_dev(keys[:, :, t:t + 1], torch), to_dev(vals[:, :, t:t + 1], torch))
        attn, lev = _gpu_scores(gpu, B, H)
        assert np.all(np.isfinite(lev)) and np.all(np.isfinite(attn)), t
        # the newest row dominates W, so its own leverage is close to 1 and the sum stays <= 1
        assert np.all(lev.sum(axis=-1) <= 1 + 1e-4)
    assert np.all(np.isfinite(to_bits(view[3])))


def test_planted_spectrum_full_size_sampled_units():
    # the curdkv_planted shape (8 x 8 heads, 16384 kept rows + a 512-token block, budget 2048) with
    # values of a planted spectrum, so the rank-16 gap is wide and leverage is asserted at 1e-3:
    # the tensor-core Gram and leverage passes at 16896 rows per unit
    B, H, S0, m, budget = 8, 8, 16384, 512, 2048
    n = S0 + m
    k_all = synth.clustered_keys(900, B, H, n, spread=0.5)
    v_all = synth.planted_spectrum_values(901, B, H, n)
    cum_old = synth.rng(902).uniform(0, 0.01, (B, H, S0))
    *_, gaps = _run_block(B, H, budget, k_all[:, :, :S0], v_all[:, :, :S0], cum_old, k_all[:, :, S0:],
                          v_all[:, :, S0:], units={(0, 0), (3, 6), (7, 2)})
    assert min(gaps) >= 1e-2


def test_long_context_full_size_sampled_units_curdkv():
    """The long-context stream at full size (4 x 8 heads, 16 blocks of 8192 tokens, budget 4096,
    rank 16; the proxy queries are each block's keys). The GPU cache runs the whole stream; three
    sampled (b, h) units start every block from the oracle's own state, loaded with
    evict_set_state, and are compared block by block: attention sums, captured energy, leverage
    and kept sets at the tolerances above, compacted K / V / positions bit for bit. Every unit is
    checked for budget, temporal order, sinks and for K / V being the input rows at its kept
    positions."""
    from kv_cache_token_bf16_gb300 import binding
    B, H, blocks, m, budget, n_sink = 4, 8, 16, 8192, 4096, 4
    gpu = _gpu_cache(B, H, budget, max_block=m, n_sink=n_sink)
    units = [(0, 0), (1, 5), (3, 7)]
    state = {}                          # unit -> the oracle's (K, V, positions, cumulative scores)
    all_k = np.empty((B, H, blocks * m, 128), np.uint16)     # every input row, by position
    all_v = np.empty_like(all_k)
    gaps = []
    for blk in range(blocks):
        k, v = synth.long_context_block(blk, B, H)
        all_k[:, :, blk * m:(blk + 1) * m] = k
        all_v[:, :, blk * m:(blk + 1) * m] = v
        if blk:
            gk, gv, gp, gs = [to_bits(t).copy() for t in gpu.view()]
            for (b, h), (ok, ov, opos, ocum) in state.items():
                gk[b, h], gv[b, h], gp[b, h], gs[b, h] = ok, ov, opos, ocum.astype(np.float32)
            gpu.set_state(to_dev(gk, torch), to_dev(gv, torch), torch.from_numpy(gp).cuda(),
                          torch.from_numpy(gs).cuda(), blk * m)
        view = gpu.update_and_fetch(to_dev(k, torch), to_dev(v, torch))
        gpu.sync()
        attn, lev = _gpu_scores(gpu, B, H)
        gk, gv, gp, gs = [to_bits(t) for t in view]
        kept_rows = min(budget, (blk + 1) * m)
        assert gp.shape == (B, H, kept_rows)
        assert np.all(np.diff(gp, axis=2) > 0) and np.all(gp[:, :, :n_sink] == np.arange(n_sink))
        for b in range(B):
            for h in range(H):
                assert np.array_equal(gk[b, h], all_k[b, h, gp[b, h]]), (blk, b, h)
                assert np.array_equal(gv[b, h], all_v[b, h, gp[b, h]]), (blk, b, h)
        for (b, h) in units:
            if blk:
                ok, ov, opos, ocum = state[(b, h)]
            else:
                ok, ov = k[b, h, :0], v[b, h, :0]
                opos, ocum = np.zeros(0, np.int32), np.zeros(0)
            k_u = np.concatenate([ok, k[b, h]])
            v_u = np.concatenate([ov, v[b, h]])
            pos_u = np.concatenate([opos, blk * m + np.arange(m, dtype=np.int32)])
            idx_g = np.searchsorted(pos_u, gp[b, h])
            assert np.array_equal(pos_u[idx_g], gp[b, h])
            gap, cum_or, kept_or = _check_unit(k_u, v_u, m, attn[b, h, :len(pos_u)], lev[b, h, :len(pos_u)],
                                               ocum.astype(np.float32).astype(np.float64), None, idx_g, n_sink, 0,
                                               budget, f"block {blk} unit {(b, h)}")
            gaps.append(gap)
            state[(b, h)] = (k_u[kept_or], v_u[kept_or], pos_u[kept_or], cum_or[kept_or])
    print(f"long-context CurDKV: rank-16 gaps {min(gaps):.3g} .. {max(gaps):.3g}")
    assert gpu.stats()["offset"] == blocks * m
