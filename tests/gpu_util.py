"""Helpers for GPU parity tests: move seeded numpy inputs to the device and
bring library views back as raw bits."""
import numpy as np


def to_dev(x, torch):
    """numpy storage array (uint16 bf16 bits or float32) -> contiguous CUDA tensor."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(x).cuda()


def to_bits(t):
    """CUDA tensor -> numpy array with the same bits (bf16 -> uint16)."""
    import torch
    t = t.contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def assert_cache_equal(gpu_view, ref, what=""):
    """Kept K/V/pos/score bit-exact against an OracleCache."""
    gk, gv, gp, gs = gpu_view
    k, v, p, s = to_bits(gk), to_bits(gv), to_bits(gp), to_bits(gs)
    assert p.shape == ref.pos.shape, f"{what}: kept rows {p.shape} vs oracle {ref.pos.shape}"
    if not np.array_equal(p, ref.pos):
        bad = np.argwhere(p != ref.pos)
        raise AssertionError(f"{what}: positions differ at {len(bad)} places, first {bad[:5].tolist()}")
    assert np.array_equal(k, ref.k), f"{what}: kept keys differ"
    assert np.array_equal(v, ref.v), f"{what}: kept values differ"
    # scores bit for bit; a NaN score (a key with a NaN element) must be NaN on
    # both sides, its payload is the arithmetic's own (CUDA's square root
    # returns the canonical NaN, numpy passes the input payload through)
    ref_s = ref.score.astype(np.float32)
    nan_g, nan_r = np.isnan(s), np.isnan(ref_s)
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN scores at different rows"
    assert s[~nan_g].tobytes() == ref_s[~nan_r].tobytes(), f"{what}: stored scores differ"


# ---------------------------------------------------------------------------
# Key-SVD fallback: the GPU and the oracle each freeze their own filter (fp32
# power iteration against an fp64 SVD), so their projections differ by a
# bounded amount and kept sets are compared outside that band.
# ---------------------------------------------------------------------------
U32 = 2.0 ** -24


def projection_tolerance(k_rows, f_gpu, f_oracle):
    """Bound on |sigma_gpu - sigma_oracle| for the canonical fp32 projections
    of the same keys [n, D] on two unit filters: |k| * |f_gpu - f_oracle|
    (Cauchy-Schwarz) plus each side's fp32 rounding (12 roundings deep in the
    canonical order, bounded here by 16 u * sum |k_d f_d|)."""
    from oracle.bf16 import to_f64
    x = to_f64(k_rows)
    fg, fo = np.asarray(f_gpu, np.float64), np.asarray(f_oracle, np.float64)
    d = float(np.linalg.norm(fg - fo))
    return np.linalg.norm(x, axis=-1) * d + 2 * 16 * U32 * (np.abs(x) @ np.maximum(np.abs(fg), np.abs(fo)))


def kept_sets_agree_outside_band(score, idx_o, idx_g, tol, n_sink, recent, budget):
    """Keep-high selection over ``score`` [n] (the oracle's): do the oracle's kept
    indices ``idx_o`` and the GPU's ``idx_g`` agree on every row whose priority
    lies more than 2 * (tol_i + tol_cutoff) from the cutoff, with equal counts?"""
    from oracle import select as osel
    n = len(score)
    if len(idx_o) != len(idx_g):
        return False
    if n <= budget:
        return np.array_equal(np.sort(idx_o), np.sort(idx_g))
    prio = osel.priority(np.asarray(score, np.float64))
    prot = osel.protected_mask(n, n_sink, recent)
    unp = np.flatnonzero(~prot)
    q = budget - int(prot.sum())
    order = unp[np.argsort(-prio[unp], kind="stable")]
    cut = order[q - 1]
    clear = np.abs(prio - prio[cut]) > 2 * (tol + tol[cut])
    in_o = np.isin(np.arange(n), idx_o)
    in_g = np.isin(np.arange(n), idx_g)
    return bool(np.array_equal(in_o[clear], in_g[clear]))


def check_own_filter_update(view, ref, f_gpu, what):
    """Compare a GPU update with an oracle that froze its OWN key-SVD filter.

    ``view`` holds the GPU's kept K, V, positions and scores (tensors, or
    numpy arrays of their bits); ``f_gpu`` its frozen filters [B, H, D] or None.

    Before either side froze, the caches must be equal bit for bit. After:
    * the kept counts are equal and every row whose oracle priority lies more
      than twice the projection tolerance (its own plus the cutoff row's)
      from the cutoff is kept by both sides or by neither;
    * the GPU's kept K / V are the input rows at its kept positions, bit for
      bit, and its stored scores lie within the tolerance of the oracle's;
    * where the kept sets agree, positions equal the oracle's exactly.
    An in-band disagreement re-points the oracle's kept rows of that unit at
    the GPU's kept positions (the oracle's own rows and scores there) so later
    updates compare like with like. Returns the number of such resyncs."""
    from oracle import select as osel
    gk, gv, gp, gs = [t if isinstance(t, np.ndarray) else to_bits(t) for t in view]
    if ref.filters_bh is None:
        assert f_gpu is None, f"{what}: the GPU froze before the oracle"
        assert np.array_equal(gp, ref.pos) and np.array_equal(gk, ref.k) and np.array_equal(gv, ref.v), \
            f"{what}: pass-through rows differ"
        assert gs.tobytes() == ref.score.astype(np.float32).tobytes(), f"{what}: pass-through scores differ"
        return 0
    assert f_gpu is not None, f"{what}: the oracle froze before the GPU"
    k_all, v_all, pos_all = ref.last_rows
    sc_all = np.asarray(ref.last_scores, np.float64)
    B, H, n = pos_all.shape
    assert gp.shape == ref.pos.shape, f"{what}: kept rows {gp.shape} vs oracle {ref.pos.shape}"
    resyncs = 0
    for b in range(B):
        for h in range(H):
            tol = projection_tolerance(k_all[b, h], f_gpu[b, h], ref.filters_bh[b, h])
            idx_g = np.searchsorted(pos_all[b, h], gp[b, h])
            assert np.all(idx_g < n) and np.array_equal(pos_all[b, h, idx_g], gp[b, h]), \
                f"{what}: GPU kept a position that was not offered"
            assert np.all(np.diff(gp[b, h]) > 0), f"{what}: temporal order"
            assert np.array_equal(gk[b, h], k_all[b, h, idx_g]) and np.array_equal(gv[b, h], v_all[b, h, idx_g]), \
                f"{what}: kept K/V are not the input rows at the kept positions"
            assert np.all(np.abs(gs[b, h].astype(np.float64) - sc_all[b, h, idx_g]) <= tol[idx_g]), \
                f"{what}: stored scores of unit {(b, h)} outside the projection tolerance"
            idx_o = ref.last_kept[b, h]
            if np.array_equal(idx_g, idx_o):
                continue
            assert kept_sets_agree_outside_band(sc_all[b, h], idx_o, idx_g, tol, ref.n_sink, ref.recent,
                                                ref.budget), f"{what}: unit {(b, h)} kept sets differ outside the band"
            ref.k[b, h], ref.v[b, h] = k_all[b, h, idx_g], v_all[b, h, idx_g]
            ref.pos[b, h], ref.score[b, h] = pos_all[b, h, idx_g], sc_all[b, h, idx_g]
            ref.last_kept[b, h] = idx_g
            resyncs += 1
    return resyncs
