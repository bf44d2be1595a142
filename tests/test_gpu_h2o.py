"""GPU parity of the H2O-adapted scorer (cumulative proxy-attention mass).

The mass comes from the same tensor-core softmax passes as CurDKV's proxy
attention (fp32 logits from bf16 keys, fp32 sums of ex2 terms), so it is
compared with the oracle's fp64 mass to a relative 1e-4 (+ 1e-7 m absolute);
a new row's own weight is left out exactly, so the last row of a block has
mass exactly 0 on both sides. Kept sets are compared band-tolerantly: equal
counts, and every row whose oracle score lies more than twice the tolerance
from the cutoff is kept by both or neither; compacted K/V/positions are the
original rows of the kept positions. Each block starts from the oracle's own
state (evict_set_state), so no GPU output feeds the oracle.
"""
import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import synth
from oracle import h2o as oh2o
from oracle import select as osel
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


def _gpu_mass(cache, B, H):
    from kv_cache_token_bf16_gb300 import binding
    n = binding.evict_curdkv_scores(cache.handle, None, None)
    attn = torch.empty((B, H, n), dtype=torch.float32, device="cuda")
    inc = torch.empty_like(attn)
    binding.evict_curdkv_scores(cache.handle, attn.data_ptr(), inc.data_ptr())
    cache.sync()
    return attn.cpu().numpy().astype(np.float64), inc.cpu().numpy().astype(np.float64)


def _run_block(B, H, budget, k_old, v_old, cum_old, k_new, v_new, n_sink=4, recent=0, units=None):
    """One GPU update from the oracle-provided state; checks every (or the listed) unit. Returns the GPU
    kept positions."""
    from kv_cache_token_bf16_gb300 import binding
    k0, m = k_old.shape[2], k_new.shape[2]
    gpu = binding.EvictCache("h2o", B, H, budget=budget, n_sink=n_sink, recent=recent, max_block=m,
                             max_kept=max(k0, budget))
    if k0:
        pos0 = np.broadcast_to(np.arange(k0, dtype=np.int32), (B, H, k0)).copy()
        gpu.set_state(to_dev(k_old, torch), to_dev(v_old, torch), torch.from_numpy(pos0).cuda(),
                      torch.from_numpy(cum_old.astype(np.float32)).cuda(), k0)
    view = gpu.update_and_fetch(to_dev(k_new, torch), to_dev(v_new, torch))
    gpu.sync()
    mass_g, inc_g = _gpu_mass(gpu, B, H)
    assert np.array_equal(mass_g, inc_g)
    gk, gv, gp, gs = [to_bits(t) for t in view]
    k_all = np.concatenate([k_old, k_new], axis=2)
    v_all = np.concatenate([v_old, v_new], axis=2)
    n = k0 + m
    for b in range(B):
        for h in range(H):
            if units is not None and (b, h) not in units:
                continue
            what = f"unit {(b, h)}"
            mass = oh2o.proxy_mass(k_all[b, h], m)
            assert np.allclose(mass_g[b, h], mass, rtol=1e-4, atol=1e-7 * m), f"{what}: mass"
            assert mass_g[b, h, -1] == 0.0, f"{what}: the newest row must start from exactly 0"
            kept = gp[b, h]
            assert np.all(np.diff(kept) > 0)
            assert np.array_equal(gk[b, h], k_all[b, h, kept]) and np.array_equal(gv[b, h], v_all[b, h, kept])
            cum_or = oh2o.cumulative(cum_old[b, h].astype(np.float32).astype(np.float64), mass)
            tol = 1e-4 * mass + 1e-7 * m + 2e-7 * np.abs(cum_or)
            if n > budget:
                assert len(kept) == budget
                kept_or = osel.kept_indices(osel.priority(cum_or)[None, None], n_sink, recent, budget)[0, 0]
                prot = osel.protected_mask(n, n_sink, recent)
                unp = np.flatnonzero(~prot)
                cutoff = np.sort(cum_or[unp])[::-1][budget - prot.sum() - 1]
                clear = np.abs(cum_or - cutoff) > 2 * tol
                in_or, in_g = np.isin(np.arange(n), kept_or), np.isin(np.arange(n), kept)
                assert np.array_equal(in_or[clear], in_g[clear]), f"{what}: kept set differs outside the band"
                # stored scores are the cumulative scores of the kept rows
                assert np.allclose(gs[b, h], cum_or[kept], rtol=0, atol=2 * tol[kept].max())
            else:
                assert np.array_equal(kept, np.arange(n))
    return gp


@pytest.mark.parametrize("k0,m,budget", [(0, 300, 64), (0, 129, 200), (500, 257, 128), (1000, 1, 64),
                                         (127, 128, 100), (0, 513, 100), (300, 1100, 256), (129, 640, 700),
                                         # short blocks: the fused one-CTA-per-unit attention (m <= 8 and
                                         # m * n <= 16384), its boundary, and the tensor-core path just past it
                                         (0, 1, 64), (600, 5, 128), (2040, 8, 512), (2041, 8, 512), (3, 8, 6),
                                         (700, 9, 128)])
def test_h2o_blocks(k0, m, budget):
    B, H = 1, 2
    n = k0 + m
    k_all = synth.clustered_keys(300 + n, B, H, n, spread=0.5)
    v_all = synth.gaussian_block(400 + n, B, H, n)[1]
    cum_old = synth.rng(5).uniform(0, 2.0, (B, H, k0))
    _run_block(B, H, budget, k_all[:, :, :k0], v_all[:, :, :k0], cum_old, k_all[:, :, k0:], v_all[:, :, k0:])


def test_h2o_stream_of_blocks_and_decode_steps():
    # appends, then evictions, then single-token steps; each call resynced to the oracle's state
    B, H, budget = 2, 2, 96
    k_all, v_all = synth.gaussian_block(31, B, H, 400)
    ref = OracleCache("h2o", B, H, budget=budget, n_sink=4)
    cuts = [0, 40, 80, 200, 330] + list(range(331, 345))
    for a, b in zip(cuts[:-1], cuts[1:]):
        kp = ref.pos                                   # the oracle's kept rows before the call
        k_old = np.stack([[k_all[x, y, kp[x, y]] for y in range(H)] for x in range(B)]) if ref.n_kept else \
            k_all[:, :, :0]
        v_old = np.stack([[v_all[x, y, kp[x, y]] for y in range(H)] for x in range(B)]) if ref.n_kept else \
            v_all[:, :, :0]
        _run_block(B, H, budget, k_old, v_old, ref.score, k_all[:, :, a:b], v_all[:, :, a:b])
        ref.update_and_fetch(k_all[:, :, a:b], v_all[:, :, a:b])


def test_h2o_planted_geometry_keeps_both_classes():
    # the pages' blind spot: identical-key classes with divergent values are not told apart
    rates = []
    for seed in range(4):
        p = synth.curdkv_planted(batch=1, n_kv_heads=2, existing=1024, incoming=64, seed=2000 + seed)
        kept = _run_block(1, 2, 128, p["k"][:, :, :1024], p["v"][:, :, :1024], np.zeros((1, 2, 1024)),
                          p["k"][:, :, 1024:], p["v"][:, :, 1024:])
        for h in range(2):
            rates.append(np.mean(p["cls"][0, h, kept[0, h, 4:]] == 2))
    assert 0.2 < np.mean(rates) < 0.8


def test_h2o_planted_full_size_sampled_units():
    # the planted workload at full size: 8 x 8 heads, 16384 kept rows + a 512-token block, budget 2048
    B, H, S0, m = 8, 8, 16384, 512
    p = synth.curdkv_planted(B, H, existing=S0, incoming=m)
    kept = _run_block(B, H, 2048, p["k"][:, :, :S0], p["v"][:, :, :S0], np.zeros((B, H, S0)), p["k"][:, :, S0:],
                      p["v"][:, :, S0:], units={(0, 0), (5, 3), (7, 7)})
    assert kept.shape == (B, H, 2048) and np.all(np.diff(kept, axis=2) > 0)
