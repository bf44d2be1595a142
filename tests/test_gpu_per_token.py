"""GPU per-token mode for CurDKV and H2O ("CurDKV-adapted — Value-Aware
Leverage-Score Eviction", §How it works: steps 1-5 for every incoming token;
step 5 evicts the lowest-cumulative non-sink token, the first of equals).

* One m-token call equals m single-token calls bit for bit (the mode is a
  loop of m = 1 steps on the device).
* Zero values make every CurDKV leverage exactly 0: the argmin rule then
  evicts the oldest non-sink token at every step, an exact pattern.
* Against the oracle, step by step from the GPU's own kept state: every
  eviction decision with a clear margin (the two lowest unprotected
  cumulative scores further apart than their tolerances) must agree, and
  a good share of the decisions must be clear.
"""
import numpy as np
import pytest

from kv_cache_token_bf16_gb300 import synth
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


def _cache(method, B, H, budget, n_sink=2, max_block=64):
    from kv_cache_token_bf16_gb300 import binding
    return binding.EvictCache(method, B, H, budget=budget, n_sink=n_sink, max_block=max_block, rank_cap=4,
                              per_token=True)


@pytest.mark.parametrize("method", ["curdkv", "h2o"])
def test_one_call_equals_single_token_calls(method):
    B, H, budget = 2, 2, 24
    keys = synth.clustered_keys(41, B, H, 90, spread=0.8)
    vals = synth.planted_spectrum_values(42, B, H, 90, rank=4)
    a, b = _cache(method, B, H, budget), _cache(method, B, H, budget)
    pos = torch.arange(1000, 1090, dtype=torch.int32, device="cuda").expand(B, 90).contiguous()
    a.update_and_fetch(to_dev(keys[:, :, :30], torch), to_dev(vals[:, :, :30], torch))
    va = a.update_and_fetch(to_dev(keys[:, :, 30:], torch), to_dev(vals[:, :, 30:], torch), pos[:, 30:].contiguous())
    b.update_and_fetch(to_dev(keys[:, :, :30], torch), to_dev(vals[:, :, :30], torch))
    for t in range(30, 90):
        vb = b.update_and_fetch(to_dev(keys[:, :, t:t + 1], torch), to_dev(vals[:, :, t:t + 1], torch),
                                pos[:, t:t + 1].contiguous())
    a.sync()
    b.sync()
    for x, y in zip(va, vb):
        assert np.array_equal(to_bits(x), to_bits(y))
    p = to_bits(va[2])
    assert np.all((p < 30) | ((p >= 1030) & (p < 1090)))     # the block's tokens carry the given positions
    assert a.stats()["offset"] == 90


def test_zero_values_evict_the_oldest_non_sink():
    B, H, budget, sinks, S = 1, 2, 10, 3, 40
    keys = synth.gaussian_block(43, B, H, S)[0]
    vals = np.zeros_like(keys)
    c = _cache("curdkv", B, H, budget, n_sink=sinks)
    view = c.update_and_fetch(to_dev(keys, torch), to_dev(vals, torch))
    c.sync()
    want = list(range(sinks)) + list(range(S - (budget - sinks), S))
    for h in range(H):
        assert to_bits(view[2])[0, h].tolist() == want
        assert not np.any(to_bits(view[3])[0, h])


@pytest.mark.parametrize("method", ["curdkv", "h2o"])
def test_per_token_steps_match_the_oracle_where_decisions_are_clear(method):
    # every step restarts the oracle from the GPU's kept state (its stored scores included), so
    # the tolerance covers only the step's own increment
    B, H, budget, S = 2, 4, 16, 56
    if method == "curdkv":
        # planted two-class geometry: near-uniform attention, leverage set by the values
        p = synth.curdkv_planted(batch=B, n_kv_heads=H, existing=0, incoming=S, seed=46)
        keys, vals = p["k"], p["v"]
    else:
        keys = synth.clustered_keys(44, B, H, S, spread=0.8)
        vals = synth.planted_spectrum_values(45, B, H, S, rank=4)
    gpu = _cache(method, B, H, budget)
    view = gpu.update_and_fetch(to_dev(keys[:, :, :budget], torch), to_dev(vals[:, :, :budget], torch))
    clear_steps = agree = 0
    for t in range(budget, S):
        gpu.sync()
        kp, vp, pp, sp = [to_bits(x).copy() for x in view]
        view = gpu.update_and_fetch(to_dev(keys[:, :, t:t + 1], torch), to_dev(vals[:, :, t:t + 1], torch))
        gpu.sync()
        gp = to_bits(view[2])
        ref = OracleCache(method, B, H, budget=budget, n_sink=2, rank_cap=4, per_token=True)
        ref.set_state(kp, vp, pp, sp.astype(np.float64), t)
        ref.update_and_fetch(keys[:, :, t:t + 1], vals[:, :, t:t + 1])
        inc = ref.last_leverage if method == "curdkv" else ref.last_mass
        for b in range(B):
            for h in range(H):
                cum = ref.last_scores[b, h]
                # the increment's error (leverage: 1e-3 relative + 1e-9 of its unit sum; attention
                # mass: 1e-4 relative + 1e-7) plus the fp32 rounding of the stored score
                if method == "curdkv":
                    tol = 1e-3 * inc[b, h] + 1e-9 + 2e-7 * np.abs(cum)
                else:
                    tol = 1e-4 * inc[b, h] + 1e-7 + 2e-7 * np.abs(cum)
                unp = np.flatnonzero(~osel.protected_mask(len(cum), 2, 0))
                order = unp[np.argsort(cum[unp], kind="stable")]
                lo, nxt = order[0], order[1]
                if cum[nxt] - cum[lo] > tol[lo] + tol[nxt]:
                    clear_steps += 1
                    assert np.array_equal(gp[b, h], ref.pos[b, h]), (t, b, h)
                    agree += 1
    assert clear_steps >= 0.4 * (S - budget) * B * H, clear_steps
    assert gpu.stats()["offset"] == S
