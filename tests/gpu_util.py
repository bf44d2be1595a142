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
