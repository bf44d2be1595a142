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
    ref_s = ref.score.astype(np.float32)
    assert s.tobytes() == ref_s.tobytes(), f"{what}: stored scores differ"
