"""The C-ABI library loads, exports every declared symbol and validates
configurations on the host (no GPU needed: validation runs before any CUDA
call)."""
import ctypes
import os
import re

import pytest

from kv_cache_token_bf16_gb300 import binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "evict.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(evict_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for required in ("evict_init", "evict_update_and_fetch", "evict_stats", "evict_qfilters_calibrate",
                     "evict_set_state", "evict_sync", "evict_destroy", "evict_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def _cfg(**kw):
    base = dict(method=binding.EVICT_KNORM, dtype=binding.EVICT_BF16, batch=1, n_kv_heads=1, head_dim=128,
                budget=64, n_sink=4, recent=0, max_block=128, max_kept=0, keep_low=1, sign=1, filters=None,
                n_filter_heads=0, rank_cap=0, stream=None)
    base.update(kw)
    return binding.EvictConfig(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(n_sink=4, recent=60), binding.EVICT_EINVAL),            # n_sink + recent >= budget
    (dict(n_sink=64), binding.EVICT_EINVAL),
    (dict(head_dim=64), binding.EVICT_EINVAL),
    (dict(budget=0), binding.EVICT_EINVAL),
    (dict(batch=0), binding.EVICT_EINVAL),
    (dict(max_block=0), binding.EVICT_EINVAL),
    (dict(method=7), binding.EVICT_EINVAL),
    (dict(dtype=3), binding.EVICT_EINVAL),
    (dict(keep_low=2), binding.EVICT_EINVAL),
    (dict(method=binding.EVICT_QFILTERS, sign=0, filters=8), binding.EVICT_EINVAL),   # invalid sign
    # no filters: the key-SVD fallback, which needs calib_tokens >= 0 and keeps calib_tokens - 1 rows
    (dict(method=binding.EVICT_QFILTERS, sign=1, filters=None, calib_tokens=-1), binding.EVICT_EINVAL),
    (dict(method=binding.EVICT_QFILTERS, sign=1, filters=None, calib_tokens=49100), binding.EVICT_ELIMIT),
    (dict(method=binding.EVICT_QFILTERS, n_kv_heads=8, filters=8, n_filter_heads=4), binding.EVICT_EINVAL),
    (dict(method=binding.EVICT_CURDKV, dtype=binding.EVICT_FP32), binding.EVICT_EINVAL),
    (dict(method=binding.EVICT_H2O, dtype=binding.EVICT_FP32), binding.EVICT_EINVAL),
    (dict(method=binding.EVICT_KNORM, per_token=1), binding.EVICT_EINVAL),          # per-token: CurDKV/H2O only
    (dict(method=binding.EVICT_CURDKV, per_token=2), binding.EVICT_EINVAL),
    (dict(method=binding.EVICT_CURDKV, rank_cap=500), binding.EVICT_ELIMIT),
    (dict(budget=40000, max_block=20000), binding.EVICT_ELIMIT),  # raised, never truncated
])
def test_invalid_configurations_are_rejected_before_any_cuda_call(lib, kw, code):
    h = ctypes.c_void_p()
    rc = lib.evict_init(ctypes.byref(_cfg(**kw)), ctypes.byref(h))
    assert rc == code
    assert h.value is None
    assert lib.evict_last_error().decode()


def test_null_arguments_are_rejected(lib):
    assert lib.evict_init(None, None) == binding.EVICT_EINVAL
    view = binding.EvictView()
    assert lib.evict_update_and_fetch(None, None, None, None, 1, ctypes.byref(view)) == binding.EVICT_EINVAL
    assert lib.evict_stats(None, None) == binding.EVICT_EINVAL
    assert lib.evict_sync(None) == binding.EVICT_EINVAL
    lib.evict_destroy(None)


def test_no_alloc_refuses_misaligned_pointers_without_a_gpu(lib):
    # the alignment check runs before any CUDA call, so fake addresses are safe here
    cfg = _cfg(budget=64, max_block=0)
    base = 0x10000
    for k, v, ko, vo, po, so, what in ((base + 2, base, base, base, base, base, "16-byte aligned"),
                                       (base, base, base, base + 8, base, base, "16-byte aligned"),
                                       (base, base, base, base, base + 2, base, "4-byte aligned"),
                                       (base, base, base, base, base, base + 1, "4-byte aligned")):
        with pytest.raises(binding.EvictError, match=what) as e:
            binding.evict_prefill_noalloc(cfg, k, v, None, 100, ko, vo, po, so)
        assert e.value.code == binding.EVICT_EINVAL
