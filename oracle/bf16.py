"""bf16 storage format for the oracle (test infrastructure only).

bf16 is the upper half of an IEEE binary32: widening is a 16-bit shift and
is exact. Caches store keys and values in their input format, and the pages
require kept keys to be copied bit-identically ("Q-Filters — Query-Agnostic
Projection Eviction", §Adaptation notes, on the apply kernel copying keys
bit-identically), so the oracle carries raw bit patterns and widens only to
compute scores.
"""
import numpy as np


def to_f32(x: np.ndarray) -> np.ndarray:
    """Widen a storage array to float32: uint16 = bf16 bits, float32 as is."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32)
    if x.dtype == np.float32:
        return x
    raise TypeError(f"unsupported storage dtype {x.dtype}")


def to_f64(x: np.ndarray) -> np.ndarray:
    """Widen to float64 (float64 input is returned as is)."""
    x = np.asarray(x)
    if x.dtype == np.float64:
        return x
    return to_f32(x).astype(np.float64)


def element_bytes(x: np.ndarray) -> int:
    return np.asarray(x).dtype.itemsize
