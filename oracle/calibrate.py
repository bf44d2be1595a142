"""One-time Q-Filters calibration from query activations.

Test infrastructure only.

Source: "Q-Filters — Query-Agnostic Projection Eviction",
§Calibrated — the paper's actual mechanism: take the SVD of each head's
query activations Q^h [N, D] without mean-centering, keep the top right
singular vector v1 and fix its sign as sgn(1^T u1) * v1; under GQA, average
the filters of each query-head group onto its KV head. §Evidence: GQA
averaging keeps the filters unit-norm.

Key-SVD fallback ("Q-Filters", §Calibrated vs key-SVD fallback and §Key-SVD
fallback): with no calibrated filter, the filter is the top right singular
vector of the MEAN-CENTRED keys observed so far, frozen once estimated. The
pages say the sign is ambiguous; reading: the component of largest magnitude
is made positive (the lowest index on ties), and the configured sign is
applied on top.

Readings:
* sgn(0) is taken as +1.
* Query head h belongs to KV head h // G with G = H_q / H_kv (contiguous
  groups, the usual repeat-kv order).
* The group average is renormalised to unit length; an average shorter than
  1e-6 is degenerate and raises.
"""
import numpy as np

from .bf16 import to_f64

DEGENERATE_NORM = 1e-6


def compute_qfilter(q: np.ndarray) -> np.ndarray:
    """Sign-fixed top right singular vector of one head's queries [N, D] (fp64)."""
    x = to_f64(q)
    u, _, vt = np.linalg.svd(x, full_matrices=False)
    sign = 1.0 if np.sum(u[:, 0]) >= 0 else -1.0
    return sign * vt[0]


def average_gqa(filters: np.ndarray, n_kv_heads: int) -> np.ndarray:
    """Average [H_q, D] filters over contiguous groups onto [H_kv, D], unit norm."""
    h_q, d = filters.shape
    if h_q % n_kv_heads:
        raise ValueError("query heads must be a multiple of KV heads")
    g = h_q // n_kv_heads
    avg = filters.reshape(n_kv_heads, g, d).mean(axis=1)
    norms = np.linalg.norm(avg, axis=1)
    if np.any(norms < DEGENERATE_NORM):
        raise ValueError("degenerate GQA filter average")
    return avg / norms[:, None]


def calibrate(queries: np.ndarray, n_kv_heads: int) -> np.ndarray:
    """Queries [H_q, N, D] (bf16 bits or fp32) -> filters [H_kv, D] fp64."""
    per_head = np.stack([compute_qfilter(queries[h]) for h in range(queries.shape[0])])
    return average_gqa(per_head, n_kv_heads)


def centered_top_direction(q: np.ndarray) -> np.ndarray:
    """The mean-centred estimator the page warns against (for the contrast pin)."""
    x = to_f64(q)
    x = x - x.mean(axis=0, keepdims=True)
    _, _, vt = np.linalg.svd(x, full_matrices=False)
    return vt[0]


def key_svd_filter(keys: np.ndarray) -> np.ndarray:
    """Key-SVD fallback filter of one (b, h): keys [n, D] -> unit direction (fp64).

    Top right singular vector of the mean-centred keys; the largest-magnitude
    component is made positive (the first one on ties). Two cases the page
    leaves open: keys that are all equal have no direction, and the filter is
    then the first coordinate axis e_0; a non-finite key has no SVD, and the
    freeze raises ValueError.
    """
    x = to_f64(keys)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite key at the key-SVD freeze")
    x = x - x.mean(axis=0, keepdims=True)
    if not np.any(x):
        e0 = np.zeros(x.shape[1])
        e0[0] = 1.0
        return e0
    _, _, vt = np.linalg.svd(x, full_matrices=False)
    v = vt[0]
    j = int(np.argmax(np.abs(v)))
    return v if v[j] >= 0 else -v
