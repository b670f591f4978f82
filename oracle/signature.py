"""Oracle for MSCRED signature matrices: a plain fp64 CPU loop.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle/``): only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may use
it; the CUDA library never does, and they share no code.

"GPU-Accelerating MSCRED with CUDA, im2col, GEMM, and a Custom PyTorch
Extension" (section "Why Signature Matrices Are Useful") describes a
signature matrix as the pairwise relationships between the signals over one
time interval, generated at several interval lengths; the definition used
(the one of the MSCRED paper that page cites) is, for signals s_i(t), an end
time e and a window length w,

    M_ij(e, w) = sum_{t = e-w}^{e-1} s_i(t) * s_j(t) / w

(the inner products of the last w samples, scaled by 1/w).  The matrices of
n_steps consecutive end times e = t_first .. t_first + n_steps - 1 for every
window form an [n_steps, n_windows, n, n] tensor: the NCHW input of the
encoder's first convolution, one channel per window.
"""
from __future__ import annotations

import numpy as np


def signature_matrices(series, windows, t_first: int, n_steps: int):
    """Return (M, den), both fp64 [n_steps, len(windows), n, n].

    ``series`` is [n_signals, T] (any float dtype, widened exactly to fp64).
    den[b, c, i, j] = sum over the same samples of |s_i(t)| * |s_j(t)| / w,
    the scale the GPU result's error is measured against.
    """
    s = np.asarray(series, dtype=np.float64)
    if s.ndim != 2:
        raise ValueError("series must be [n_signals, T]")
    n, T = s.shape
    windows = [int(w) for w in windows]
    if n_steps < 1 or not windows or min(windows) < 1:
        raise ValueError("need n_steps >= 1 and windows >= 1")
    if t_first - max(windows) < 0 or t_first + n_steps - 1 > T:
        raise ValueError("every window must lie inside the series")
    M = np.zeros((n_steps, len(windows), n, n))
    den = np.zeros_like(M)
    for b in range(n_steps):
        e = t_first + b
        for c, w in enumerate(windows):
            acc = np.zeros((n, n))
            aacc = np.zeros((n, n))
            for t in range(e - w, e):
                col = s[:, t]
                acc += np.outer(col, col)
                aacc += np.outer(np.abs(col), np.abs(col))
            M[b, c] = acc / w
            den[b, c] = aacc / w
    return M, den


def error_ratio(got, ref, den) -> float:
    """max |got - ref| / den over all entries; entries with den == 0 must be exact 0."""
    g = np.asarray(got, dtype=np.float64)
    if g.shape != ref.shape:
        raise ValueError(f"shape {g.shape} != {ref.shape}")
    if not np.all(np.isfinite(g)):
        return float("inf")
    diff = np.abs(g - ref)
    zero = den == 0
    if np.any(diff[zero] != 0):
        return float("inf")
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(zero, 0.0, diff / np.where(zero, 1.0, den))
    return float(r.max()) if r.size else 0.0
