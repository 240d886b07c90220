"""Oracle Gram accumulation (f64): H += X^T X, H stored as the upper
triangle by rows.

Follows the calibration step of ``cortiq-cli src/gptq.rs`` (the device
Hessian accumulators: ``gram_alloc`` / ``gram_add_dev`` per linear input, one
call per window of tokens) and the packed layout of the fold page
(``cortiq-engine src/gpu_wgpu/gptq_dev.rs``, ``poff``: row r starts at
r (2n - r + 1) / 2).  The pages sum over tokens (counts kept apart), so
there is no normalization here.

Test infrastructure: see the package docstring.
"""
from __future__ import annotations

import numpy as np


def pack_upper(h):
    """Upper triangle of a square matrix by rows (the fold page's layout)."""
    h = np.asarray(h)
    n = h.shape[0]
    return np.concatenate([h[r, r:] for r in range(n)])


def gram_add(hp, x):
    """Return hp + packed(X^T X) in f64; X is [T, n] (tokens x channels)."""
    x = np.asarray(x, dtype=np.float64)
    g = x.T @ x
    return np.asarray(hp, dtype=np.float64) + pack_upper(g)
