"""Oracle fold operator (f64), following ``cortiq-cli src/gptq.rs``,
``gptq_fold_operator_par`` (the host route: Cholesky, inverse, second
Cholesky), plus a plain restatement of the device builder ``build_a``
(``cortiq-engine src/gpu_wgpu/gptq_dev.rs``) used only to check that step.

Test infrastructure: see the package docstring.
"""
from __future__ import annotations

import numpy as np
import scipy.linalg
import scipy.linalg.lapack


class NotSPD(Exception):
    """Damping beyond 10 x mean(diag) still left a non-positive pivot."""


def unpack_upper(hp, n: int) -> np.ndarray:
    """Dense symmetric f64 matrix from the upper triangle stored by rows.

    Layout of the fold page (``poff``): row r starts at ``r (2n - r + 1)/2``;
    element (a <= b) sits at ``poff(a) + (b - a)``.
    """
    hp = np.asarray(hp, dtype=np.float32)
    assert hp.shape == (n * (n + 1) // 2,)
    h = np.empty((n, n), dtype=np.float64)
    off = 0
    for r in range(n):
        row = hp[off : off + n - r]
        h[r, r:] = row
        h[r:, r] = row
        off += n - r
    return h


def _diag_from_packed(hp, n: int) -> np.ndarray:
    r = np.arange(n, dtype=np.int64)
    return np.asarray(hp, dtype=np.float32)[r * (2 * n - r + 1) // 2]


def _chol_ok(a: np.ndarray):
    """Lower Cholesky factor, or None when a pivot is not positive or not
    finite (the host's ``!(s > 0) || !s.is_finite()`` test)."""
    try:
        lo = np.linalg.cholesky(a)
    except np.linalg.LinAlgError:
        return None
    if not np.all(np.isfinite(lo)):
        return None
    return lo


def fold_damping(hp, n: int):
    """(dead mask, fixed-up f64 H, base) -- the host's pre-damping steps.

    dead_i <=> !(H_ii > 0) on the stored f32 value (NaN counts as dead);
    a dead channel's row and column become 0 and its diagonal 1; then
    ``base = max(mean(diag), 1e-12)``.
    """
    h = unpack_upper(hp, n)
    hd32 = _diag_from_packed(hp, n)
    dead = ~(hd32 > 0)
    h[dead, :] = 0.0
    h[:, dead] = 0.0
    h[dead, dead] = 1.0
    mean = float(np.trace(h)) / max(n, 1)
    base = max(mean, 1e-12)
    return dead, h, base


def fold(hp, n: int, lam: float = 0.01):
    """The fold operator of one Hessian group.

    Returns ``(U, D, dead, lam_used)``:

    * ``U`` -- f64 n x n, upper, positive diagonal, ``U^T U = H_d^-1`` (cast
      it to f32 for the page's f32 operator);
    * ``D`` -- f64 n, ``sqrt(H_ii + damp)`` for live channels and
      ``-sqrt(1 + damp)`` for dead ones (the device page's signed scale);
    * ``dead`` -- bool n; ``lam_used`` -- the damping factor that factored.

    Raises ``NotSPD`` once lambda passes 10 (the device page's ``None``; the
    host page silently returns U = I there instead).
    """
    dead, h, base = fold_damping(hp, n)
    lam = max(float(lam), 0.0)
    diag = np.arange(n)
    hdiag0 = h[diag, diag].copy()
    while True:
        if not np.isfinite(lam * base):
            raise NotSPD(f"non-finite damping (base={base})")
        h[diag, diag] = hdiag0 + lam * base
        lo = _chol_ok(h)
        if lo is not None:
            break
        lam = 1e-4 if lam == 0.0 else lam * 10.0
        if lam > 10.0:
            raise NotSPD("no damping up to 10 x mean(diag) makes H positive definite")
    del h
    damp = lam * base
    # L^-1 and H_d^-1 = L^-T L^-1 (LAPACK potri: triangular inverse, then
    # the product), M = chol(H_d^-1), U = M^T.
    hinv, info = scipy.linalg.lapack.dpotri(lo, lower=1)
    if info != 0:
        raise NotSPD(f"potri failed (info={info})")
    del lo
    hinv = np.tril(hinv) + np.tril(hinv, -1).T
    m = _chol_ok(hinv)
    del hinv
    if m is None:
        raise NotSPD("H_d^-1 did not factor")
    u = np.ascontiguousarray(m.T)
    hd32 = _diag_from_packed(hp, n).astype(np.float64)
    d = np.where(dead, -np.sqrt(1.0 + damp), np.sqrt(np.where(dead, 0.0, hd32) + damp))
    return u, d, dead, lam


def equilibrated_reversed(hp, n: int, lam: float):
    """Lower triangle of ``A~ = P D^-1 H_d D^-1 P`` (f64), the device page's
    ``build_a`` matrix: ``A~[i][j] = (H[ii][jj] + delta*damp) / (d_ii d_jj)``
    with ``ii = n-1-i``; a dead channel contributes an identity row/column.
    Also returns the signed D and damp."""
    dead, h, base = fold_damping(hp, n)
    damp = max(float(lam), 0.0) * base
    hd32 = _diag_from_packed(hp, n).astype(np.float64)
    d = np.where(dead, -np.sqrt(1.0 + damp), np.sqrt(np.where(dead, 0.0, hd32) + damp))
    hraw = unpack_upper(hp, n)
    a = (hraw + damp * np.eye(n)) / np.outer(np.abs(d), np.abs(d))
    a[dead, :] = 0.0
    a[:, dead] = 0.0
    a[dead, dead] = 1.0
    a = a[::-1, ::-1]
    return np.tril(a), d, damp
