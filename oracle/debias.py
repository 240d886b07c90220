"""Oracle output debias of a quantized row ladder (f64).

Follows ``cortiq-cli src/gptq.rs``, ``q2tp_debias_hessian`` /
``q4tp_debias_hessian`` (``debias_tiled_hessian``) and their GEMM form
``q2tp_debias_gemm``: per row r the regression slope

    b_r = (W^ H W^T)_rr / (W H W^T)_rr = (w^_r . H w_r) / (w_r . H w_r)

of the quantized outputs on the original ones (W the original weights,
W^ the dequantized ones through the row's ladder, H the calibration
Hessian), removed through the row's f16 ``lo``; codes, rungs and the step
stay.  Here in f64 throughout (H from the packed f32 values).

Reading where the page is silent (the update itself, ``q2tp_unshrink_row``,
is called but not shown): every non-zero rung of a row is ``2^(lo + ...)``,
so dividing the row's outputs by b is the shift ``lo -> lo - log2 b``:
``lo' = f16(lo + log2(den / num))`` (in f64, then rounded to f16) when
num > 0 and den > 0, else lo is kept; the rungs are rebuilt from (lo', step)
(q2tp: rung 0 stays 0, rung c = 2^(lo' + (c-1) step); q4tp: rung c =
2^(lo' + c step)), a row whose rungs were all 0 keeps them, and each
(row, group) scale becomes the new rung value of its rung.

Test infrastructure: see the package docstring.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
GROUP = 32


def dequant(q, rungs, tab, two_bit):
    """W^ [rows, n] f64 from codes (q2tp: 0..3, level q - 1.5; q4tp: -8..7,
    level q) and each (row, group) rung of the row's ladder."""
    q = np.asarray(q, dtype=np.float64)
    rows, n = q.shape
    tab = np.asarray(tab, dtype=np.float64)
    s = tab[np.arange(rows)[:, None], np.asarray(rungs)]            # [rows, gpr]
    lev = q - 1.5 if two_bit else q
    return lev * np.repeat(s, GROUP, axis=1)


def slopes(w0, what, h):
    """(num, den) per row: num = w^ . H w, den = w . H w (f64)."""
    w = np.asarray(w0, dtype=np.float64)
    y = w @ np.asarray(h, dtype=np.float64)   # H symmetric: row r of W H is H w_r
    num = np.einsum("ij,ij->i", np.asarray(what, dtype=np.float64), y)
    den = np.einsum("ij,ij->i", w, y)
    return num, den


def unshrink(lost, tab, num, den, two_bit):
    """(tab', lost') after removing the slope b = num/den through lo."""
    lost = np.array(lost, dtype=F32, copy=True)
    tab = np.asarray(tab, dtype=F32)
    rows = lost.shape[0]
    out = np.array(tab, copy=True)
    for r in range(rows):
        if not (num[r] > 0 and den[r] > 0):
            continue
        lo, st = float(lost[r, 0]), float(lost[r, 1])
        lo2 = float(np.float16(lo + np.log2(den[r] / num[r])))
        lost[r, 0] = lo2
        if not np.any(tab[r] > 0):
            continue
        c = np.arange(32, dtype=np.float64)
        if two_bit:
            out[r, 0] = 0.0
            out[r, 1:] = np.exp2(lo2 + (c[1:] - 1.0) * st).astype(F32)
        else:
            out[r] = np.exp2(lo2 + c * st).astype(F32)
    return out, lost


def debias(w0, h, q, rungs, tab, lost, two_bit=True):
    """The whole debias of one quantized matrix.  Returns dict(tab, lost,
    scales [rows, gpr] f32 (new rung values), num, den)."""
    what = dequant(q, rungs, tab, two_bit)
    num, den = slopes(w0, what, h)
    tab2, lost2 = unshrink(lost, tab, num, den, two_bit)
    rows = tab2.shape[0]
    scales = tab2[np.arange(rows)[:, None], np.asarray(rungs)].astype(F32)
    return dict(tab=tab2, lost=lost2, scales=scales, num=num, den=den)
