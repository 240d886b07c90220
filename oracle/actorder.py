"""Oracle act-order q4tp (f32 sweep, f64 fold), following ``cortiq-cli
src/gptq.rs``: ``act_order_perm`` (channels by descending H_ii, ties by
index, Rust ``total_cmp`` order), ``permute_sym`` (H[perm][perm]) and
``gptq_quantize_q4tp_act_order`` (channels eliminated in perm order against
the fold operator of the permuted Hessian; each tile's rung fixed up front,
"static groups", so only the codes move).

Reading where the pages are silent: the static rung is "the converter's own
choice from the original weights", and the converter is not on the pages.
Here it is the q4tp rung rule on the dead-zeroed original tile with unit
weights (no Hessian: the converter is a round-to-nearest encoder) -- nominal
from absmax, best of nominal-2..+1 by the plain squared error.

Test infrastructure: see the package docstring.
"""
from __future__ import annotations

import numpy as np

from .fold import unpack_upper
from .gram import pack_upper
from .q4tp import F32, GROUP, _pick_rung, _round_col


def total_cmp_key(x):
    """Rust f32::total_cmp as a signed integer key (NaN and -0.0 ordered)."""
    b = np.asarray(x, dtype=np.float32).view(np.int32).astype(np.int64)
    return np.where(b < 0, b ^ 0x7FFFFFFF, b)


def act_order_perm(hdiag):
    """Indices by descending H_ii (total order), ties by ascending index."""
    key = total_cmp_key(hdiag)
    idx = np.arange(key.size)
    return np.lexsort((idx, -key))


def permute_packed(hp, n, perm):
    """Packed upper triangle of H[perm][perm]."""
    h = unpack_upper(hp, n)
    return pack_upper(h[np.ix_(perm, perm)]).astype(np.float32)


def converter_rungs(w_dz, tab, lost):
    """Static rung per (row, group): the rung rule with unit weights on the
    dead-zeroed original weights (reading in the module docstring)."""
    w = np.asarray(w_dz, dtype=F32)
    rows, n = w.shape
    ones = np.ones(GROUP, dtype=F32)
    out = np.zeros((rows, n // GROUP), dtype=np.int64)
    for g in range(n // GROUP):
        out[:, g] = _pick_rung(w[:, g * GROUP:(g + 1) * GROUP], ones, tab, lost)
    return out


def sweep_q4tp_act_order(w0, u_perm, dead, perm, tab, rungs):
    """The host page's act-order sweep in f32.

    w0 [rows, n] original order (dead columns zeroed here), u_perm the fold
    operator of H[perm][perm] (f32), rungs [rows, n/32] static.  Column a of
    the sweep is channel perm[a]: code clamp(rne(w / s)) with s the static
    scale of its original group, e = (w - q s) / U_aa, then
    w[a+1..] -= e * U[a, a+1..] in permuted order.  Returns dict(q [rows, n]
    in original channel order, scale [rows, n/32], e [rows, n] permuted).
    """
    w0 = np.asarray(w0, dtype=F32)
    rows, n = w0.shape
    perm = np.asarray(perm)
    u = np.asarray(u_perm, dtype=F32)
    tab = np.asarray(tab, dtype=F32)
    wdz = w0.copy()
    if dead is not None:
        wdz[:, np.asarray(dead, dtype=bool)] = 0.0
    ridx = np.arange(rows)
    scale = tab[ridx[:, None], rungs]  # [rows, gpr]
    w = wdz[:, perm].copy()
    sperm = scale[:, perm // GROUP]
    q_orig = np.zeros((rows, n), dtype=np.int8)
    e_all = np.zeros((rows, n), dtype=F32)
    for a in range(n):
        s = sperm[:, a]
        q = _round_col(w[:, a], s)
        q_orig[:, perm[a]] = q.astype(np.int8)
        d = u[a, a]
        e = (w[:, a] - q * s) / d if d > 0 else np.zeros(rows, dtype=F32)
        e_all[:, a] = e
        nz = np.nonzero(e != 0)[0]
        if a + 1 < n and nz.size:
            w[nz, a + 1:] = w[nz, a + 1:] - e[nz, None] * u[a, a + 1:][None, :]
    return dict(q=q_orig, scale=scale, e=e_all)
