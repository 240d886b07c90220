"""Oracle q4tp ladder, rung rule and GPTQ sweep (f32, as the pages compute).

Follows ``cortiq-cli src/gptq.rs``, ``gptq_quantize_q4tp`` (host sweep) and
``cortiq-engine src/gpu_wgpu/gptq_dev.rs``, WGSL ``q4tp_group`` (the same rule
per row and group).  The pages fix f32 for the sweep, so every step here is
f32 with one rounding per operation and no fused multiply-add (numpy's
elementwise ufuncs), in the pages' order.  ``sweep_q4tp_f64`` is the same
loop in f64 for the algebraic identities the tests check.

Readings where the pages are silent:

* ladder -- the converter (``encode_q4tp`` / ``q4tp_ladder``) is not on the
  pages, only its shape: per row an f16 ``(lo, step)`` and 32 rungs
  ``2^(lo + c step)``, nominal from ``absmax / 7``.  Reading: over the
  dead-zeroed original row, ``x_g = f32(absmax_g / 7)`` for groups with
  ``absmax_g > 0``; ``lo = f16(log2 min x_g)``; ``step = f16(max(0,
  (log2 max x_g - lo) / 31))`` or 0 when ``min == max``; rung
  ``c = f32(2^(lo + c step))`` with the exponent in f64; an all-zero row
  has ``lo = step = 0`` and every rung 0.
* nominal rung -- ``log2`` of an f32 differs by an ulp between libraries;
  here (and in the library) it is the f64 ``log2`` rounded to f32 (the
  correctly rounded f32 value, barring a 2^-29 chance), the rest of the
  formula stays f32: ``t = (log2(amax/7) - lo) / step``, rounded half away
  from zero (Rust ``f32::round``), clamped to [0, 31].

Test infrastructure: see the package docstring.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
GROUP = 32
NRUNG = 32


def _f16(x):
    """Round f64 values to the nearest f16 (ties to even), back as f64."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def ladder(w_dz):
    """Per-row rung table ``tab`` [rows, 32] f32 and ``lost`` [rows, 2] f32
    (lo, step) from the dead-zeroed original weights (reading stated in the
    module docstring)."""
    w = np.asarray(w_dz, dtype=F32)
    rows, n = w.shape
    assert n % GROUP == 0
    amax = np.abs(w).reshape(rows, n // GROUP, GROUP).max(axis=2)  # f32, exact
    x = amax / F32(7.0)  # f32 division
    pos = amax > 0
    tab = np.zeros((rows, NRUNG), dtype=F32)
    lost = np.zeros((rows, 2), dtype=F32)
    for r in range(rows):
        xs = x[r][pos[r]]
        if xs.size == 0:
            continue
        xmin = float(xs.min())
        xmax = float(xs.max())
        lo = float(_f16(np.log2(xmin)))
        if xmax > xmin:
            st = float(_f16(max(0.0, (np.log2(xmax) - lo) / 31.0)))
        else:
            st = 0.0
        c = np.arange(NRUNG, dtype=np.float64)
        tab[r] = np.exp2(lo + c * st).astype(F32)
        lost[r] = (lo, st)
    return tab, lost


def _round_half_away(t):
    """Nearest integer, ties away from zero, exactly (f32 in, f32 out)."""
    a = np.abs(t)
    f = np.floor(a)
    r = f + (a - f >= F32(0.5)).astype(F32)
    return np.copysign(r, t).astype(F32)


def nominal_rung(amax, lo, st):
    """Nominal rung per row: 0 unless amax > 0 and step > 0; else
    clamp(round_half_away((log2(f32(amax/7)) - lo) / step), 0, 31) in f32
    (log2 as the f64 value rounded to f32)."""
    amax = np.asarray(amax, dtype=F32)
    lo = np.asarray(lo, dtype=F32)
    st = np.asarray(st, dtype=F32)
    ok = (amax > 0) & (st > 0)
    out = np.zeros(amax.shape, dtype=np.int64)
    if np.any(ok):
        with np.errstate(all="ignore"):
            x = amax[ok] / F32(7.0)
            l2 = np.log2(x.astype(np.float64)).astype(F32)
            t = (l2 - lo[ok]) / st[ok]
            r = np.clip(_round_half_away(t), F32(0), F32(NRUNG - 1))
        out[ok] = r.astype(np.int64)
    return out


def _pick_rung(tile, hw, tab, lost):
    """Rung per row for one group tile (rows x 32, the corrected weights):
    best of nominal-2 .. min(nominal+1, 31) by the hw-weighted error of
    clamp(rne(w * (1/s)), -8, 7); strict '<' (lowest index wins a tie);
    skips rungs with s <= 0; an all-zero tile keeps rung 0."""
    rows = tile.shape[0]
    amax = np.abs(tile).max(axis=1)
    nom = nominal_rung(amax, lost[:, 0], lost[:, 1])
    best_c = nom.copy()
    best_e = np.full(rows, np.inf, dtype=F32)
    lo_c = np.maximum(nom - 2, 0)
    hi_c = np.minimum(nom + 1, NRUNG - 1)
    ridx = np.arange(rows)
    with np.errstate(all="ignore"):
        for k in range(4):
            cand = lo_c + k
            valid = (cand <= hi_c) & (amax > 0)
            cand = np.minimum(cand, NRUNG - 1)
            s_c = tab[ridx, cand]
            valid &= s_c > 0
            iv = F32(1.0) / s_c
            err = np.zeros(rows, dtype=F32)
            for t in range(GROUP):
                q = np.clip(np.rint(tile[:, t] * iv), F32(-8), F32(7))
                d = tile[:, t] - q * s_c
                err = err + (hw[t] * d) * d
            take = valid & (err < best_e)
            best_e = np.where(take, err, best_e)
            best_c = np.where(take, cand, best_c)
    return best_c


def _round_col(wj, s):
    with np.errstate(all="ignore"):
        q = np.clip(np.rint(wj / s), F32(-8), F32(7))
    return np.where(s > 0, q, F32(0)).astype(F32)


def group_q4tp(tile, hw, tab, lost, ublk):
    """One 32-column group for every row, exactly the per-row device rule
    (WGSL ``q4tp_group``): rung, then per column j the code
    ``q = clamp(rne(w_j / s), -8, 7)``, ``e_j = (w_j - q s) / U_jj``
    (0 when U_jj <= 0) and the in-group feedback ``w_t -= e_j U_jt``, t > j.

    tile [rows, 32] f32 (copied), hw [32] f32, tab [rows, 32], lost [rows, 2],
    ublk [32, 32] f32 = U[c0:c0+32, c0:c0+32].
    Returns (rung [rows] int, q [rows, 32] int8, e [rows, 32] f32).
    """
    w = np.array(tile, dtype=F32, copy=True)
    hw = np.asarray(hw, dtype=F32)
    tab = np.asarray(tab, dtype=F32)
    lost = np.asarray(lost, dtype=F32)
    ublk = np.asarray(ublk, dtype=F32)
    rows = w.shape[0]
    rung = _pick_rung(w, hw, tab, lost)
    s = tab[np.arange(rows), rung]
    qs = np.zeros((rows, GROUP), dtype=np.int8)
    es = np.zeros((rows, GROUP), dtype=F32)
    for j in range(GROUP):
        q = _round_col(w[:, j], s)
        qs[:, j] = q.astype(np.int8)
        ujj = ublk[j, j]
        if ujj > 0:
            e = (w[:, j] - q * s) / ujj
        else:
            e = np.zeros(rows, dtype=F32)
        es[:, j] = e
        nz = e != 0
        if j + 1 < GROUP and np.any(nz):
            w[nz, j + 1 :] = w[nz, j + 1 :] - e[nz, None] * ublk[j, j + 1 :][None, :]
    return rung, qs, es


def sweep_q4tp(w0, u, hw, tab, lost, dead=None, record=False):
    """The host q4tp GPTQ sweep (``gptq_quantize_q4tp``), f32.

    w0 [rows, n] f32 (dead columns are zeroed here first), u [n, n] f32 upper
    fold operator, hw [n] f32 rung-error weights (raw H_ii), tab/lost from
    ``ladder``.  Per group: the rung from the current (corrected) weights;
    then for each column j the code, ``e = (w - q s) / U_jj`` and at once
    the full-row update ``w[:, j+1:] -= e * U[j, j+1:]``.

    Returns dict(rung [rows, gpr] int, q [rows, n] int8, scale [rows, gpr] f32,
    e [rows, n] f32, and with record=True tiles [gpr, rows, 32]: each group's
    starting tile).
    """
    w = np.array(w0, dtype=F32, copy=True)
    u = np.asarray(u, dtype=F32)
    hw = np.asarray(hw, dtype=F32)
    tab = np.asarray(tab, dtype=F32)
    lost = np.asarray(lost, dtype=F32)
    rows, n = w.shape
    assert n % GROUP == 0 and u.shape == (n, n)
    gpr = n // GROUP
    if dead is not None:
        w[:, np.asarray(dead, dtype=bool)] = 0.0
    rung = np.zeros((rows, gpr), dtype=np.int64)
    scale = np.zeros((rows, gpr), dtype=F32)
    qall = np.zeros((rows, n), dtype=np.int8)
    eall = np.zeros((rows, n), dtype=F32)
    tiles = np.zeros((gpr, rows, GROUP), dtype=F32) if record else None
    ridx = np.arange(rows)
    for g in range(gpr):
        c0 = g * GROUP
        if record:
            tiles[g] = w[:, c0 : c0 + GROUP]
        c = _pick_rung(w[:, c0 : c0 + GROUP], hw[c0 : c0 + GROUP], tab, lost)
        s = tab[ridx, c]
        rung[:, g] = c
        scale[:, g] = s
        for j in range(c0, c0 + GROUP):
            q = _round_col(w[:, j], s)
            qall[:, j] = q.astype(np.int8)
            d = u[j, j]
            if d > 0:
                e = (w[:, j] - q * s) / d
            else:
                e = np.zeros(rows, dtype=F32)
            eall[:, j] = e
            nz = np.nonzero(e != 0)[0]
            if j + 1 < n and nz.size:
                w[nz, j + 1 :] = w[nz, j + 1 :] - e[nz, None] * u[j, j + 1 :][None, :]
    out = dict(rung=rung, q=qall, scale=scale, e=eall)
    if record:
        out["tiles"] = tiles
    return out


def sweep_q4tp_f64(w0, u, hw, tab, lost, dead=None):
    """``sweep_q4tp`` with every weight, residual and update in f64 (codes are
    still the rung rule's); for the identities W0 - Q = E U and
    tr((W0-Q) H_d (W0-Q)^T) = ||E||_F^2.  Returns (rung, q, scale, e) with e f64."""
    w = np.array(w0, dtype=np.float64, copy=True)
    u = np.asarray(u, dtype=np.float64)
    hw = np.asarray(hw, dtype=np.float64)
    tab = np.asarray(tab, dtype=np.float64)
    lost = np.asarray(lost, dtype=np.float64)
    rows, n = w.shape
    gpr = n // GROUP
    if dead is not None:
        w[:, np.asarray(dead, dtype=bool)] = 0.0
    rung = np.zeros((rows, gpr), dtype=np.int64)
    scale = np.zeros((rows, gpr), dtype=np.float64)
    qall = np.zeros((rows, n), dtype=np.int8)
    eall = np.zeros((rows, n), dtype=np.float64)
    ridx = np.arange(rows)
    for g in range(gpr):
        c0 = g * GROUP
        tile = w[:, c0 : c0 + GROUP]
        amax = np.abs(tile).max(axis=1)
        nom = nominal_rung(amax.astype(F32), lost[:, 0], lost[:, 1])
        best_c, best_e = nom.copy(), np.full(rows, np.inf)
        for k in range(4):
            cand = np.maximum(nom - 2, 0) + k
            valid = (cand <= np.minimum(nom + 1, NRUNG - 1)) & (amax > 0)
            cand = np.minimum(cand, NRUNG - 1)
            s_c = tab[ridx, cand]
            valid &= s_c > 0
            with np.errstate(all="ignore"):
                q = np.clip(np.rint(tile / s_c[:, None]), -8, 7)
                err = ((tile - q * s_c[:, None]) ** 2 * hw[c0 : c0 + GROUP][None, :]).sum(axis=1)
            take = valid & (err < best_e)
            best_e = np.where(take, err, best_e)
            best_c = np.where(take, cand, best_c)
        s = tab[ridx, best_c]
        rung[:, g] = best_c
        scale[:, g] = s
        for j in range(c0, c0 + GROUP):
            with np.errstate(all="ignore"):
                q = np.where(s > 0, np.clip(np.rint(w[:, j] / s), -8, 7), 0.0)
            qall[:, j] = q.astype(np.int8)
            e = (w[:, j] - q * s) / u[j, j] if u[j, j] > 0 else np.zeros(rows)
            eall[:, j] = e
            w[:, j + 1 :] -= e[:, None] * u[j, j + 1 :][None, :]
    return rung, qall, scale, eall


def dequant_q4tp(q, scale):
    """Q[r, c] = q[r, c] * scale[r, c // 32] in f32 (q = nibble - 8)."""
    q = np.asarray(q)
    rows, n = q.shape
    s = np.repeat(np.asarray(scale, dtype=F32), GROUP, axis=1)
    return q.astype(F32) * s


def nibbles_to_codes(plane, rows, n):
    """Signed codes [rows, n] from the nibble plane: a (row, group) tile is 16
    bytes at (row * n/32 + group) * 16; column j of the group sits in byte
    j // 2, low nibble for even j; nibble = q + 8."""
    b = np.asarray(plane, dtype=np.uint8).reshape(rows, n // GROUP, GROUP // 2)
    lo = (b & 0x0F).astype(np.int16) - 8
    hi = (b >> 4).astype(np.int16) - 8
    out = np.empty((rows, n // GROUP, GROUP), dtype=np.int8)
    out[:, :, 0::2] = lo
    out[:, :, 1::2] = hi
    return out.reshape(rows, n)


def output_error(w0, qw, h):
    """tr((W0 - Q) H (W0 - Q)^T) in f64 (the layer-output error on the
    calibration set, up to the 1/T of H)."""
    d = np.asarray(w0, dtype=np.float64) - np.asarray(qw, dtype=np.float64)
    return float(np.sum((d @ np.asarray(h, dtype=np.float64)) * d))
