"""Oracle q2tp "placed" rule: ladder placement, group rule and GPTQ sweep.

Follows ``cortiq-engine src/gpu_wgpu/gptq_dev.rs``, WGSL ``q2_level`` and
``q2tp_group`` (the per-(row, group) rule: a full search over rungs 1..31,
rounding onto the four levels -1.5, -0.5, 0.5, 1.5 times the scale, in-group
feedback), and ``cortiq-cli src/gptq.rs``, ``Q2tpRule::Placed``,
``gptq_quantize_q2tp`` / ``Q2Sweep::rows`` (the host sweep: lazy blocks of
128 columns, residuals into the rest of the block at once and into the
later columns once per block) and ``gptq_quantize_q2tp_dev`` (ladders
placed from the dead-zeroed weights, rung weights ``H_ii`` clipped at 0).
The sweep and the group rule are f32 with one rounding per operation and no
fused multiply-add, in the pages' order; the placement is f64.

Readings where the pages are silent (the converter functions
``q2tp_place_row`` and ``det_q2tp_ladder`` are called but not shown):

* group scale -- "the H_ii-weighted MSE-optimal group scale" is read as the
  exact minimiser over s > 0 of
  ``E(s) = sum_t h_t (w_t - (q2_level(w_t/s + 1.5) - 1.5) s)^2``.  E is
  continuous and piecewise quadratic in s (an element sits on an outer level
  +-1.5 s when |w_t| > s, on an inner one +-0.5 s below), every piece is
  convex and every kink is concave, so the minimum is the stationary point
  of one piece: for an outer set O,
  ``s_O = (1.5 sum_O h|w| + 0.5 sum_rest h|w|) / (2.25 sum_O h + 0.25 sum_rest h)``.
  The oracle evaluates E at s_O for every "top-k by |w|" set O (k = 0..32)
  and keeps the smallest E.  Ties: the page asks for "the" optimal scale and
  names no tie-break, while a group can have two exact optima (all |w_t|
  equal: s = a/1.5 with every weight outer and s = 2a with every weight
  inner, both E = 0) whose f64 scores differ only by rounding.  So scores
  within TIE_REL * sum_t h_t w_t^2 of the smallest count as equal (an f64
  32-term score carries errors near 1e-16 of that sum), and the smallest
  such s is taken.  A group takes part only
  when some t has ``h_t > 0`` and ``w_t != 0``; otherwise E has no positive
  minimiser and the group is left out of the ladder.
* ladder -- the layout of the host page's ``q2tp`` params: an f16 pair
  ``(lo, step)`` per row, rung 0 = 0 (the all-zero group, ``sweep_q2tp``'s
  "rung 0 = 0"), rungs 1..31 on a geometric ladder.  The cortiq rule's
  nominal ``1 + round((log2(absmax/1.5) - lo)/step)`` clamped to
  ``[0, Q2TP_LMAX]`` fixes rung c >= 1 at ``2^(lo + (c-1) step)`` and
  ``Q2TP_LMAX = 30``.  Reading: ``lo = f16(log2 min s*_g)``,
  ``step = f16(max(0, (log2 max s*_g - lo)/30))`` (0 when min == max) over
  the groups that take part, rung c = f32(2^(lo + (c-1) step)) with the
  exponent in f64; a row where no group takes part gets lo = step = 0 and
  every rung 0.
* rung search on the host (``q2tp_best_rung``, not shown) -- the device
  kernel's rule, which is on the page.

Test infrastructure: see the package docstring.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
GROUP = 32
NRUNG = 32
LMAX = 30  # rungs 1..LMAX+1
TIE_REL = 1e-12  # placement: scores this close (relative to sum h w^2) are ties
Q2_BLOCK = 128  # host page: columns per lazy-update block


def q2_level(x):
    """clamp(round_ties_even(clamp(x, -1, 4)), 0, 3), elementwise, in the
    input's precision (WGSL ``round`` rounds half to even)."""
    x = np.asarray(x)
    return np.clip(np.rint(np.clip(x, -1.0, 4.0)), 0.0, 3.0).astype(x.dtype)


# ---------------------------------------------------------------- placement


def group_err_f64(w, h, s):
    """E(s) = sum_t h_t (w_t - (q2_level(w_t/s + 1.5) - 1.5) s)^2 in f64 for
    one group (w, h of length 32) at the scale(s) s > 0 (scalar or array)."""
    w = np.asarray(w, dtype=np.float64)
    h = np.asarray(h, dtype=np.float64)
    s = np.atleast_1d(np.asarray(s, dtype=np.float64))
    q = q2_level(w[None, :] / s[:, None] + 1.5)
    d = w[None, :] - (q - 1.5) * s[:, None]
    return (h[None, :] * d * d).sum(axis=1)


def takes_part(w, h):
    """True if some channel has h > 0 and a non-zero weight."""
    w = np.asarray(w)
    h = np.asarray(h)
    return bool(np.any((h > 0) & (w != 0)))


def place_scale(w, h):
    """The weighted-MSE-optimal scale s* > 0 of one group (f64), or 0.0 when
    the group does not take part (reading in the module docstring)."""
    w = np.asarray(w, dtype=np.float64)
    h = np.asarray(h, dtype=np.float64)
    h = np.where(h > 0, h, 0.0)
    if not takes_part(w, h):
        return 0.0
    a = np.abs(w)
    order = np.argsort(-a, kind="stable")
    cands = []
    for k in range(GROUP + 1):
        outer = np.zeros(GROUP, dtype=bool)
        outer[order[:k]] = True
        num = 1.5 * np.sum(h[outer] * a[outer]) + 0.5 * np.sum(h[~outer] * a[~outer])
        den = 2.25 * np.sum(h[outer]) + 0.25 * np.sum(h[~outer])
        if den > 0 and num > 0:
            cands.append(num / den)
    cands = np.array(sorted(set(cands)))
    errs = group_err_f64(w, h, cands)
    band = errs.min() + TIE_REL * float(np.sum(h * a * a))
    return float(cands[np.nonzero(errs <= band)[0][0]])  # ascending: the smallest tied s


def _f16(x):
    return float(np.float16(np.float64(x)))


def ladder_q2tp(w_dz, hw):
    """Per-row placed ladder: tab [rows, 32] f32 (rung 0 = 0), lost
    [rows, 2] f32 = (lo, step), and the group scales s* [rows, n/32] f64
    (0 for groups that do not take part).  w_dz: dead-zeroed weights;
    hw: H_ii (clipped at 0 here)."""
    w = np.asarray(w_dz, dtype=F32)
    hw = np.asarray(hw, dtype=F32)
    rows, n = w.shape
    assert n % GROUP == 0
    gpr = n // GROUP
    gs = np.zeros((rows, gpr), dtype=np.float64)
    tab = np.zeros((rows, NRUNG), dtype=F32)
    lost = np.zeros((rows, 2), dtype=F32)
    for r in range(rows):
        for g in range(gpr):
            gs[r, g] = place_scale(w[r, g * GROUP:(g + 1) * GROUP], hw[g * GROUP:(g + 1) * GROUP])
        sp = gs[r][gs[r] > 0]
        if sp.size == 0:
            continue
        smin, smax = float(sp.min()), float(sp.max())
        lo = _f16(np.log2(smin))
        st = _f16(max(0.0, (np.log2(smax) - lo) / LMAX)) if smax > smin else 0.0
        c = np.arange(1, NRUNG, dtype=np.float64)
        tab[r, 1:] = np.exp2(lo + (c - 1.0) * st).astype(F32)
        lost[r] = (lo, st)
    return tab, lost, gs


# ---------------------------------------------------------------- group rule


def _pick_rung(tile, hg, tab):
    """Rung per row (WGSL ``q2tp_group``): 0 if the tile is all zero, else the
    best of 1..31 by sum_t hg_t d_t d_t, d_t = w_t - (q2_level(w_t (1/s) +
    1.5) - 1.5) s, summed in column order in f32; rungs with s <= 0 skipped;
    strict '<' from best = (3.4e38, rung 1)."""
    rows = tile.shape[0]
    amax = np.abs(tile).max(axis=1)
    best_c = np.where(amax > 0, 1, 0).astype(np.int64)
    best_e = np.full(rows, F32(3.4e38), dtype=F32)
    with np.errstate(all="ignore"):
        for cand in range(1, NRUNG):
            s_c = tab[:, cand]
            valid = (amax > 0) & (s_c > 0)
            iv = F32(1.0) / np.where(valid, s_c, F32(1.0))
            err = np.zeros(rows, dtype=F32)
            for t in range(GROUP):
                x = tile[:, t] * iv + F32(1.5)  # two f32 roundings
                d = tile[:, t] - (q2_level(x) - F32(1.5)) * s_c
                err = err + (hg[t] * d) * d
            take = valid & (err < best_e)
            best_e = np.where(take, err, best_e)
            best_c = np.where(take, cand, best_c)
    return best_c


def _round_col(wj, s):
    with np.errstate(all="ignore"):
        q = q2_level(wj / s + F32(1.5))
    return np.where(s > 0, q, F32(0)).astype(F32)


def group_q2tp(tile, hw, tab, ublk):
    """One 32-column group for every row (WGSL ``q2tp_group``): rung, then per
    column j the code q = q2_level(w_j / s + 1.5) (0 when s <= 0),
    e_j = (w_j - (q - 1.5) s) / U_jj (0 when U_jj <= 0) and w_t -= e_j U_jt
    for t > j.  hw is clipped at 0.

    Returns (rung [rows] int, q [rows, 32] uint8 in 0..3, e [rows, 32] f32)."""
    w = np.array(tile, dtype=F32, copy=True)
    hw = np.asarray(hw, dtype=F32)
    hw = np.where(hw > 0, hw, F32(0)).astype(F32)
    tab = np.asarray(tab, dtype=F32)
    ublk = np.asarray(ublk, dtype=F32)
    rows = w.shape[0]
    rung = _pick_rung(w, hw, tab)
    s = tab[np.arange(rows), rung]
    qs = np.zeros((rows, GROUP), dtype=np.uint8)
    es = np.zeros((rows, GROUP), dtype=F32)
    for j in range(GROUP):
        q = _round_col(w[:, j], s)
        qs[:, j] = q.astype(np.uint8)
        ujj = ublk[j, j]
        e = (w[:, j] - (q - F32(1.5)) * s) / ujj if ujj > 0 else np.zeros(rows, dtype=F32)
        es[:, j] = e
        nz = e != 0
        if j + 1 < GROUP and np.any(nz):
            w[nz, j + 1:] = w[nz, j + 1:] - e[nz, None] * ublk[j, j + 1:][None, :]
    return rung, qs, es


# ---------------------------------------------------------------- sweep


def sweep_q2tp(w0, u, hw, tab, dead=None, block=Q2_BLOCK, record=False):
    """The host q2tp GPTQ sweep, placed rule, natural order (``Q2Sweep::rows``),
    f32.

    w0 [rows, n] f32 (dead columns zeroed here first), u [n, n] f32 upper fold
    operator, hw [n] rung-error weights (clipped at 0), tab from
    ``ladder_q2tp``.  Columns go in lazy blocks of ``block``: at each group's
    first column the rung from the current tile; per column j the code and
    e_j = (w_j - (q - 1.5) s)/U_jj, then w[:, j+1:b1] -= e_j U[j, j+1:b1]
    (rows with e_j == 0 skipped); after the block, for every later column c,
    acc = sum over the block's columns t, in order, of e_t U[t, c] (f32,
    separate multiply and add, from 0) and w[:, c] -= acc.

    Returns dict(rung [rows, gpr], q [rows, n] uint8 0..3, scale [rows, gpr]
    f32, e [rows, n] f32; with record=True also tiles [gpr, rows, 32]: each
    group's tile when its rung is picked)."""
    w = np.array(w0, dtype=F32, copy=True)
    u = np.asarray(u, dtype=F32)
    hw = np.asarray(hw, dtype=F32)
    hw = np.where(hw > 0, hw, F32(0)).astype(F32)
    tab = np.asarray(tab, dtype=F32)
    rows, n = w.shape
    assert n % GROUP == 0 and u.shape == (n, n) and block % GROUP == 0
    gpr = n // GROUP
    if dead is not None:
        w[:, np.asarray(dead, dtype=bool)] = 0.0
    rung = np.zeros((rows, gpr), dtype=np.int64)
    scale = np.zeros((rows, gpr), dtype=F32)
    qall = np.zeros((rows, n), dtype=np.uint8)
    eall = np.zeros((rows, n), dtype=F32)
    tiles = np.zeros((gpr, rows, GROUP), dtype=F32) if record else None
    ridx = np.arange(rows)
    s = np.zeros(rows, dtype=F32)
    for b0 in range(0, n, block):
        b1 = min(b0 + block, n)
        for j in range(b0, b1):
            g = j // GROUP
            if j % GROUP == 0:
                tile = w[:, j:j + GROUP]
                if record:
                    tiles[g] = tile
                c = _pick_rung(tile, hw[j:j + GROUP], tab)
                rung[:, g] = c
                s = tab[ridx, c]
                scale[:, g] = s
            q = _round_col(w[:, j], s)
            qall[:, j] = q.astype(np.uint8)
            d = u[j, j]
            e = (w[:, j] - (q - F32(1.5)) * s) / d if d > 0 else np.zeros(rows, dtype=F32)
            eall[:, j] = e
            nz = np.nonzero(e != 0)[0]
            if j + 1 < b1 and nz.size:
                w[nz, j + 1:b1] = w[nz, j + 1:b1] - e[nz, None] * u[j, j + 1:b1][None, :]
        if b1 < n:
            acc = np.zeros((rows, n - b1), dtype=F32)
            for t in range(b0, b1):
                acc = acc + eall[:, t, None] * u[t, b1:][None, :]
            w[:, b1:] = w[:, b1:] - acc
    out = dict(rung=rung, q=qall, scale=scale, e=eall)
    if record:
        out["tiles"] = tiles
    return out


def sweep_q2tp_f64(w0, u, hw, tab, dead=None):
    """The same sweep with weights, residuals and updates in f64 and every
    update applied to the whole rest of the row at once (the rung search and
    the codes as the rule, in f64); for the identities W0 - Q = E U and
    tr((W0-Q) H_d (W0-Q)^T) = ||E||_F^2.  Returns (rung, q, scale, e f64)."""
    w = np.array(w0, dtype=np.float64, copy=True)
    u = np.asarray(u, dtype=np.float64)
    hw = np.asarray(hw, dtype=np.float64)
    hw = np.where(hw > 0, hw, 0.0)
    tab = np.asarray(tab, dtype=np.float64)
    rows, n = w.shape
    gpr = n // GROUP
    if dead is not None:
        w[:, np.asarray(dead, dtype=bool)] = 0.0
    rung = np.zeros((rows, gpr), dtype=np.int64)
    scale = np.zeros((rows, gpr), dtype=np.float64)
    qall = np.zeros((rows, n), dtype=np.uint8)
    eall = np.zeros((rows, n), dtype=np.float64)
    ridx = np.arange(rows)
    for g in range(gpr):
        c0 = g * GROUP
        tile = w[:, c0:c0 + GROUP]
        amax = np.abs(tile).max(axis=1)
        best_c = np.where(amax > 0, 1, 0)
        best_e = np.full(rows, 3.4e38)
        for cand in range(1, NRUNG):
            s_c = tab[:, cand]
            valid = (amax > 0) & (s_c > 0)
            with np.errstate(all="ignore"):
                sv = np.where(valid, s_c, 1.0)
                q = q2_level(tile / sv[:, None] + 1.5)
                err = (hw[c0:c0 + GROUP][None, :] * (tile - (q - 1.5) * sv[:, None]) ** 2).sum(axis=1)
            take = valid & (err < best_e)
            best_e = np.where(take, err, best_e)
            best_c = np.where(take, cand, best_c)
        s = tab[ridx, best_c]
        rung[:, g] = best_c
        scale[:, g] = s
        for j in range(c0, c0 + GROUP):
            with np.errstate(all="ignore"):
                q = np.where(s > 0, q2_level(w[:, j] / np.where(s > 0, s, 1.0) + 1.5), 0.0)
            qall[:, j] = q.astype(np.uint8)
            e = (w[:, j] - (q - 1.5) * s) / u[j, j] if u[j, j] > 0 else np.zeros(rows)
            eall[:, j] = e
            w[:, j + 1:] -= e[:, None] * u[j, j + 1:][None, :]
    return rung, qall, scale, eall


def dequant_q2tp(q, scale):
    """Q[r, c] = (q[r, c] - 1.5) * scale[r, c // 32] in f32 (q in 0..3)."""
    q = np.asarray(q)
    s = np.repeat(np.asarray(scale, dtype=F32), GROUP, axis=1)
    return (q.astype(F32) - F32(1.5)) * s


def plane_to_codes(plane, rows, n):
    """Codes [rows, n] (0..3) from the 2-bit plane: a (row, group) tile is 8
    bytes at (row * n/32 + group) * 8; column j of the group sits in byte
    j // 4 at bits 2 (j % 4) (the host page's chunk layout; the same bytes
    as the WGSL kernel's two little-endian words with bits 2 (j % 16))."""
    b = np.asarray(plane, dtype=np.uint8).reshape(rows, n // GROUP, GROUP // 4)
    out = np.empty((rows, n // GROUP, GROUP), dtype=np.uint8)
    for k in range(4):
        out[:, :, k::4] = (b >> (2 * k)) & 3
    return out.reshape(rows, n)
