"""Pins for the oracle q2tp "placed" rule (CPU only).

The oracle follows the fold page's WGSL ``q2_level`` / ``q2tp_group`` and the
host page's ``gptq_quantize_q2tp`` (placed rule).  The checks come from
outside that code: hand tables of the level map, brute force over codes and
rungs, closed forms of the optimal group scale (equal magnitudes, a single
spike), a dense scan of the scale, exact ladders from powers of two, the
GPTQ identities (W0 - Q = E U, ||E||^2 = tr((W0-Q) H_d (W0-Q)^T)), the
textbook OBS loop, and GPTQ beating round-to-nearest on correlated data.
"""
import itertools
import os

import numpy as np
import pytest

import oracle
from oracle import q2tp as o2

F32 = np.float32


def pack(h):
    n = h.shape[0]
    return np.concatenate([h[r, r:] for r in range(n)]).astype(np.float32)


def corr_problem(rows, n, t, seed, loud=(5,), dead=()):
    rng = np.random.default_rng(seed)
    lat = rng.uniform(-0.5, 0.5, (t, 4))
    mix = rng.uniform(-0.5, 0.5, (4, n))
    x = lat @ mix + 0.2 * rng.uniform(-0.5, 0.5, (t, n))
    for c in loud:
        x[:, c] *= 8.0
    for c in dead:
        x[:, c] = 0.0
    x = x.astype(F32)
    h = x.astype(np.float64).T @ x.astype(np.float64)
    w = rng.uniform(-0.5, 0.5, (rows, n)).astype(F32)
    return x, h, w


def prep(w, h, lam=0.01):
    n = h.shape[0]
    hp = pack(h.astype(F32))
    u, d, dead, lam = oracle.fold(hp, n, lam)
    wdz = w.copy()
    wdz[:, dead] = 0
    hw = np.diag(oracle.unpack_upper(hp, n)).astype(F32)
    tab, lost, gs = o2.ladder_q2tp(wdz, hw)
    return u, dead, tab, lost, hw, lam


# ---------------------------------------------------------------- level map

def test_q2_level_table():
    # clamp(round_half_even(clamp(x, -1, 4)), 0, 3), worked by hand
    # (tests/golden/q2_level.txt, with its citation).
    path = os.path.join(os.path.dirname(__file__), "golden", "q2_level.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    xs = [float(a) for a, _ in rows]
    want = [int(b) for _, b in rows]
    got = o2.q2_level(np.array(xs, dtype=F32))
    assert got.tolist() == want


def test_levels_are_nearest_of_four():
    # (q - 1.5) s is the nearest of -1.5 s, -0.5 s, 0.5 s, 1.5 s (away from
    # the midpoints, where either neighbour is nearest).
    rng = np.random.default_rng(0)
    s = 0.37
    w = rng.uniform(-1.2, 1.2, 5000)
    lv = np.array([-1.5, -0.5, 0.5, 1.5]) * s
    near = lv[np.argmin(np.abs(w[:, None] - lv[None, :]), axis=1)]
    q = o2.q2_level(w / s + 1.5)
    mid = np.min(np.abs(np.abs(w[:, None]) - np.array([0.0, s])[None, :]), axis=1) < 1e-9
    assert np.array_equal(((q - 1.5) * s)[~mid], near[~mid])


def test_codes_minimise_weighted_error_bruteforce():
    # For a fixed scale the weighted error is separable: the best of all 4^5
    # code vectors is the level map applied per column.
    rng = np.random.default_rng(1)
    s = 0.05
    hw = rng.uniform(0.1, 3, 5)
    grid = np.array(list(itertools.product(range(4), repeat=5)), dtype=np.float64)
    for _ in range(30):
        w = rng.uniform(-0.1, 0.1, 5)
        err = (((w[None, :] - (grid - 1.5) * s) ** 2) * hw).sum(axis=1)
        assert np.array_equal(grid[np.argmin(err)], o2.q2_level(w / s + 1.5))


# ---------------------------------------------------------------- placement

def test_place_scale_equal_magnitudes():
    # |w_t| = a for every t: two scales fit exactly (E = 0), s = a/1.5 (every
    # weight on an outer level) and s = 2a (every weight on an inner level);
    # their f64 scores differ by rounding only, so they tie and the smaller,
    # a/1.5, is taken, whatever the signs and weights.
    rng = np.random.default_rng(2)
    for a in (0.3, 1e-3, 17.0, 0.05):
        for trial in range(5):
            w = a * rng.choice([-1.0, 1.0], 32)
            h = rng.uniform(0.1, 5, 32)
            s = o2.place_scale(w, h)
            assert abs(s / (a / 1.5) - 1) < 1e-12
            assert o2.group_err_f64(w, h, s)[0] <= 1e-28 * a * a
            assert o2.group_err_f64(w, h, 2 * a)[0] <= 1e-28 * a * a


def test_place_scale_tie_band():
    # Two pieces whose exact scores differ by far more than the band are not
    # ties: shrinking the outer weights a little makes the all-inner fit
    # (s = 2 * median-like scale) strictly better or worse, and the smaller
    # score wins whichever scale it has.
    w = np.full(32, 0.05)
    w[:16] = 0.05 * (1 - 1e-3)
    h = np.ones(32)
    s = o2.place_scale(w, h)
    cands = np.linspace(0.01, 0.15, 20001)
    e = o2.group_err_f64(w, h, cands)
    assert o2.group_err_f64(w, h, s)[0] <= e.min() + 1e-15


def test_place_scale_single_spike_closed_form():
    # One weight a, 31 zeros, unit weights.  Outer piece: s = 1.5 a / (2.25 +
    # 31 * 0.25) = 0.15 a (inside its piece, s <= a), E = (a - 0.225 a)^2 +
    # 31 (0.075 a)^2 = 0.775 a^2; the all-inner piece's stationary point
    # (a/16) lies outside it.  So s* = 0.15 a.
    w = np.zeros(32)
    w[11] = -2.0
    s = o2.place_scale(w, np.ones(32))
    assert s == pytest.approx(0.3, rel=1e-12)
    assert o2.group_err_f64(w, np.ones(32), s)[0] == pytest.approx(0.775 * 4.0, rel=1e-12)


def test_place_scale_beats_dense_scan():
    # No scale on a dense geometric grid (plus a local refinement around the
    # best grid point) has a smaller weighted error than s*.
    rng = np.random.default_rng(3)
    for trial in range(40):
        w = rng.standard_normal(32) * 0.02
        if trial % 3 == 0:
            w[rng.integers(0, 32)] *= 12.0  # an outlier
        h = rng.lognormal(0.0, 1.0, 32)
        if trial % 4 == 1:
            h[rng.integers(0, 32, 5)] = 0.0
        s = o2.place_scale(w, h)
        e_star = o2.group_err_f64(w, h, s)[0]
        amax = np.abs(w).max()
        grid = amax * np.exp(np.linspace(np.log(1e-3), np.log(3.0), 40001))
        eg = o2.group_err_f64(w, h, grid)
        k = int(np.argmin(eg))
        fine = np.linspace(grid[max(k - 1, 0)], grid[min(k + 1, len(grid) - 1)], 4001)
        ef = o2.group_err_f64(w, h, fine)
        assert e_star <= min(eg.min(), ef.min()) * (1 + 1e-12)


def test_place_scale_invariances():
    rng = np.random.default_rng(4)
    w = rng.standard_normal(32) * 0.03
    h = rng.uniform(0.2, 4, 32)
    s = o2.place_scale(w, h)
    assert o2.place_scale(8.0 * w, h) == 8.0 * s          # scale covariance (exact)
    assert o2.place_scale(w, 0.25 * h) == s               # weight scaling (exact)
    assert o2.place_scale(-w, h) == s                     # signs
    p = rng.permutation(32)
    assert o2.place_scale(w[p], h[p]) == pytest.approx(s, rel=1e-12)


def test_place_scale_unweighted_channels():
    # A weight on an h = 0 channel does not enter E; a group whose non-zero
    # weights all sit on such channels does not take part (scale 0).
    rng = np.random.default_rng(5)
    w = rng.standard_normal(32) * 0.03
    h = rng.uniform(0.2, 4, 32)
    h[[3, 17]] = 0.0
    s = o2.place_scale(w, h)
    w2 = w.copy()
    w2[[3, 17]] = [5.0, -9.0]
    assert o2.place_scale(w2, h) == pytest.approx(s, rel=1e-14)
    z = np.zeros(32)
    z[[3, 17]] = [1.0, 2.0]
    assert o2.place_scale(z, h) == 0.0
    assert o2.place_scale(np.zeros(32), h) == 0.0


# ---------------------------------------------------------------- ladder

def test_ladder_powers_of_two():
    # A group holding one weight a among zeros (unit weights) has s* = 0.15 a
    # (the single-spike closed form); with a = 2^p / 0.15 the group scales are
    # 2^p up to the f32 rounding of a, so lo = min p and step = (max p -
    # min p)/30 after the f16 rounding: p in {-10, -5, 5} gives step 0.5 and
    # rung c = 2^(-10 + (c-1)/2) exactly; rung 0 is 0.
    ps = [-5, -10, 5]
    row = np.zeros(32 * len(ps), dtype=F32)
    for g, p in enumerate(ps):
        row[g * 32 + 7 + g] = (-1) ** g * F32(2.0 ** p / 0.15)
    tab, lost, gs = o2.ladder_q2tp(row[None, :], np.ones(96, dtype=F32))
    np.testing.assert_allclose(gs[0], [2.0 ** -5, 2.0 ** -10, 2.0 ** 5], rtol=1e-7)
    assert lost[0].tolist() == [-10.0, 0.5]
    assert tab[0, 0] == 0.0
    want = [2.0 ** (-10 + (c - 1) / 2) for c in range(1, 32)]
    assert np.array_equal(tab[0, 1:], np.array(want, dtype=F32))


def test_ladder_degenerate_rows():
    hw = np.ones(64, dtype=F32)
    hw[40:] = 0.0
    w = np.zeros((3, 64), dtype=F32)
    w[1, 5] = 3.0           # one group takes part: step 0
    w[2, 40:44] = 0.5       # non-zero weights only on h = 0 channels
    tab, lost, _ = o2.ladder_q2tp(w, hw)
    assert np.all(tab[0] == 0) and np.all(lost[0] == 0)
    assert np.all(tab[2] == 0) and np.all(lost[2] == 0)
    lo1 = float(np.float16(np.log2(0.45)))     # s* = 0.15 * 3 (single spike)
    assert lost[1].tolist() == [F32(lo1), 0.0]
    assert tab[1, 0] == 0 and np.all(tab[1, 1:] == F32(2.0 ** lo1))
    # Two groups with the same scale: min == max, step 0.
    w2 = np.zeros((1, 64), dtype=F32)
    w2[0, 3] = 3.0
    w2[0, 60] = -3.0
    tab2, lost2, gs2 = o2.ladder_q2tp(w2, np.ones(64, dtype=F32))
    assert gs2[0, 0] == gs2[0, 1] and lost2[0].tolist() == [F32(lo1), 0.0]


# ---------------------------------------------------------------- group rule

def test_group_rung_is_full_argmin():
    # The chosen rung's weighted error (f64, nearest levels) is <= that of
    # every rung 1..31, strictly below the lower ones, up to f32 rounding.
    rng = np.random.default_rng(7)
    rows = 150
    tile = (rng.standard_normal((rows, 32)) * 0.02).astype(F32)
    hw = rng.uniform(0.01, 5, 32).astype(F32)
    wide = np.tile(tile, (1, 6)) * rng.uniform(0.3, 3, (1, 192)).astype(F32)
    tab, lost, _ = o2.ladder_q2tp(wide, np.tile(hw, 6))
    rung, q, e = o2.group_q2tp(tile, hw, tab, np.eye(32, dtype=F32))
    for r in range(rows):
        errs = {}
        for c in range(1, 32):
            s = np.float64(tab[r, c])
            errs[c] = float(o2.group_err_f64(tile[r], hw, s)[0])
        c0 = int(rung[r])
        assert 1 <= c0 <= 31
        for c, v in errs.items():
            if c < c0:
                assert errs[c0] < v * (1 + 1e-5)
            else:
                assert errs[c0] <= v * (1 + 1e-5)
        s0 = np.float64(tab[r, c0])
        assert np.array_equal(q[r], o2.q2_level(tile[r].astype(np.float64) / s0 + 1.5).astype(np.uint8))


def test_group_degenerate_cases():
    rng = np.random.default_rng(8)
    tile = (rng.standard_normal((6, 32)) * 0.02).astype(F32)
    tile[0] = 0.0
    tab = np.zeros((6, 32), dtype=F32)
    tab[:, 1:] = np.geomspace(1e-3, 0.05, 31, dtype=F32)[None, :]
    tab[3, 1:9] = 0.0  # rungs with s <= 0 are skipped
    tab[4, :] = 0.0    # nothing valid: the default rung 1 with s = 0
    hw = rng.uniform(0.5, 2, 32).astype(F32)
    rung, q, e = o2.group_q2tp(tile, hw, tab, np.eye(32, dtype=F32))
    assert rung[0] == 0 and np.all(q[0] == 0) and np.all(e[0] == 0)
    assert rung[3] >= 9
    assert rung[4] == 1 and np.all(q[4] == 0)
    np.testing.assert_array_equal(e[4], tile[4])  # e = (w - (-1.5) * 0) / 1
    # hw = 0: every error is 0 and the strict '<' keeps the first valid rung.
    rung0, _, _ = o2.group_q2tp(tile, np.zeros(32, F32), tab, np.eye(32, dtype=F32))
    assert rung0.tolist() == [0, 1, 1, 9, 1, 1]


def test_group_feedback_identity():
    # Inside a tile the recursion gives w_start - Q = E U_blk (f64 check of
    # the f32 rule): the feedback sign, index and divisor.
    rng = np.random.default_rng(9)
    rows = 40
    tile = (rng.standard_normal((rows, 32)) * 0.02).astype(F32)
    a = rng.standard_normal((32, 32))
    ublk = np.triu(a * 0.1) + np.diag(rng.uniform(0.5, 1.5, 32))
    ublk = ublk.astype(F32)
    tab = np.zeros((rows, 32), dtype=F32)
    tab[:, 1:] = np.geomspace(2e-3, 0.1, 31, dtype=F32)[None, :]
    hw = np.ones(32, dtype=F32)
    rung, q, e = o2.group_q2tp(tile, hw, tab, ublk)
    s = tab[np.arange(rows), rung].astype(np.float64)
    qv = (q.astype(np.float64) - 1.5) * s[:, None]
    gap = (tile.astype(np.float64) - qv) - e.astype(np.float64) @ ublk.astype(np.float64)
    assert np.abs(gap).max() < 1e-6


def test_plane_layout():
    rng = np.random.default_rng(10)
    rows, n = 3, 96
    q = rng.integers(0, 4, (rows, n))
    plane = np.zeros(rows * n // 4, dtype=np.uint8)
    for r in range(rows):
        for c in range(n):
            g, j = divmod(c, 32)
            plane[(r * (n // 32) + g) * 8 + j // 4] |= q[r, c] << (2 * (j % 4))
    assert np.array_equal(o2.plane_to_codes(plane, rows, n), q)
    # The same bytes as two little-endian words with bits 2 (j % 16).
    words = np.zeros(rows * n // 16, dtype=np.uint32)
    for r in range(rows):
        for c in range(n):
            g, j = divmod(c, 32)
            words[(r * (n // 32) + g) * 2 + j // 16] |= np.uint32(q[r, c]) << np.uint32(2 * (j % 16))
    assert np.array_equal(words.view(np.uint8), plane)


# ---------------------------------------------------------------- sweep

def test_identity_w0_minus_q_equals_e_u():
    _, h, w = corr_problem(16, 160, 300, 11, dead=(40,))
    u, dead, tab, lost, hw, lam = prep(w, h)
    wdz = w.copy()
    wdz[:, dead] = 0
    rung, q, sc, e = o2.sweep_q2tp_f64(w, u, hw, tab, dead)
    qw = (q.astype(np.float64) - 1.5) * np.repeat(sc, 32, axis=1)
    np.testing.assert_allclose(wdz - qw, e @ u, rtol=0, atol=1e-12)
    dd, hf, base = oracle.fold_damping(pack(h.astype(F32)), 160)
    hd = hf + lam * base * np.eye(160)
    assert oracle.output_error(wdz, qw, hd) == pytest.approx(float((e * e).sum()), rel=1e-10)
    r32 = o2.sweep_q2tp(w, u.astype(F32), hw, tab, dead)
    q32 = o2.dequant_q2tp(r32["q"], r32["scale"]).astype(np.float64)
    gap = (wdz - q32) - r32["e"].astype(np.float64) @ u
    assert np.abs(gap).max() < 2e-5 * np.abs(w).max()
    assert (r32["q"] == q).mean() > 0.99


def test_block_width_changes_only_rounding():
    # Lazy blocks of 32, 128 and 160 columns are the same recursion: the
    # codes agree and the residuals differ by f32 summation order only.
    _, h, w = corr_problem(24, 160, 400, 12)
    u, dead, tab, lost, hw, _ = prep(w, h)
    u32 = u.astype(F32)
    ref = o2.sweep_q2tp(w, u32, hw, tab, dead, block=128)
    for b in (32, 160):
        r = o2.sweep_q2tp(w, u32, hw, tab, dead, block=b)
        assert (r["q"] == ref["q"]).mean() > 0.995
        both = (r["q"] == ref["q"]).all(axis=1)
        np.testing.assert_allclose(r["e"][both], ref["e"][both], rtol=0, atol=1e-4 * np.abs(ref["e"]).max())


def test_sweep_matches_textbook_obs_loop():
    # Every rung equal, so the codes depend on the update rule alone; the OBS
    # loop moves the remaining weights by -(w_j - Q_j) inv(H_d[j:, j:])[0, 1:]
    # / inv(H_d[j:, j:])[0, 0] after each column.
    n, rows = 32, 6
    _, h, w = corr_problem(rows, n, 200, 13)
    u, dead, _, _, hw, lam = prep(w, h)
    dd, hf, base = oracle.fold_damping(pack(h.astype(F32)), n)
    hd = hf + lam * base * np.eye(n)
    s = 0.12
    tab = np.full((rows, 32), s)
    tab[:, 0] = 0.0
    rung, q, sc, e = o2.sweep_q2tp_f64(w, u, hw, tab)
    for r in range(rows):
        wt = w[r].astype(np.float64).copy()
        for j in range(n):
            qj = o2.q2_level(np.float64(wt[j] / s + 1.5))
            assert qj == q[r, j]
            if j + 1 < n:
                t = np.linalg.inv(hd[j:, j:])
                wt[j + 1:] -= (wt[j] - (qj - 1.5) * s) * t[0, 1:] / t[0, 0]


def test_diagonal_h_is_groupwise():
    rng = np.random.default_rng(14)
    n, rows = 128, 20
    h = np.diag(rng.uniform(0.5, 4, n)).astype(F32)
    w = (rng.standard_normal((rows, n)) * 0.02).astype(F32)
    u, dead, tab, lost, hw, _ = prep(w, h)
    res = o2.sweep_q2tp(w, u.astype(F32), hw, tab, dead)
    for g in range(n // 32):
        c0 = g * 32
        rung, q, e = o2.group_q2tp(w[:, c0:c0 + 32], hw[c0:c0 + 32], tab,
                                   u.astype(F32)[c0:c0 + 32, c0:c0 + 32])
        assert np.array_equal(rung, res["rung"][:, g])
        assert np.array_equal(q, res["q"][:, c0:c0 + 32])


def test_group_rule_reproduces_sweep_tiles():
    # The group rule fed each group's tile (as the sweep saw it at the
    # group's first column) reproduces codes, rungs and residuals bit for bit.
    _, h, w = corr_problem(24, 192, 400, 15, dead=(70,))
    u, dead, tab, lost, hw, _ = prep(w, h)
    u32 = u.astype(F32)
    res = o2.sweep_q2tp(w, u32, hw, tab, dead, record=True)
    for g in range(6):
        c0 = g * 32
        rung, q, e = o2.group_q2tp(res["tiles"][g], hw[c0:c0 + 32], tab, u32[c0:c0 + 32, c0:c0 + 32])
        assert np.array_equal(rung, res["rung"][:, g])
        assert np.array_equal(q, res["q"][:, c0:c0 + 32])
        assert np.array_equal(e.view(np.uint32), res["e"][:, c0:c0 + 32].view(np.uint32))


def test_dead_group_is_independent():
    rows, n = 10, 96
    x, h, w = corr_problem(rows, n, 300, 16, dead=tuple(range(32, 64)))
    u, dead, tab, lost, hw, lam = prep(w, h)
    res = o2.sweep_q2tp(w, u.astype(F32), hw, tab, dead)
    keep = np.r_[0:32, 64:96]
    h2 = h[np.ix_(keep, keep)]
    lam2 = lam * ((np.trace(h) + 32) / n) / (np.trace(h2) / 64)
    u2, _, _, _ = oracle.fold(pack(h2.astype(F32)), 64, lam2)
    res2 = o2.sweep_q2tp(w[:, keep], u2.astype(F32), hw[keep], tab)
    assert np.all(res["rung"][:, 1] == 0)
    assert np.all(res["e"][:, 32:64] == 0)
    assert (res["q"][:, keep] == res2["q"]).mean() > 0.999


def test_gptq_beats_rtn_on_output_error():
    rows, n, t = 24, 96, 400
    x, h, w = corr_problem(rows, n, t, 17)
    u, dead, tab, lost, hw, _ = prep(w, h)
    g = o2.sweep_q2tp(w, u.astype(F32), hw, tab, dead)
    r = o2.sweep_q2tp(w, np.eye(n, dtype=F32), hw, tab, dead)
    eg = oracle.output_error(w, o2.dequant_q2tp(g["q"], g["scale"]), h)
    er = oracle.output_error(w, o2.dequant_q2tp(r["q"], r["scale"]), h)
    assert eg < 0.8 * er
