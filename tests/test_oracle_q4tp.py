"""Pins for the oracle ladder, rung rule and q4tp sweep (CPU only).

The oracle follows ``cortiq-cli src/gptq.rs``, ``gptq_quantize_q4tp`` and the
fold page's WGSL ``q4tp_group``.  The checks below come from outside that
code: brute force over codes and rungs, exact ladders built from powers of
two, the algebraic identities of the GPTQ recursion (W0 - Q = E U and
||E||_F^2 = tr((W0-Q) H_d (W0-Q)^T)), a textbook OBS loop with explicit
inverses of trailing blocks, and the pages' own quality claim (GPTQ output
error below 0.8 x round-to-nearest with the same ladder on correlated data).
"""
import itertools

import numpy as np
import pytest

import oracle
from oracle import q4tp as oq

F32 = np.float32


def pack(h):
    n = h.shape[0]
    return np.concatenate([h[r, r:] for r in range(n)]).astype(np.float32)


def corr_problem(rows, n, t, seed, loud=(5,), dead=()):
    """Correlated activations (4 latent factors + noise, one loud channel):
    the setting of the pages' GPTQ-vs-RTN test, drawn with numpy here."""
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
    tab, lost = oracle.ladder(wdz)
    hw = np.diag(oracle.unpack_upper(hp, n)).astype(F32)
    return u, dead, tab, lost, hw, lam


# ---------------------------------------------------------------- ladder

def test_ladder_powers_of_two():
    # Group absmax 7 * 2^k gives x_g = 2^k exactly: lo = min k, and the top
    # rung reaches max k up to the f16 rounding of step.
    ks = [-6, -3, -1, -4]
    row = np.zeros(32 * len(ks), dtype=F32)
    for g, k in enumerate(ks):
        row[g * 32 + 3] = -7.0 * 2.0 ** k
        row[g * 32 + 9] = 0.5 * 2.0 ** k
    tab, lost = oracle.ladder(row[None, :])
    assert lost[0, 0] == -6.0
    want_step = float(np.float16(5.0 / 31.0))
    assert lost[0, 1] == F32(want_step)
    assert tab[0, 0] == F32(2.0 ** -6)
    assert np.all(np.diff(tab[0]) > 0)
    assert abs(np.log2(tab[0, 31]) - (-6 + 31 * want_step)) < 1e-6
    assert abs(np.log2(tab[0, 31]) - (-1)) < 31 * 2.0 ** -13


def test_ladder_degenerate_rows():
    w = np.zeros((3, 64), dtype=F32)
    w[1, 5] = 3.5  # one non-zero group: a single x -> step 0
    w[2, :] = 0.7  # two groups with the same absmax -> step 0
    tab, lost = oracle.ladder(w)
    assert np.all(tab[0] == 0) and np.all(lost[0] == 0)
    assert lost[1, 1] == 0 and np.all(tab[1] == tab[1, 0])
    assert tab[1, 0] == F32(2.0 ** float(np.float16(np.log2(0.5))))
    assert lost[2, 1] == 0


# ---------------------------------------------------------------- nominal

def test_nominal_rounds_half_away():
    # lo = 0, step = 1: t = log2(amax / 7) exactly for amax = 7 * 2^t.
    lo = np.zeros(5, dtype=F32)
    st = np.ones(5, dtype=F32)
    amax = F32(7.0) * np.array([2.0 ** 2.5, 2.0 ** 3.0, 2.0 ** -0.5, 2.0 ** 40, 2.0 ** 0.49], dtype=F32)
    nom = oq.nominal_rung(amax, lo, st)
    # 2^2.5 is not exact in f32; its log2 lands within an ulp of 2.5.
    t = np.log2(np.float64(amax) / 7.0)
    assert nom[1] == 3 and nom[2] == 0 and nom[3] == 31 and nom[4] == 0
    assert nom[0] in (2, 3) and abs(nom[0] - t[0]) <= 0.5 + 1e-6
    # An exact tie at .5 goes away from zero: amax/7 = 2^0.5 is not exact,
    # so build it with step 2: t = log2(x)/2 = 0.5 for x = 2.
    nom2 = oq.nominal_rung(np.array([14.0], dtype=F32), np.zeros(1, F32), np.full(1, 2.0, F32))
    assert nom2[0] == 1
    assert oq.nominal_rung(np.zeros(1, F32), lo[:1], st[:1])[0] == 0
    assert oq.nominal_rung(np.ones(1, F32), lo[:1], np.zeros(1, F32))[0] == 0


def test_nominal_matches_log_within_half():
    rng = np.random.default_rng(0)
    amax = np.exp(rng.uniform(-8, 2, 2000)).astype(F32)
    lo = F32(-7.25)
    st = F32(0.0625)
    nom = oq.nominal_rung(amax, np.full(2000, lo), np.full(2000, st))
    t = (np.log2(np.float64(amax) / 7) - lo) / st
    inside = (t > -0.5 + 1e-4) & (t < 31.5 - 1e-4)
    assert np.all(np.abs(nom[inside] - t[inside]) <= 0.5 + 1e-4)
    assert np.all(nom[t < -0.5 - 1e-4] == 0)
    assert np.all(nom[t > 31.5 + 1e-4] == 31)


# ---------------------------------------------------------------- codes

def test_codes_minimise_weighted_error_bruteforce():
    # For a fixed scale the weighted error is separable, so the best code
    # vector over all 16^4 candidates must equal clamp(rne(w/s), -8, 7).
    rng = np.random.default_rng(1)
    s = F32(0.013)
    hw = rng.uniform(0.1, 3, 4)
    grid = np.array(list(itertools.product(range(-8, 8), repeat=4)), dtype=np.float64)
    for _ in range(30):
        w = (rng.uniform(-0.13, 0.13, 4)).astype(F32)
        err = (((w[None, :] - grid * s) ** 2) * hw).sum(axis=1)
        best = grid[np.argmin(err)]
        q = np.clip(np.rint(w / s), -8, 7)
        assert np.array_equal(best, q)


def test_group_rung_is_window_argmin():
    # The chosen rung's weighted error is <= every rung in the window
    # nominal-2..nominal+1 (strictly below the lower-indexed ones).
    rng = np.random.default_rng(2)
    rows = 200
    tile = (rng.standard_normal((rows, 32)) * 0.02).astype(F32)
    hw = rng.uniform(0.01, 5, 32).astype(F32)
    tab, lost = oracle.ladder(np.tile(tile, (1, 8)) * rng.uniform(0.5, 2, (1, 256)).astype(F32))
    u = np.eye(32, dtype=F32)
    rung, q, e = oracle.group_q4tp(tile, hw, tab, lost, u)
    amax = np.abs(tile).max(axis=1)
    nom = oq.nominal_rung(amax, lost[:, 0], lost[:, 1])
    for r in range(rows):
        errs = {}
        for c in range(max(nom[r] - 2, 0), min(nom[r] + 1, 31) + 1):
            s = np.float64(tab[r, c])
            qq = np.clip(np.rint(tile[r].astype(np.float64) / s), -8, 7)
            errs[c] = float(((tile[r] - qq * s) ** 2 * hw).sum())
        c0 = rung[r]
        assert c0 in errs
        for c, v in errs.items():
            if c < c0:
                assert errs[c0] < v * (1 + 1e-5)
            else:
                assert errs[c0] <= v * (1 + 1e-5)


def test_zero_weights_pick_lowest_in_window():
    # hw = 0 makes every candidate's error 0: the strict '<' keeps the first
    # (lowest) rung of the window.
    rng = np.random.default_rng(3)
    tile = (rng.standard_normal((50, 32)) * 0.02).astype(F32)
    tab, lost = oracle.ladder(np.tile(tile, (1, 4)) * rng.uniform(0.3, 3, (1, 128)).astype(F32))
    rung, _, _ = oracle.group_q4tp(tile, np.zeros(32, F32), tab, lost, np.eye(32, dtype=F32))
    nom = oq.nominal_rung(np.abs(tile).max(axis=1), lost[:, 0], lost[:, 1])
    assert np.array_equal(rung, np.maximum(nom - 2, 0))


def test_nibble_plane_layout():
    rng = np.random.default_rng(4)
    rows, n = 3, 64
    q = rng.integers(-8, 8, (rows, n))
    plane = np.zeros(rows * n // 2, dtype=np.uint8)
    for r in range(rows):
        for c in range(n):
            g, j = divmod(c, 32)
            b = (r * (n // 32) + g) * 16 + j // 2
            nib = q[r, c] + 8
            plane[b] |= nib if j % 2 == 0 else nib << 4
    assert np.array_equal(oracle.nibbles_to_codes(plane, rows, n), q)


# ---------------------------------------------------------------- sweep

def test_identity_w0_minus_q_equals_e_u():
    _, h, w = corr_problem(16, 96, 300, 5, dead=(40,))
    u, dead, tab, lost, hw, lam = prep(w, h)
    wdz = w.copy()
    wdz[:, dead] = 0
    # f64 recursion: exact up to f64 rounding.
    rung, q, sc, e = oracle.sweep_q4tp_f64(w, u, hw, tab, lost, dead)
    qw = q.astype(np.float64) * np.repeat(sc, 32, axis=1)
    np.testing.assert_allclose(wdz - qw, e @ u, rtol=0, atol=1e-12)
    # ||E||^2 = tr((W0-Q) H_d (W0-Q)^T), since U H_d U^T = I.
    dd, hf, base = oracle.fold_damping(pack(h.astype(F32)), 96)
    hd = hf + lam * base * np.eye(96)
    lhs = oracle.output_error(wdz, qw, hd)
    assert lhs == pytest.approx(float((e * e).sum()), rel=1e-10)
    # The f32 sweep obeys the same identity up to f32 rounding.
    r32 = oracle.sweep_q4tp(w, u.astype(F32), hw, tab, lost, dead)
    q32 = oracle.dequant_q4tp(r32["q"], r32["scale"]).astype(np.float64)
    gap = (wdz - q32) - r32["e"].astype(np.float64) @ u
    assert np.abs(gap).max() < 2e-5 * np.abs(w).max()
    assert (r32["q"] == q).mean() > 0.99


def test_sweep_matches_textbook_obs_loop():
    # One rung only (step = 0 -> every rung equal), so codes depend only on
    # the update rule; the textbook OBS loop uses explicit inverses of the
    # trailing blocks of H_d: after rounding column j, the remaining weights
    # move by -(w_j - q_j s) * inv(H_d[j:, j:])[0, 1:] / inv(H_d[j:, j:])[0, 0].
    n, rows = 32, 6
    _, h, w = corr_problem(rows, n, 200, 6)
    u, dead, _, _, hw, lam = prep(w, h)
    dd, hf, base = oracle.fold_damping(pack(h.astype(F32)), n)
    hd = hf + lam * base * np.eye(n)
    s = 0.04
    tab = np.full((rows, 32), s, dtype=np.float64)
    lost = np.zeros((rows, 2))
    rung, q, sc, e = oracle.sweep_q4tp_f64(w, u, hw, tab, lost)
    for r in range(rows):
        wt = w[r].astype(np.float64).copy()
        for j in range(n):
            qj = np.clip(np.rint(wt[j] / s), -8, 7)
            assert qj == q[r, j]
            if j + 1 < n:
                t = np.linalg.inv(hd[j:, j:])
                wt[j + 1 :] -= (wt[j] - qj * s) * t[0, 1:] / t[0, 0]


def test_diagonal_h_is_groupwise_rtn():
    # Diagonal H: U is diagonal, no residual reaches another column, so the
    # sweep equals the group rule applied to the untouched tiles.
    rng = np.random.default_rng(7)
    n, rows = 128, 20
    h = np.diag(rng.uniform(0.5, 4, n)).astype(F32)
    w = (rng.standard_normal((rows, n)) * 0.02).astype(F32)
    u, dead, tab, lost, hw, _ = prep(w, h)
    res = oracle.sweep_q4tp(w, u.astype(F32), hw, tab, lost, dead)
    for g in range(n // 32):
        c0 = g * 32
        rung, q, e = oracle.group_q4tp(w[:, c0:c0 + 32], hw[c0:c0 + 32], tab, lost,
                                       u.astype(F32)[c0:c0 + 32, c0:c0 + 32])
        assert np.array_equal(rung, res["rung"][:, g])
        assert np.array_equal(q, res["q"][:, c0:c0 + 32])


def test_group_kernel_reproduces_sweep_tiles():
    # The per-group rule fed each group's starting tile reproduces the
    # sweep's codes and residuals bit for bit (the in-group feedback is the
    # same f32 sequence as the full-row update).
    _, h, w = corr_problem(24, 128, 400, 8, dead=(70,))
    u, dead, tab, lost, hw, _ = prep(w, h)
    u32 = u.astype(F32)
    res = oracle.sweep_q4tp(w, u32, hw, tab, lost, dead, record=True)
    for g in range(4):
        c0 = g * 32
        rung, q, e = oracle.group_q4tp(res["tiles"][g], hw[c0:c0 + 32], tab, lost, u32[c0:c0 + 32, c0:c0 + 32])
        assert np.array_equal(rung, res["rung"][:, g])
        assert np.array_equal(q, res["q"][:, c0:c0 + 32])
        assert np.array_equal(e.view(np.uint32), res["e"][:, c0:c0 + 32].view(np.uint32))


def test_dead_group_is_independent():
    # A whole dead group (32 channels that never fire) is decoupled: the
    # other groups' codes equal those of the problem without it, once the
    # damping is matched (dead channels count 1 in mean(diag)).
    rows, n = 10, 96
    x, h, w = corr_problem(rows, n, 300, 9, dead=tuple(range(32, 64)))
    u, dead, tab, lost, hw, lam = prep(w, h)
    res = oracle.sweep_q4tp(w, u.astype(F32), hw, tab, lost, dead)
    keep = np.r_[0:32, 64:96]
    h2 = h[np.ix_(keep, keep)]
    mean_full = (np.trace(h) + 32) / n
    lam2 = lam * mean_full / (np.trace(h2) / 64)
    u2, _, _, _ = oracle.fold(pack(h2.astype(F32)), 64, lam2)
    res2 = oracle.sweep_q4tp(w[:, keep], u2.astype(F32), hw[keep], tab, lost)
    assert np.all(res["q"][:, 32:64] == 0)
    assert np.all(res["e"][:, 32:64] == 0)
    assert (res["q"][:, keep] == res2["q"]).mean() > 0.999


def test_gptq_beats_rtn_on_output_error():
    # The pages' claim: on correlated inputs the GPTQ output error is below
    # 0.8 x the round-to-nearest error with the same ladder.
    rows, n, t = 24, 96, 400
    x, h, w = corr_problem(rows, n, t, 12345)
    u, dead, tab, lost, hw, _ = prep(w, h)
    g = oracle.sweep_q4tp(w, u.astype(F32), hw, tab, lost, dead)
    r = oracle.sweep_q4tp(w, np.eye(n, dtype=F32), hw, tab, lost, dead)
    eg = oracle.output_error(w, oracle.dequant_q4tp(g["q"], g["scale"]), h)
    er = oracle.output_error(w, oracle.dequant_q4tp(r["q"], r["scale"]), h)
    assert eg < 0.8 * er
