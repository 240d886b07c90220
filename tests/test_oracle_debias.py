"""Pins for the oracle output debias (CPU only).

The oracle follows the host page's ``q2tp_debias_hessian`` /
``q4tp_debias_hessian``.  The checks come from outside that code: the slope
through explicit activations (H = X^T X) and as a least-squares fit, exact
power-of-two shrinkage moving lo by exactly one, the identity and degenerate
rows, invariance to the scale of H, the debiased slope landing within the
f16 rounding of lo, and the page's claim that the placed 2-bit rule shrinks
the outputs (slope < 1).
"""
import numpy as np
import pytest

import oracle
from oracle import debias as od
from oracle import q2tp as o2

F32 = np.float32


def pack(h):
    n = h.shape[0]
    return np.concatenate([h[r, r:] for r in range(n)]).astype(np.float32)


def q2_problem(rows, n, t, seed):
    rng = np.random.default_rng(seed)
    lat = rng.uniform(-0.5, 0.5, (t, 4))
    mix = rng.uniform(-0.5, 0.5, (4, n))
    x = (lat @ mix + 0.2 * rng.uniform(-0.5, 0.5, (t, n))).astype(F32)
    h = x.astype(np.float64).T @ x.astype(np.float64)
    w = rng.uniform(-0.5, 0.5, (rows, n)).astype(F32)
    u, d, dead, lam = oracle.fold(pack(h.astype(F32)), n, 0.01)
    hw = np.diag(h).astype(F32)
    tab, lost, _ = o2.ladder_q2tp(w, hw)
    res = o2.sweep_q2tp(w, u.astype(F32), hw, tab)
    return x, h, w, tab, lost, res


def test_slope_through_activations_and_least_squares():
    x, h, w, tab, lost, res = q2_problem(12, 64, 300, 0)
    what = od.dequant(res["q"], res["rung"], tab, True)
    num, den = od.slopes(w, what, h)
    xd = x.astype(np.float64)
    for r in range(12):
        yw = xd @ w[r].astype(np.float64)
        yq = xd @ what[r]
        assert num[r] == pytest.approx(yq @ yw, rel=1e-10)
        assert den[r] == pytest.approx(yw @ yw, rel=1e-10)
        beta = np.linalg.lstsq(yw[:, None], yq, rcond=None)[0][0]
        assert num[r] / den[r] == pytest.approx(beta, rel=1e-9)


def test_placed_rule_shrinks_outputs():
    # The page: MSE-optimal 2-bit rounding shrinks the outputs (slope below
    # 1; with GPTQ's error feedback a single row can land above 1, so the
    # check is on the mean over rows).
    x, h, w, tab, lost, res = q2_problem(48, 96, 400, 1)
    out = od.debias(w, h, res["q"], res["rung"], tab, lost, True)
    b = out["num"] / out["den"]
    assert b.mean() < 0.99 and np.all(b > 0.5)


@pytest.mark.parametrize("two_bit", [True, False])
def test_half_scale_moves_lo_by_one(two_bit):
    # W^ = W / 2 exactly (W built on the levels of twice the ladder): the
    # slope is 1/2, lo rises by exactly 1 and every rung doubles.
    rng = np.random.default_rng(2)
    rows, n = 5, 96
    lo, st = -5.0, 0.25
    c = np.arange(32, dtype=np.float64)
    tab = np.zeros((rows, 32), dtype=F32)
    if two_bit:
        tab[:, 1:] = np.exp2(lo + (c[1:] - 1) * st).astype(F32)
        q = rng.integers(0, 4, (rows, n))
        rungs = rng.integers(1, 32, (rows, n // 32))
    else:
        tab[:] = np.exp2(lo + c * st).astype(F32)
        q = rng.integers(-8, 8, (rows, n))
        rungs = rng.integers(0, 32, (rows, n // 32))
    lost = np.tile(np.array([lo, st], dtype=F32), (rows, 1))
    what = od.dequant(q, rungs, tab, two_bit)
    w = (2.0 * what).astype(F32)
    a = rng.standard_normal((n, n))
    h = a @ a.T + n * np.eye(n)
    out = od.debias(w, h, q, rungs, tab, lost, two_bit)
    assert np.all(out["lost"][:, 0] == lo + 1) and np.all(out["lost"][:, 1] == st)
    np.testing.assert_array_equal(out["tab"], 2 * tab)
    np.testing.assert_array_equal(out["scales"], 2 * tab[np.arange(rows)[:, None], rungs])


def test_identity_and_degenerate_rows():
    x, h, w, tab, lost, res = q2_problem(6, 64, 200, 3)
    q, rungs = res["q"].copy(), res["rung"].copy()
    what = od.dequant(q, rungs, tab, True)
    w2 = what.astype(F32)            # row 0..: W^ = W exactly -> slope 1
    w2[1] = -w2[1]                   # slope -1: kept
    w2[2] = 0.0                      # den = 0: kept
    tab2 = tab.copy()
    tab2[3] = 0.0                    # a row without a ladder: stays zero
    out = od.debias(w2, h, q, rungs, tab2, lost, True)
    assert out["lost"][0, 0] == lost[0, 0] and np.array_equal(out["tab"][0], tab2[0])
    for r in (1, 2):
        assert np.array_equal(out["lost"][r], lost[r]) and np.array_equal(out["tab"][r], tab2[r])
    assert np.all(out["tab"][3] == 0)


def test_h_scale_invariance_and_debiased_slope():
    x, h, w, tab, lost, res = q2_problem(16, 96, 300, 4)
    out = od.debias(w, h, res["q"], res["rung"], tab, lost, True)
    out2 = od.debias(w, 37.5 * h, res["q"], res["rung"], tab, lost, True)
    np.testing.assert_array_equal(out["lost"], out2["lost"])
    # Re-measured slope with the new scales: within the f16 rounding of lo'.
    what = od.dequant(res["q"], res["rung"], out["tab"], True)
    num, den = od.slopes(w, what, h)
    for r in range(16):
        lo2 = np.float16(out["lost"][r, 0])
        half_ulp = float(np.spacing(np.abs(lo2))) / 2
        assert abs(np.log2(num[r] / den[r])) <= half_ulp * (1 + 1e-6) + 1e-12
