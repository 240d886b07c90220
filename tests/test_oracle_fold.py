"""Pins for the oracle fold (CPU only).

The oracle computes the fold the host way (``cortiq-cli src/gptq.rs``,
``gptq_fold_operator_par``: chol(H_d), its inverse, H_d^-1, chol again).
Each test here checks it against something that is not that route:
closed forms, exact algebra, the OBS identity through an LU inverse of
trailing blocks, and invariants.
"""
import numpy as np
import pytest
import sympy

import oracle
import synth


def pack(h):
    n = h.shape[0]
    return np.concatenate([h[r, r:] for r in range(n)]).astype(np.float32)


def spd(n, seed, t=None, scales=None, dead=()):
    rng = np.random.default_rng(seed)
    t = t or 3 * n
    x = rng.standard_normal((n, t))
    if scales is not None:
        x *= np.asarray(scales)[:, None]
    for d in dead:
        x[d] = 0
    return (x @ x.T / t).astype(np.float32)


def test_diagonal_closed_form():
    # Diagonal H: H_d^-1 is diagonal, so U = diag(1/sqrt(h_i + damp)),
    # damp = lambda * mean(diag) (dead diagonal counted as 1).
    h = np.diag([4.0, 0.0, 9.0, 0.25, 1.0]).astype(np.float32)
    lam = 0.01
    u, d, dead, lam_used = oracle.fold(pack(h), 5, lam)
    assert lam_used == lam
    assert list(dead) == [False, True, False, False, False]
    mean = (4 + 1 + 9 + 0.25 + 1) / 5
    damp = lam * mean
    want = np.diag([1 / np.sqrt(4 + damp), 1 / np.sqrt(1 + damp), 1 / np.sqrt(9 + damp),
                    1 / np.sqrt(0.25 + damp), 1 / np.sqrt(1 + damp)])
    np.testing.assert_allclose(u, want, rtol=1e-14, atol=0)
    assert d[1] < 0 and np.all(d[[0, 2, 3, 4]] > 0)
    np.testing.assert_allclose(np.abs(d), np.sqrt(np.array([4, 1, 9, 0.25, 1]) + damp), rtol=1e-15)


def test_two_by_two_exact():
    # H_d = [[a, b], [b, c]]: H_d^-1 = [[c, -b], [-b, a]] / det, and the
    # upper U with U^T U = H_d^-1 is u00 = sqrt(c/det), u01 = -b/sqrt(c det),
    # u11 = 1/sqrt(c) (exact algebra, sympy).
    a, b, c = sympy.Rational(4), sympy.Rational(2), sympy.Rational(3)
    for lam in (0.0, 0.01):
        h = np.array([[4, 2], [2, 3]], dtype=np.float32)
        u, _, _, lam_used = oracle.fold(pack(h), 2, lam)
        assert lam_used == lam
        damp = sympy.Rational(lam).limit_denominator(10**6) * (a + c) / 2
        ad, cd = a + damp, c + damp
        det = ad * cd - b * b
        want = [[sympy.sqrt(cd / det), -b / sympy.sqrt(cd * det)], [0, 1 / sympy.sqrt(cd)]]
        want = np.array([[float(sympy.N(v, 30)) for v in row] for row in want])
        np.testing.assert_allclose(u, want, rtol=1e-14, atol=1e-16)


def test_three_by_three_exact():
    # Exact rational H, lambda = 0: U from sympy's exact inverse and
    # Cholesky of the reversed matrix (H^-1 = U^T U, U upper).
    hi = sympy.Matrix([[6, 2, 1], [2, 5, 2], [1, 2, 4]])
    h = np.array(hi.tolist(), dtype=np.float32)
    u, _, _, _ = oracle.fold(pack(h), 3, 0.0)
    inv = hi.inv()
    # U^T U = inv  <=>  (P U P)(P U P)^T... solve directly: U upper, entries
    # from the trailing-block recursion U[j, j:] = row0(inv(H[j:, j:])) / sqrt(.[0,0]).
    want = sympy.zeros(3, 3)
    for j in range(3):
        t = hi[j:, j:].inv()
        for k in range(j, 3):
            want[j, k] = t[0, k - j] / sympy.sqrt(t[0, 0])
    assert sympy.simplify(want.T * want - inv) == sympy.zeros(3, 3)
    np.testing.assert_allclose(u, np.array(want.evalf(30).tolist(), dtype=np.float64), rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("seed", [0, 1])
def test_obs_rows_via_lu_inverse(seed):
    # Row j of the fold operator is the first row of inv(H_d[j:, j:]) over
    # the square root of its first entry (the OBS step after eliminating
    # columns < j, the fold page's doc comment); checked with an LU inverse.
    n = 24
    rng = np.random.default_rng(seed)
    sc = np.exp(1.5 * rng.standard_normal(n))
    sc[3] *= 100
    h = spd(n, seed, t=2 * n, scales=sc, dead=(7,))
    u, _, dead, lam = oracle.fold(pack(h), n, 0.01)
    dd, hf, base = oracle.fold_damping(pack(h), n)
    hd = hf + lam * base * np.eye(n)
    for j in range(n):
        t = np.linalg.inv(hd[j:, j:])
        np.testing.assert_allclose(u[j, j:], t[0] / np.sqrt(t[0, 0]), rtol=1e-9, atol=1e-12 * np.abs(u).max())
        assert np.all(u[j, :j] == 0)


def test_reconstruction_and_shape():
    cfg = synth.config("tiny", n=192, T=400)
    hp = synth.make_h_packed(cfg).numpy()
    u, d, dead, lam = oracle.fold(hp, cfg.n, 0.01)
    dd, hf, base = oracle.fold_damping(hp, cfg.n)
    hd = hf + lam * base * np.eye(cfg.n)
    assert np.all(np.tril(u, -1) == 0)
    assert np.all(np.diag(u) > 0)
    r = u.T @ u @ hd - np.eye(cfg.n)
    assert np.abs(r).max() < 1e-10
    assert dead.sum() == cfg.n_dead


def test_dead_channel_decoupled():
    n = 16
    h = spd(n, 3, dead=(2, 11))
    u, d, dead, lam = oracle.fold(pack(h), n, 0.05)
    _, _, base = oracle.fold_damping(pack(h), n)
    damp = lam * base
    for k in (2, 11):
        assert dead[k]
        assert abs(u[k, k] - 1 / np.sqrt(1 + damp)) < 1e-14
        row = np.delete(u[k], k)
        col = np.delete(u[:, k], k)
        assert np.all(row == 0) or np.abs(row).max() < 1e-15
        assert np.abs(col).max() < 1e-15
        assert d[k] == -np.sqrt(1 + damp)


def test_scale_invariance():
    # No dead channels: H -> c H scales damp by c, so U -> U / sqrt(c).
    n = 20
    h = spd(n, 5)
    u1, _, _, _ = oracle.fold(pack(h), n, 0.01)
    u2, _, _, _ = oracle.fold(pack(h * np.float32(16.0)), n, 0.01)
    np.testing.assert_allclose(u2, u1 / 4.0, rtol=1e-12, atol=1e-15)


def test_rank_deficient_raises_lambda():
    # Rank n/2 with lambda = 0: the first attempt has a zero pivot, the
    # retry uses 1e-4 (0 -> 1e-4, then x10).
    n = 32
    h = spd(n, 7, t=n // 2)
    u, _, _, lam = oracle.fold(pack(h), n, 0.0)
    assert lam >= 1e-4
    assert lam in (1e-4, 1e-3, 1e-2, 1e-1, 1.0, 10.0) or abs(np.log10(lam) - round(np.log10(lam))) < 1e-9


def test_indefinite_is_not_spd():
    # Eigenvalues 101 and -99: even damp = 10 * mean(diag) = 10 leaves a
    # negative eigenvalue, so every attempt fails.
    h = np.array([[1, 100], [100, 1]], dtype=np.float32)
    with pytest.raises(oracle.NotSPD):
        oracle.fold(pack(h), 2, 0.01)
    # ...while a milder one is repaired by the x10 schedule (0.01 -> 0.1 -> 1).
    h2 = np.array([[1, 1.5], [1.5, 1]], dtype=np.float32)
    u, _, _, lam = oracle.fold(pack(h2), 2, 0.01)
    assert lam == pytest.approx(1.0)


def test_nan_is_not_spd():
    h = spd(8, 1)
    h[2, 5] = h[5, 2] = np.nan
    with pytest.raises(oracle.NotSPD):
        oracle.fold(pack(h), 8, 0.01)


def test_all_dead_is_identity_scaled():
    n = 6
    h = np.zeros((n, n), dtype=np.float32)
    u, d, dead, lam = oracle.fold(pack(h), n, 0.01)
    assert dead.all()
    np.testing.assert_allclose(u, np.eye(n) / np.sqrt(1.01), rtol=1e-15)


def test_equilibrated_reversed_reconstructs_hd():
    n = 40
    rng = np.random.default_rng(2)
    h = spd(n, 2, scales=np.exp(rng.standard_normal(n)), dead=(5,))
    hp = pack(h)
    a_low, d, damp = oracle.equilibrated_reversed(hp, n, 0.01)
    a = a_low + np.tril(a_low, -1).T
    live = d > 0
    # D P A P D equals the damped H on live channels, identity on dead ones.
    b = a[::-1, ::-1] * np.outer(np.abs(d), np.abs(d))
    hd = h.astype(np.float64) + damp * np.eye(n)
    np.testing.assert_allclose(b[np.ix_(live, live)], hd[np.ix_(live, live)], rtol=1e-12, atol=1e-12)
    assert b[5, 5] == pytest.approx(1 + damp)
    # Unit diagonal: d_i^2 = H_ii + damp for live channels, 1 for dead ones.
    np.testing.assert_allclose(np.diag(a), 1.0, rtol=1e-12)
