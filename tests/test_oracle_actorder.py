"""Pins for the oracle act-order q4tp (CPU only): the permutation against a
brute-force sort with Rust total_cmp semantics, the permuted fold against the
OBS identity in permuted order, the diagonal-H closed form (codes = static
round-to-nearest), the recursion identity W0 - Q = E U in permuted order, and
the pages' claims (the loud channel goes first; GPTQ beats round-to-nearest).
"""
import functools

import numpy as np
import pytest

import oracle

F32 = np.float32


def pack(h):
    n = h.shape[0]
    return np.concatenate([h[r, r:] for r in range(n)]).astype(F32)


def test_perm_matches_bruteforce_total_order():
    vals = np.array([1.0, 3.0, -0.0, 0.0, 3.0, np.nan, -2.0, 5.0, 1.0, np.inf], dtype=F32)

    def rust_total_cmp(a, b):
        # IEEE 754 totalOrder: -NaN < -inf < ... < -0 < +0 < ... < +inf < +NaN
        def key(x):
            bits = np.array([x], dtype=F32).view(np.int32)[0]
            return int(bits) if bits >= 0 else -(int(bits) & 0x7FFFFFFF) - 1
        return (key(a) > key(b)) - (key(a) < key(b))

    idx = list(range(len(vals)))
    idx.sort(key=functools.cmp_to_key(lambda a, b: rust_total_cmp(vals[b], vals[a]) or (a - b)))
    assert list(oracle.act_order_perm(vals)) == idx
    # NaN (positive) first, then +inf, 5, the tie 3 @ 1 before 3 @ 4, ...
    assert idx[:4] == [5, 9, 7, 1]
    assert idx.index(3) < idx.index(2)  # +0 before -0 in descending order


def test_permuted_fold_obs_rows():
    rng = np.random.default_rng(3)
    n = 20
    x = rng.standard_normal((n, 60)) * np.exp(rng.standard_normal((n, 1)))
    h = (x @ x.T / 60).astype(F32)
    hd32 = np.diag(h).astype(F32)
    perm = oracle.act_order_perm(hd32)
    assert np.all(np.diff(hd32[perm]) <= 0)
    up, _, _, lam = oracle.fold(oracle.permute_packed(pack(h), n, perm), n, 0.01)
    hp = h.astype(np.float64)[np.ix_(perm, perm)]
    hdmp = hp + lam * np.trace(hp) / n * np.eye(n)
    for j in range(n):
        t = np.linalg.inv(hdmp[j:, j:])
        np.testing.assert_allclose(up[j, j:], t[0] / np.sqrt(t[0, 0]), rtol=1e-9, atol=1e-12)


def test_diagonal_h_is_static_rtn():
    # Diagonal H: no residual reaches another channel, so every code is
    # clamp(rne(w / s)) with the static scale of its group.
    rng = np.random.default_rng(4)
    n, rows = 96, 10
    h = np.diag(rng.uniform(0.5, 4, n)).astype(F32)
    w = (rng.standard_normal((rows, n)) * 0.02).astype(F32)
    tab, lost = oracle.ladder(w)
    rungs = oracle.converter_rungs(w, tab, lost)
    perm = oracle.act_order_perm(np.diag(h).astype(F32))
    up = oracle.fold(oracle.permute_packed(pack(h), n, perm), n, 0.01)[0].astype(F32)
    res = oracle.sweep_q4tp_act_order(w, up, None, perm, tab, rungs)
    s = np.repeat(tab[np.arange(rows)[:, None], rungs], 32, axis=1)
    want = np.clip(np.rint(w / s), -8, 7)
    assert np.array_equal(res["q"], want.astype(np.int8))


def test_identity_and_loud_channel_first():
    rng = np.random.default_rng(12345)
    rows, n, t = 24, 96, 400
    lat = rng.uniform(-0.5, 0.5, (t, 4))
    mix = rng.uniform(-0.5, 0.5, (4, n))
    x = lat @ mix + 0.2 * rng.uniform(-0.5, 0.5, (t, n))
    x[:, 5] *= 8.0
    h = x.T @ x
    w = rng.uniform(-0.5, 0.5, (rows, n)).astype(F32)
    hd32 = np.diag(h).astype(F32)
    perm = oracle.act_order_perm(hd32)
    assert perm[0] == 5  # the loud channel goes first (the pages' test)
    tab, lost = oracle.ladder(w)
    rungs = oracle.converter_rungs(w, tab, lost)
    up = oracle.fold(oracle.permute_packed(pack(h.astype(F32)), n, perm), n, 0.01)[0]
    res = oracle.sweep_q4tp_act_order(w, up.astype(F32), None, perm, tab, rungs)
    qw = res["q"].astype(np.float64) * np.repeat(res["scale"], 32, axis=1)
    # W0 - Q = E U in permuted order (f32 recursion, to round-off)
    gap = (w.astype(np.float64) - qw)[:, perm] - res["e"].astype(np.float64) @ up
    assert np.abs(gap).max() < 2e-5
    # GPTQ with act order beats the converter's round-to-nearest encoding.
    q_rtn = np.clip(np.rint(w / np.repeat(res["scale"], 32, axis=1)), -8, 7)
    e_ao = oracle.output_error(w, qw, h)
    e_rtn = oracle.output_error(w, q_rtn * np.repeat(res["scale"], 32, axis=1), h)
    assert e_ao < 0.8 * e_rtn


def test_static_rungs_are_unit_weight_window_argmin():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((40, 64)) * 0.03).astype(F32)
    tab, lost = oracle.ladder(w)
    rungs = oracle.converter_rungs(w, tab, lost)
    from oracle import q4tp as oq
    for r in range(40):
        for g in range(2):
            tile = w[r, 32 * g:32 * g + 32]
            nom = oq.nominal_rung(np.abs(tile).max()[None], lost[r:r + 1, 0], lost[r:r + 1, 1])[0]
            errs = {}
            for c in range(max(nom - 2, 0), min(nom + 1, 31) + 1):
                s = np.float64(tab[r, c])
                q = np.clip(np.rint(tile / s), -8, 7)
                errs[c] = ((tile - q * s) ** 2).sum()
            best = min(errs, key=lambda c: (errs[c], c))
            assert rungs[r, g] == best or abs(errs[rungs[r, g]] - errs[best]) <= 1e-6 * errs[best]
