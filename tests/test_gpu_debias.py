"""Output debias on the device against the oracle.

Inputs come from the oracle (its fold, ladder and sweep give the codes,
rungs, ladders and scales that both sides debias).  Tolerances: num and den
within 1e-5 (relative; W H in 3xTF32 with f32 accumulation against f64),
lo' equal on >= 99.5 % of rows (f16 rounding of lo + log2(den/num)), and
the rebuilt rungs and scales bit-exact wherever lo' agrees.
"""
import numpy as np
import pytest

import oracle
import synth
from oracle import debias as od

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F32 = np.float32
DEV = "cuda"


def np_(t):
    return t.detach().cpu().numpy()


def small_problem(n, rows, seed=0, sigma=1.5, n_out=2, n_dead=2):
    cfg = synth.Config(f"n{n}", n, rows, 4 * n, 0.02, sigma, n_out, n_dead, 0.01, seed)
    hp, w = synth.make_problem(cfg, "cpu")
    return cfg, hp.numpy(), w.numpy()


def q2_plane(q):
    rows, n = q.shape
    q = q.astype(np.uint8).reshape(rows, n // 4, 4)
    return (q[..., 0] | (q[..., 1] << 2) | (q[..., 2] << 4) | (q[..., 3] << 6)).reshape(-1)


def q4_plane(q):
    rows, n = q.shape
    nib = (q.astype(np.int16) + 8).astype(np.uint8).reshape(rows, n // 2, 2)
    return (nib[..., 0] | (nib[..., 1] << 4)).reshape(-1)


def oracle_quantized(hp, w, n, bits, uo=None, dead=None):
    if uo is None:
        uo, do, dead, lam = oracle.fold(hp, n, 0.01)
    hw = oracle.unpack_upper(hp, n).diagonal().astype(F32)
    wz = w.copy()
    wz[:, dead] = 0
    if bits == 2:
        tab, lost, _ = oracle.ladder_q2tp(wz, hw)
        res = oracle.sweep_q2tp(w, uo.astype(F32), hw, tab, dead)
        plane = q2_plane(res["q"])
    else:
        tab, lost = oracle.ladder(wz)
        res = oracle.sweep_q4tp(w, uo.astype(F32), hw, tab, lost, dead)
        plane = q4_plane(res["q"])
    return res, tab, lost, plane


def run_and_compare(hp, w, n, bits, res, tab, lost, plane):
    from gptq_post_weight_gb300 import _lib

    rows = w.shape[0]
    tab_d = torch.from_numpy(tab.copy()).to(DEV)
    lost_d = torch.from_numpy(lost.copy()).to(DEV)
    sc_d = torch.from_numpy(np.ascontiguousarray(res["scale"], dtype=F32).reshape(-1)).to(DEV)
    rung_d = torch.from_numpy(res["rung"].astype(np.uint8).reshape(-1)).to(DEV)
    nd = _lib.debias(bits, torch.from_numpy(w).to(DEV), torch.from_numpy(hp).to(DEV),
                     torch.from_numpy(plane).to(DEV), rung_d, tab_d, lost_d, sc_d, want_num_den=True)
    h = oracle.unpack_upper(hp, n)
    want = od.debias(w, h, res["q"], res["rung"], tab, lost, two_bit=(bits == 2))
    nd = np_(nd)
    np.testing.assert_allclose(nd[:, 0], want["num"], rtol=1e-5)
    np.testing.assert_allclose(nd[:, 1], want["den"], rtol=1e-5)
    lost_g, tab_g, sc_g = np_(lost_d), np_(tab_d), np_(sc_d).reshape(rows, -1)
    same = (lost_g == want["lost"]).all(axis=1)
    assert same.mean() >= 0.995, np.nonzero(~same)
    assert np.array_equal(tab_g[same].view(np.uint32), want["tab"][same].view(np.uint32))
    assert np.array_equal(sc_g[same].view(np.uint32), want["scales"][same].view(np.uint32))
    return nd, want


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("n,rows", [(256, 64), (416, 45), (1024, 300)])
def test_debias_matches_oracle(lib, bits, n, rows):
    cfg, hp, w = small_problem(n, rows, seed=n + bits)
    res, tab, lost, plane = oracle_quantized(hp, w, n, bits)
    nd, want = run_and_compare(hp, w, n, bits, res, tab, lost, plane)
    if bits == 2:
        b = want["num"] / want["den"]
        assert b.mean() < 1.0  # the placed rule shrinks the outputs


def test_debias_exact_halving(lib):
    # W = 2 W^ exactly: the slope is 1/2, lo rises by exactly 1 and every
    # rung and scale doubles, bit for bit.
    from gptq_post_weight_gb300 import _lib

    rng = np.random.default_rng(3)
    rows, n = 70, 256
    lo, st = -6.0, 0.125
    c = np.arange(32, dtype=np.float64)
    tab = np.zeros((rows, 32), dtype=F32)
    tab[:, 1:] = np.exp2(lo + (c[1:] - 1) * st).astype(F32)
    lost = np.tile(np.array([lo, st], dtype=F32), (rows, 1))
    q = rng.integers(0, 4, (rows, n))
    rungs = rng.integers(1, 32, (rows, n // 32))
    scales = tab[np.arange(rows)[:, None], rungs]
    w = (2.0 * od.dequant(q, rungs, tab, True)).astype(F32)
    x = rng.standard_normal((3 * n, n)).astype(F32)
    h = (x.astype(np.float64).T @ x.astype(np.float64)).astype(F32)
    hp = np.concatenate([h[r, r:] for r in range(n)]).astype(F32)
    tab_d = torch.from_numpy(tab.copy()).to(DEV)
    lost_d = torch.from_numpy(lost.copy()).to(DEV)
    sc_d = torch.from_numpy(scales.reshape(-1).copy()).to(DEV)
    _lib.debias(2, torch.from_numpy(w).to(DEV), torch.from_numpy(hp).to(DEV),
                torch.from_numpy(q2_plane(q)).to(DEV), torch.from_numpy(rungs.astype(np.uint8).reshape(-1)).to(DEV),
                tab_d, lost_d, sc_d)
    assert np.all(np_(lost_d)[:, 0] == lo + 1) and np.all(np_(lost_d)[:, 1] == st)
    np.testing.assert_array_equal(np_(tab_d), 2 * tab)
    np.testing.assert_array_equal(np_(sc_d).reshape(rows, -1), 2 * scales)


@pytest.mark.slow
def test_full_size_debias(lib, oracle_folds):
    """n = 17408: the debias of 16 sampled rows (the oracle's q2tp codes of
    those rows) through the full-width W H."""
    cfg = synth.config("n17408")
    hpd, wd = synth.make_problem(cfg, DEV)
    hp = np_(hpd)
    w = np_(wd)
    del hpd, wd
    uo, do, dead, lamo = oracle_folds(hp, cfg.n, cfg.lam, key=(cfg.name, cfg.seed))
    rng = np.random.default_rng(2)
    rows_idx = np.sort(rng.choice(cfg.rows, 16, replace=False))
    ws = np.ascontiguousarray(w[rows_idx])
    res, tab, lost, plane = oracle_quantized(hp, ws, cfg.n, 2, uo=uo, dead=dead)
    nd, want = run_and_compare(hp, ws, cfg.n, 2, res, tab, lost, plane)
    print("full-size debias slopes:", np.round(want["num"] / want["den"], 4))
