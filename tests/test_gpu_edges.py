"""Small, ragged and degenerate shapes through the device sweeps and the
debias, against the oracle (the oracle's own U and ladders go to both sides).

* n = 32 (one group): the device rule is the oracle's rule on the same
  tile, so codes, rungs and scales are bit-exact;
* wider ragged shapes (a partial last block, rows not a multiple of the
  40-row tile, over 400 rows so that the bar is measurable): the later
  columns differ from the oracle only by the f32 summation order of the
  residual updates, so the end-to-end bar applies: >= 99.9 % of codes
  agree and the output error is within 1 %;
* all-zero rows: rung 0, every code at the zero level (q4tp nibble 8, q2tp
  code 0 with scale 0), and the debias leaves them alone.
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


def problem(n, rows, seed):
    cfg = synth.Config(f"e{n}", n, rows, 4 * n, 0.02, 1.5, 1, 1, 0.01, seed)
    hp, w = synth.make_problem(cfg, "cpu")
    hp, w = hp.numpy(), w.numpy()
    uo, do, dead, lam = oracle.fold(hp, n, 0.01)
    hw = oracle.unpack_upper(hp, n).diagonal().astype(F32)
    wz = w.copy()
    wz[:, dead] = 0
    return hp, w, wz, uo.astype(F32), hw, dead


def run_q4(wz, u, hw, dead):
    from gptq_post_weight_gb300 import _lib

    rows, n = wz.shape
    tab, lost = oracle.ladder(wz)
    res = oracle.sweep_q4tp(wz, u, hw, tab, lost, dead)
    nib, rungs, scales = _lib.q4tp_sweep(torch.from_numpy(wz.copy()).to(DEV), torch.from_numpy(u).to(DEV),
                                         torch.from_numpy(hw).to(DEV), torch.from_numpy(tab).to(DEV),
                                         torch.from_numpy(lost).to(DEV))
    q = oracle.nibbles_to_codes(np_(nib), rows, n)
    return res, q, np_(rungs).reshape(rows, -1), np_(scales).reshape(rows, -1), tab


def run_q2(wz, u, hw, dead):
    from gptq_post_weight_gb300 import _lib

    rows, n = wz.shape
    tab, lost, _ = oracle.ladder_q2tp(wz, hw)
    res = oracle.sweep_q2tp(wz, u, hw, tab, dead)
    codes, rungs, scales = _lib.q2tp_sweep(torch.from_numpy(wz.copy()).to(DEV), torch.from_numpy(u).to(DEV),
                                           torch.from_numpy(hw).to(DEV), torch.from_numpy(tab).to(DEV))
    q = oracle.plane_to_codes(np_(codes), rows, n)
    return res, q, np_(rungs).reshape(rows, -1), np_(scales).reshape(rows, -1), tab


@pytest.mark.parametrize("rows", [1, 45])
def test_single_group_bit_exact(lib, rows):
    hp, w, wz, u, hw, dead = problem(32, rows, 1 + rows)
    for run in (run_q4, run_q2):
        res, q, rungs, scales, _ = run(wz, u, hw, dead)
        assert np.array_equal(q, res["q"].astype(q.dtype))
        assert np.array_equal(rungs.astype(np.int64), res["rung"])
        assert np.array_equal(scales.view(np.uint32), res["scale"].view(np.uint32))


@pytest.mark.parametrize("n,rows", [(64, 403), (160, 441), (288, 481), (96, 440), (416, 3)])
def test_ragged_shapes(lib, n, rows):
    hp, w, wz, u, hw, dead = problem(n, rows, n + rows)
    h = oracle.unpack_upper(hp, n)
    for run, deq in ((run_q4, oracle.dequant_q4tp), (run_q2, oracle.dequant_q2tp)):
        res, q, rungs, scales, _ = run(wz, u, hw, dead)
        agree = (q == res["q"].astype(q.dtype)).mean()
        assert agree >= 0.999, (run.__name__, agree)
        e_dev = oracle.output_error(wz, deq(q, scales), h)
        e_or = oracle.output_error(wz, deq(res["q"], res["scale"]), h)
        assert abs(e_dev - e_or) <= 0.01 * e_or, (run.__name__, e_dev, e_or)


def test_zero_rows(lib):
    from gptq_post_weight_gb300 import _lib

    n, rows = 96, 50
    hp, w, wz, u, hw, dead = problem(n, rows, 7)
    wz[[0, 17, 49]] = 0.0
    res, q, rungs, scales, tab = run_q4(wz, u, hw, dead)
    assert np.all(q[[0, 17, 49]] == 0) and np.all(rungs[[0, 17, 49]] == 0) and np.all(scales[[0, 17, 49]] == 0)
    res, q, rungs, scales, tab = run_q2(wz, u, hw, dead)
    assert np.all(q[[0, 17, 49]] == 0) and np.all(rungs[[0, 17, 49]] == 0) and np.all(scales[[0, 17, 49]] == 0)
    # The debias of the oracle's q2tp result: zero rows (den = 0) keep their ladder.
    plane = np.zeros(rows * n // 4, dtype=np.uint8)
    qq = res["q"].astype(np.uint8).reshape(rows, n // 4, 4)
    plane[:] = (qq[..., 0] | (qq[..., 1] << 2) | (qq[..., 2] << 4) | (qq[..., 3] << 6)).reshape(-1)
    lost = oracle.ladder_q2tp(wz, hw)[1]
    tab_d = torch.from_numpy(tab.copy()).to(DEV)
    lost_d = torch.from_numpy(lost.copy()).to(DEV)
    sc_d = torch.from_numpy(res["scale"].astype(F32).reshape(-1).copy()).to(DEV)
    _lib.debias(2, torch.from_numpy(wz).to(DEV), torch.from_numpy(hp).to(DEV), torch.from_numpy(plane).to(DEV),
                torch.from_numpy(res["rung"].astype(np.uint8).reshape(-1)).to(DEV), tab_d, lost_d, sc_d)
    want = od.debias(wz, oracle.unpack_upper(hp, n), res["q"], res["rung"], tab, lost, True)
    for r in (0, 17, 49):
        assert np.array_equal(np_(lost_d)[r], lost[r]) and np.array_equal(np_(tab_d)[r], tab[r])
        assert np.array_equal(want["lost"][r], lost[r])


def test_quantize_group_q2tp_single_group(lib):
    # The whole chain at n = 32, one row.
    from gptq_post_weight_gb300 import _lib

    hp, w, wz, u, hw, dead = problem(32, 1, 11)
    out = _lib.quantize_group_q2tp(torch.from_numpy(hp).to(DEV), 32, torch.from_numpy(w).to(DEV), 0.01)
    tab, lost, _ = oracle.ladder_q2tp(wz, hw)
    assert np.array_equal(np_(out["lost"]), lost)
    res = oracle.sweep_q2tp(wz, u, hw, tab, dead)
    q = oracle.plane_to_codes(np_(out["codes"]), 1, 32)
    assert (q == res["q"]).mean() >= 31 / 32
