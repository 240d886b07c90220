"""Act-order q4tp on the device against the oracle (same tolerances as the
natural-order path: U relative Frobenius 1e-4, permutation and static rungs
exact, >= 99.9 % of codes equal, output error within 1 %)."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F32 = np.float32


def np_(t):
    return t.detach().cpu().numpy()


def rel_fro(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / np.linalg.norm(b))


def test_perm_exact(lib):
    from gptq_post_weight_gb300 import _lib

    rng = np.random.default_rng(0)
    h = np.exp(rng.standard_normal(3000)).astype(F32)
    h[::7] = h[3]          # ties
    h[10] = 0.0
    h[11] = -0.0
    h[12] = np.nan
    h[13] = np.inf
    h[14] = -1.0
    perm = np_(_lib.act_order_perm(torch.from_numpy(h).cuda()))
    assert np.array_equal(perm, oracle.act_order_perm(h))


@pytest.mark.parametrize("n,rows,seed", [(256, 64, 0), (1024, 300, 3)])
def test_act_order_group(lib, n, rows, seed):
    from gptq_post_weight_gb300 import _lib

    cfg = synth.Config(f"ao{n}", n, rows, 4 * n, 0.02, 1.5, max(2, n // 256), 3, 0.01, seed)
    hp, w = synth.make_problem(cfg, "cpu")
    hp, w = hp.numpy(), w.numpy()
    out = _lib.quantize_group_act_order(torch.from_numpy(hp).cuda(), n, torch.from_numpy(w).cuda(), 0.01)
    hraw = oracle.unpack_upper(hp, n)
    hd32 = hraw.diagonal().astype(F32)
    perm = oracle.act_order_perm(hd32)
    assert np.array_equal(np_(out["perm"]), perm)
    up, _, _, lam = oracle.fold(oracle.permute_packed(hp, n, perm), n, 0.01)
    assert out["lam"] == lam
    assert rel_fro(np_(out["u"]), up) <= 1e-4
    dead = ~(hd32 > 0)
    wz = w.copy()
    wz[:, dead] = 0
    tab, lost = oracle.ladder(wz)
    rungs = oracle.converter_rungs(wz, tab, lost)
    assert np.array_equal(np_(out["rungs"]).reshape(rows, -1).astype(np.int64), rungs)
    res = oracle.sweep_q4tp_act_order(w, up.astype(F32), dead, perm, tab, rungs)
    q_dev = oracle.nibbles_to_codes(np_(out["nibbles"]), rows, n)
    agree = float((q_dev == res["q"]).mean())
    sc = np_(out["scales"]).reshape(rows, -1)
    assert np.array_equal(sc.view(np.uint32), res["scale"].view(np.uint32))
    e_dev = oracle.output_error(w, oracle.dequant_q4tp(q_dev, sc), hraw)
    e_or = oracle.output_error(w, oracle.dequant_q4tp(res["q"], res["scale"]), hraw)
    assert agree >= 0.999, agree
    assert abs(e_dev - e_or) <= 0.01 * e_or, (e_dev, e_or)


@pytest.mark.slow
def test_act_order_full_size(lib):
    from gptq_post_weight_gb300 import _lib

    cfg = synth.config("n17408")
    hpd, wd = synth.make_problem(cfg, "cuda")
    out = _lib.quantize_group_act_order(hpd, cfg.n, wd, cfg.lam)
    hp, w = np_(hpd), np_(wd)
    del hpd, wd
    n = cfg.n
    hd32 = np.array([hp[i * (2 * n - i + 1) // 2] for i in range(n)], dtype=F32)
    perm = oracle.act_order_perm(hd32)
    assert np.array_equal(np_(out["perm"]), perm)
    up, _, _, lam = oracle.fold(oracle.permute_packed(hp, n, perm), n, cfg.lam)
    assert rel_fro(np_(out["u"]), up) <= 1e-4
    rows_idx = np.sort(np.random.default_rng(1).choice(cfg.rows, 16, replace=False))
    dead = ~(hd32 > 0)
    wz = w[rows_idx].copy()
    wz[:, dead] = 0
    tab, lost = oracle.ladder(wz)
    rungs = oracle.converter_rungs(wz, tab, lost)
    res = oracle.sweep_q4tp_act_order(w[rows_idx], up.astype(F32), dead, perm, tab, rungs)
    q_dev = oracle.nibbles_to_codes(np_(out["nibbles"]), cfg.rows, n)[rows_idx]
    assert float((q_dev == res["q"]).mean()) >= 0.999
