"""Bounded device waits: a wait that runs out reports GPTQ_ERR_TIMEOUT and
leaves the context usable.

Every wait inside the tensor-core kernels (a stage filled by the producer's
loads, an accumulator finished by the MMAs, an accumulator drained by the
epilogue) gives up after a limit of device time, stops issuing, drains what
it started, frees its tensor memory and sets a status bit that the call
turns into GPTQ_ERR_TIMEOUT.  The test hook gptq_test_set_wait shortens the
limit to 1 ms and makes the GEMM producers issue no loads, so nothing ever
fills a stage: the waits run out on purpose, with no fault, no trap and no
copy in flight.  Covered: the single-SM GEMM (the fold's first update and
the sweep's thin update are single-SM launches) and the SM-pair GEMM (the
Gram's update is the first launch of its call).  Right after, with the
defaults back, the same calls meet their parity bars.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F32 = np.float32
TIMEOUT = 6


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_waits_run_out_then_calls_recover(lib):
    from gptq_post_weight_gb300 import _lib

    n, rows = 512, 96
    cfg = synth.Config("waits", n, rows, 4 * n, 0.02, 1.5, 2, 2, 0.01, 21)
    hp, w = synth.make_problem(cfg, "cpu")
    hp, w = hp.numpy(), w.numpy()
    uo, do, dead, lamo = oracle.fold(hp, n, 0.01)
    x = np.random.default_rng(5).standard_normal((300, n)).astype(F32)
    hpd = torch.from_numpy(hp).cuda()
    try:
        _lib.test_set_wait(1_000_000, no_loads=True)
        with pytest.raises(_lib.GptqError) as ei:
            _lib.fold(hpd, n, 0.01)
        assert ei.value.code == TIMEOUT
        u0 = torch.from_numpy(uo.astype(F32)).cuda()
        wz = torch.from_numpy(w).cuda()
        wz[:, torch.from_numpy(dead).cuda()] = 0
        hd = torch.from_numpy(oracle.unpack_upper(hp, n).diagonal().astype(F32)).cuda()
        tab, lost = _lib.ladder(wz)
        with pytest.raises(_lib.GptqError) as ei:
            _lib.q4tp_sweep(wz.clone(), u0, hd, tab, lost)
        assert ei.value.code == TIMEOUT
        hg = torch.zeros(n * (n + 1) // 2, dtype=torch.float32, device="cuda")
        with pytest.raises(_lib.GptqError) as ei:
            _lib.gram_add(hg, torch.from_numpy(x).cuda())
        assert ei.value.code == TIMEOUT
        torch.cuda.synchronize()  # the context still answers
    finally:
        _lib.test_set_wait(0, no_loads=False)

    u, d, hdev, lam = _lib.fold(hpd, n, 0.01)
    assert lam == lamo
    assert rel_fro(u.cpu().numpy(), uo) <= 1e-4
    out = _lib.quantize_group(hpd, n, torch.from_numpy(w).cuda(), 0.01)
    tab_o, lost_o = oracle.ladder(np.where(dead[None, :], 0, w).astype(F32))
    res = oracle.sweep_q4tp(w, uo.astype(F32), oracle.unpack_upper(hp, n).diagonal().astype(F32), tab_o,
                            lost_o, dead)
    q = oracle.nibbles_to_codes(out["nibbles"].cpu().numpy(), rows, n)
    assert (q == res["q"]).mean() >= 0.999
    hg = torch.zeros(n * (n + 1) // 2, dtype=torch.float32, device="cuda")
    _lib.gram_add(hg, torch.from_numpy(x).cuda())
    g = x.astype(np.float64).T @ x.astype(np.float64)
    want = np.concatenate([g[r, r:] for r in range(n)])
    assert rel_fro(hg.cpu().numpy(), want) <= 1e-5


def test_wait_setter_arguments(lib):
    from gptq_post_weight_gb300 import _lib

    with pytest.raises(_lib.GptqError) as ei:
        _lib.test_set_wait(20_000_000_000, no_loads=False)  # above 10 s
    assert ei.value.code == 1
    _lib.test_set_wait(0, no_loads=False)
