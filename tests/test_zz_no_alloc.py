"""The sweep entry point that allocates nothing.

Some callers cannot allocate device memory: a plugin whose host framework owns
all device memory and lends it only the input and output buffers, or a caller
that keeps cudaMalloc (which can synchronise the device) off its hot path.
For them gptq_q4tp_sweep_noalloc keeps its scratch in a static device array
inside the library.  This checks, through the C ABI, that it gives exactly
what the workspace entry point gives, on two calls in a row (the second
reuses the array with the first call's leftovers): with the array large
enough for groups of four blocks, and at a shape where it only holds the
pair-of-blocks layout (the layout of the 5120 x 17408 group), which is also
held against the oracle.  It refuses shapes the array cannot hold.
Collected last on purpose.
"""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _inputs(n, rows, seed):
    from gptq_post_weight_gb300 import _lib

    cfg = synth.Config(f"na{n}", n, rows, 4 * n, 0.02, 1.5, 3, 3, 0.01, seed)
    hp, w = synth.make_problem(cfg, "cpu")
    u, d, hd, lam = _lib.fold(hp.cuda(), n, 0.01)
    wz = w.cuda()
    wz[:, ~(hd > 0)] = 0
    tab, lost = _lib.ladder(wz)
    return wz, u, hd, tab, lost


def test_noalloc_sweep_matches_workspace_sweep(lib):
    from gptq_post_weight_gb300 import _lib

    for n, rows, seed in ((1024, 300, 11), (512, 97, 12)):
        wz, u, hd, tab, lost = _inputs(n, rows, seed)
        ref = _lib.q4tp_sweep(wz.clone(), u, hd, tab, lost)
        for call in range(2):
            got = _lib.q4tp_sweep_noalloc(wz.clone(), u, hd, tab, lost)
            torch.cuda.synchronize()
            for a, b in zip(ref, got):
                assert torch.equal(a, b), (n, rows, call)


def test_noalloc_sweep_pairs_of_blocks(lib):
    # rows + n above 12287: the array holds only the pair-of-blocks layout, so
    # both calls run pairs; the workspace sweep given exactly the pair
    # layout's bytes runs the same schedule and must match bit for bit, and
    # the result meets the end-to-end bar against the oracle (codes >= 99.9 %
    # equal, output error within 1 %).
    import oracle
    from gptq_post_weight_gb300 import _lib

    n, rows = 512, 12000
    assert rows * 4096 + n * 4096 > 48 << 20 >= rows * 2048 + n * 2048 + 4096
    cfg = synth.Config(f"na{n}", n, rows, 4 * n, 0.02, 1.5, 3, 3, 0.01, 13)
    hp, w = synth.make_problem(cfg, "cpu")
    hp, w = hp.numpy(), w.numpy()
    uo, do, dead, lam = oracle.fold(hp, n, 0.01)
    u32 = uo.astype(np.float32)
    wz = w.copy()
    wz[:, dead] = 0
    hraw = oracle.unpack_upper(hp, n)
    hw = hraw.diagonal().astype(np.float32)
    tab, lost = oracle.ladder(wz)
    res = oracle.sweep_q4tp(wz, u32, hw, tab, lost, dead)
    dev = [torch.from_numpy(x).cuda() for x in (wz, u32, hw, tab, lost)]
    ws = _lib.workspace(2 * rows * 1024 + 2 * n * 1024 + 1024, "cuda")
    ref = _lib.q4tp_sweep(dev[0].clone(), *dev[1:], ws=ws)
    for call in range(2):
        got = _lib.q4tp_sweep_noalloc(dev[0].clone(), *dev[1:])
        torch.cuda.synchronize()
        for a, b in zip(ref, got):
            assert torch.equal(a, b), call
    q = oracle.nibbles_to_codes(got[0].cpu().numpy(), rows, n)
    agree = float((q == res["q"]).mean())
    assert agree >= 0.999, agree
    sc = got[2].cpu().numpy().reshape(rows, -1)
    e_dev = oracle.output_error(wz, oracle.dequant_q4tp(q, sc), hraw)
    e_or = oracle.output_error(wz, oracle.dequant_q4tp(res["q"], res["scale"]), hraw)
    assert abs(e_dev - e_or) <= 0.01 * e_or, (e_dev, e_or)


def test_noalloc_sweep_rejects_oversize(lib):
    from gptq_post_weight_gb300 import _lib

    limit = 48 << 20
    # The array holds the pair-of-blocks layout (rows*2048 + n*2048 bytes)
    # of the flagship 5120 x 17408 group, not of 4096 x 24576.
    assert 5120 * 2048 + 17408 * 2048 + 4096 <= limit
    rows, n = 4096, 24576
    assert rows * 2048 + n * 2048 > limit
    w = torch.zeros(rows, n, dtype=torch.float32, device="cuda")
    u = torch.empty(n, n, dtype=torch.float32, device="cuda")  # never read: the library refuses first
    hw = torch.zeros(n, dtype=torch.float32, device="cuda")
    tab = torch.zeros(rows, 32, dtype=torch.float32, device="cuda")
    lost = torch.zeros(rows, 2, dtype=torch.float32, device="cuda")
    with pytest.raises(_lib.GptqError) as ei:
        _lib.q4tp_sweep_noalloc(w, u, hw, tab, lost)
    assert ei.value.code == 3
