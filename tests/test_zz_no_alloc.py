"""The sweep entry point that allocates nothing.

Some callers cannot allocate device memory: code that runs while its stream is
being captured into a graph, or a plugin whose host framework owns all device
memory and lends it only the input and output buffers.  For them
gptq_q4tp_sweep_noalloc keeps its scratch in a static device array inside the
library.  This checks, through the C ABI, that it gives exactly what the
workspace entry point gives, on two calls in a row (the second reuses the
array with the first call's leftovers), and that it refuses shapes its array
cannot hold.  Collected last on purpose.
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
        got = _lib.q4tp_sweep_noalloc(wz.clone(), u, hd, tab, lost)
        torch.cuda.synchronize()
        for a, b in zip(ref, got):
            assert torch.equal(a, b), (n, rows)


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
