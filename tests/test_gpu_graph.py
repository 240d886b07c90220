"""gptq_quantize_group replayed as a CUDA graph.

The library runs the first call with a given set of arguments on the stream,
captures the second into a graph (one fold attempt at the given damping, the
ladder, the sweep) and replays it from then on.  Through the C ABI this
checks that the replays give the stream path's results bit for bit (codes,
rungs, scales, the ladder, D, diag H, U and the damping used; q4tp and
q2tp), that each call
counts the same number of kernel launches, that a first attempt that fails
(H of rank n/2 at lambda = 0) falls back to the stream path's damping
retry with the same result.
"""
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _buffers(lib, n, rows):
    from gptq_post_weight_gb300 import _lib

    gpr = n // 32
    dev = "cuda"
    return dict(
        nib=torch.empty(rows * n // 2, dtype=torch.uint8, device=dev),
        rungs=torch.empty(rows * gpr, dtype=torch.uint8, device=dev),
        scales=torch.empty(rows * gpr, dtype=torch.float32, device=dev),
        tab=torch.empty(rows * 32, dtype=torch.float32, device=dev),
        lost=torch.empty(rows * 2, dtype=torch.float32, device=dev),
        u=torch.empty(n * n, dtype=torch.float32, device=dev),
        d=torch.empty(n, dtype=torch.float32, device=dev),
        hd=torch.empty(n, dtype=torch.float32, device=dev),
        ws=_lib.workspace(lib.gptq_group_workspace_bytes(rows, n), dev),
    )


def _call(lib, hp, n, w, rows, lam, b, stream, q2=False):
    import ctypes

    from gptq_post_weight_gb300 import _lib

    used = ctypes.c_double(-1.0)
    fn = lib.gptq_quantize_group_q2tp if q2 else lib.gptq_quantize_group
    code = fn(
        _lib._ptr(hp), n, float(lam), _lib._ptr(w), rows, _lib._ptr(b["nib"]), _lib._ptr(b["rungs"]),
        _lib._ptr(b["scales"]), _lib._ptr(b["tab"]), _lib._ptr(b["lost"]), _lib._ptr(b["u"]), _lib._ptr(b["d"]),
        _lib._ptr(b["hd"]), ctypes.byref(used), _lib._ptr(b["ws"]), b["ws"].numel(), stream)
    torch.cuda.synchronize()
    return code, used.value


def _snapshot(b):
    return {k: v.clone() for k, v in b.items() if k != "ws"}


@pytest.mark.parametrize("n,rows,seed,q2", [(1024, 300, 21, False), (640, 97, 22, False), (1024, 300, 23, True)])
def test_graph_replays_match_stream_path(lib, n, rows, seed, q2):
    cfg = synth.Config(f"gr{n}", n, rows, 4 * n, 0.02, 1.5, 3, 3, 0.01, seed)
    hp, w = synth.make_problem(cfg, "cuda")
    b = _buffers(lib, n, rows)
    st = torch.cuda.Stream()
    runs = []
    for call in range(4):  # stream path, capture + replay, replay, replay
        l0 = lib.gptq_launch_count()
        code, used = _call(lib, hp, n, w, rows, cfg.lam, b, st.cuda_stream, q2)
        assert code == 0, (call, code)
        runs.append((_snapshot(b), used, lib.gptq_launch_count() - l0))
    ref, used0, launches0 = runs[0]
    assert launches0 > 0
    for call, (got, used, launches) in enumerate(runs[1:], 1):
        assert used == used0, call
        assert launches == launches0, (call, launches, launches0)
        for k in ref:
            assert torch.equal(ref[k], got[k]), (call, k)


def test_graph_failed_attempt_falls_back(lib):
    # Rank n/2 at lambda = 0: the captured attempt's pivot flag is set, and
    # the call must then give what the stream path's retry gives.
    n, rows = 384, 64
    cfg = synth.Config("grd", n, rows, n // 2, 0.02, 1.0, 2, 2, 0.0, 3)
    hp, w = synth.make_problem(cfg, "cuda")
    b = _buffers(lib, n, rows)
    st = torch.cuda.Stream()
    outs = []
    for call in range(3):
        code, used = _call(lib, hp, n, w, rows, 0.0, b, st.cuda_stream)
        assert code == 0, (call, code)
        assert used >= 1e-4, (call, used)
        outs.append((_snapshot(b), used))
    for call in (1, 2):
        assert outs[call][1] == outs[0][1]
        for k in outs[0][0]:
            assert torch.equal(outs[0][0][k], outs[call][0][k]), (call, k)
