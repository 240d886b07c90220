"""The Python binding refuses buffers whose dtype, size or placement the call
cannot use, before anything reaches the library (CPU only: every case here
fails in the checks).  The kernels index each buffer by the sizes the call
states, so a short U or a ladder of the wrong height must be an error on the
host, not a read past the end of a device buffer."""
import os

import pytest

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def blib():
    from gptq_post_weight_gb300 import _lib, build

    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    _lib.load()
    return _lib


def f32(*shape):
    return torch.zeros(*shape, dtype=torch.float32)


def u8(*shape):
    return torch.zeros(*shape, dtype=torch.uint8)


def refused(fn, *args, match, **kw):
    with pytest.raises(ValueError, match=match):
        fn(*args, **kw)


def test_sweep_sizes(blib):
    rows, n = 6, 64
    w, u, hw, tab, lost = f32(rows, n), f32(n, n), f32(n), f32(rows, 32), f32(rows, 2)
    refused(blib.q4tp_sweep, w, f32(n, n - 1), hw, tab, lost, match="u must have 4096")
    refused(blib.q4tp_sweep, w, u, f32(n - 32), tab, lost, match="hw must have 64")
    refused(blib.q4tp_sweep, w, u, hw, f32(rows - 1, 32), lost, match="tab must have 192")
    refused(blib.q4tp_sweep, w, u, hw, tab, f32(rows, 3), match="lost must have 12")
    refused(blib.q4tp_sweep, f32(rows * n), u, hw, tab, lost, match="2-D")
    refused(blib.q4tp_sweep, w.double(), u, hw, tab, lost, match="w must be torch.float32")
    refused(blib.q4tp_sweep, w.t(), u, hw, tab, lost, match="contiguous")
    # Right sizes: only the placement is left to refuse.
    refused(blib.q4tp_sweep, w, u, hw, tab, lost, match="must be CUDA tensors")
    refused(blib.q4tp_sweep_noalloc, w, f32(1, 4), hw, tab, lost, match="u must have")
    refused(blib.q2tp_sweep, w, u, f32(n + 1), tab, match="hw must have")


def test_sweep_out_buffers(blib):
    rows, n = 4, 96
    gpr = n // 32
    args = (f32(rows, n), f32(n, n), f32(n), f32(rows, 32), f32(rows, 2))
    good = (u8(rows * n // 2), u8(rows * gpr), f32(rows * gpr))
    refused(blib.q4tp_sweep, *args, out=good[:2], match="out must hold 3")
    refused(blib.q4tp_sweep, *args, out=(u8(rows * n // 4),) + good[1:], match="nibbles must have")
    refused(blib.q4tp_sweep, *args, out=good[:2] + (u8(rows * gpr),), match="scales must be torch.float32")
    q2good = (u8(rows * n // 4), u8(rows * gpr), f32(rows * gpr))
    refused(blib.q2tp_sweep, *args[:4], out=(u8(rows * n // 2),) + q2good[1:], match="codes must have")


def test_chained_calls(blib):
    rows, n = 3, 64
    hp = f32(n * (n + 1) // 2)
    refused(blib.quantize_group, f32(n * n), n, f32(rows, n), match="h_packed must have 2080")
    refused(blib.quantize_group, hp, n, f32(rows, n + 32), match="96 columns, n = 64")
    refused(blib.quantize_group_q2tp, hp, n, f32(rows, n - 32), match="32 columns, n = 64")
    refused(blib.quantize_group_act_order, f32(10), n, f32(rows, n), match="h_packed must have")
    refused(blib.fold, f32(n * (n + 1) // 2 + 1), n, match="h_packed must have 2080")
    refused(blib.build_equilibrated, f32(7), n, match="h_packed must have")
    refused(blib.fold_permuted, hp, n, torch.zeros(n, dtype=torch.int64), match="perm must be torch.int32")
    refused(blib.gram_add, f32(100), f32(256, n), match="h_packed must have 2080")


def test_group_rule_and_debias(blib):
    rows = 5
    refused(blib.q4tp_group, f32(rows, 16), f32(32, 32), f32(32), f32(rows, 32), f32(rows, 2),
            match=r"\[rows, 32\]")
    refused(blib.q4tp_group, f32(rows, 32), f32(16, 32), f32(32), f32(rows, 32), f32(rows, 2),
            match="ublk must have 1024")
    refused(blib.q2tp_group, f32(rows, 32), f32(32, 32), f32(31), f32(rows, 32), match="hw must have 32")
    refused(blib.q2tp_place, f32(rows, 64), f32(32), match="hw must have 64")
    n = 64
    gpr = n // 32
    w, hp = f32(rows, n), f32(n * (n + 1) // 2)
    tail = (u8(rows * gpr), f32(rows, 32), f32(rows, 2), f32(rows * gpr))
    refused(blib.debias, 2, w, hp, u8(rows * n // 2), *tail, match="codes must have 80")
    refused(blib.debias, 4, w, hp, u8(rows * n // 4), *tail, match="codes must have 160")
    refused(blib.debias, 2, w, hp, u8(rows * n // 4), u8(rows * gpr), f32(rows, 32), f32(rows, 2),
            f32(rows * gpr + 1), match="scales must have 10")
    refused(blib.static_rungs, w, f32(rows, 31), f32(rows, 2), match="tab must have 160")
    refused(blib.q4tp_sweep_act_order, w, f32(n, n), torch.zeros(n, dtype=torch.int32), f32(rows, 32),
            u8(rows * gpr - 1), match="rungs must have 10")
