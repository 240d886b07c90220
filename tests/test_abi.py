"""The C-ABI library loads, exports every symbol include/gptq_fold.h
declares, and rejects bad arguments before any device work (CPU only: no
call here reaches a kernel)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gptq_fold.h")


@pytest.fixture(scope="module")
def clib():
    from gptq_post_weight_gb300 import _lib, build

    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.load()


def declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gptq_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared()
    for want in ("gptq_fold", "gptq_q4tp_sweep", "gptq_quantize_group", "gptq_ladder",
                 "gptq_q4tp_group", "gptq_fold_workspace_bytes"):
        assert want in names


def test_every_declared_symbol_is_exported(clib):
    from gptq_post_weight_gb300 import _lib

    for name in declared():
        assert hasattr(clib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_workspace_sizes(clib):
    assert clib.gptq_fold_workspace_bytes(0) == 0
    assert clib.gptq_fold_workspace_bytes(70000) == 0
    n = 17408
    need = clib.gptq_fold_workspace_bytes(n)
    # One N x N working matrix, plus the TF32 hi/lo panels of a group of
    # four steps (L and Y parts: 4 buffers of N x 4 NB) and small buffers.
    panels = 4 * n * (4 * 128) * 4
    assert need >= n * n * 4 + panels
    assert need < (n * n * 4 + panels) * 1.01
    assert clib.gptq_sweep_workspace_bytes(5120, n) > 0
    assert clib.gptq_group_workspace_bytes(5120, n) > need


def test_argument_errors_before_launch(clib):
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: every call below fails its checks first
    mis = P((1 << 20) + 4)
    ws = P(1 << 21)
    lam = ctypes.c_double()
    # shape errors
    assert clib.gptq_fold(fake, 0, 0.01, fake, None, None, None, ws, 1 << 40, None) == 2
    assert clib.gptq_ladder(fake, 4, 48, fake, fake, None) == 2
    assert clib.gptq_q4tp_sweep(fake, 4, 40, fake, fake, fake, fake, fake, fake, fake, ws, 1 << 40, None) == 2
    assert clib.gptq_q4tp_sweep(fake, 0, 64, fake, fake, fake, fake, fake, fake, fake, ws, 1 << 40, None) == 2
    # null / misaligned pointers
    assert clib.gptq_fold(None, 16, 0.01, fake, None, None, None, ws, 1 << 40, None) == 1
    assert clib.gptq_fold(mis, 16, 0.01, fake, None, None, None, ws, 1 << 40, None) == 1
    assert clib.gptq_fold(fake, 16, float("nan"), fake, None, None, ctypes.byref(lam), ws, 1 << 40, None) == 1
    assert clib.gptq_q4tp_group(fake, 8, fake, fake, None, fake, fake, fake, fake, fake, None) == 1
    # workspace too small
    assert clib.gptq_fold(fake, 16, 0.01, fake, None, None, None, ws, 16, None) == 3
    assert clib.gptq_q4tp_sweep(fake, 4, 64, fake, fake, fake, fake, fake, fake, fake, ws, 16, None) == 3
    assert clib.gptq_quantize_group(fake, 64, 0.01, fake, 4, fake, fake, fake, None, None, None, None,
                                    None, None, ws, 16, None) == 3
    assert clib.gptq_status_string(4).startswith(b"not positive definite")


def test_q2tp_and_debias_argument_errors(clib):
    P = ctypes.c_void_p
    fake = P(1 << 20)
    mis = P((1 << 20) + 4)
    ws = P(1 << 21)
    # shapes: n % 32 != 0, rows = 0
    assert clib.gptq_q2tp_place(fake, 4, 48, fake, fake, fake, None, None) == 2
    assert clib.gptq_q2tp_sweep(fake, 4, 40, fake, fake, fake, fake, fake, fake, ws, 1 << 40, None) == 2
    assert clib.gptq_q2tp_sweep(fake, 0, 64, fake, fake, fake, fake, fake, fake, ws, 1 << 40, None) == 2
    assert clib.gptq_debias(2, fake, 4, 40, fake, fake, fake, fake, fake, fake, None, ws, 1 << 40, None) == 2
    # pointers, codec width
    assert clib.gptq_q2tp_place(fake, 4, 64, mis, fake, fake, None, None) == 1
    assert clib.gptq_q2tp_place(fake, 4, 64, fake, fake, fake, mis, None) == 1
    assert clib.gptq_q2tp_group(fake, 8, fake, fake, None, fake, fake, fake, fake, None) == 1
    assert clib.gptq_debias(3, fake, 4, 64, fake, fake, fake, fake, fake, fake, None, ws, 1 << 40, None) == 1
    assert clib.gptq_debias(2, fake, 4, 64, fake, fake, fake, fake, fake, fake, mis, ws, 1 << 40, None) == 1
    # workspace too small
    assert clib.gptq_q2tp_sweep(fake, 4, 64, fake, fake, fake, fake, fake, fake, ws, 16, None) == 3
    assert clib.gptq_quantize_group_q2tp(fake, 64, 0.01, fake, 4, fake, fake, fake, None, None, None,
                                         None, None, None, ws, 16, None) == 3
    assert clib.gptq_debias(4, fake, 4, 64, fake, fake, fake, fake, fake, fake, None, ws, 16, None) == 3
    assert clib.gptq_debias_workspace_bytes(5120, 17408) >= 2 * 17408 * 17408 * 4
    assert clib.gptq_debias_workspace_bytes(0, 64) == 0


def test_gram_and_act_order_argument_errors(clib):
    P = ctypes.c_void_p
    fake = P(1 << 20)
    mis = P((1 << 20) + 4)
    ws = P(1 << 21)
    big = 1 << 40
    # Gram: shapes, pointers, workspace; an empty window (T = 0) is a no-op.
    assert clib.gptq_gram_workspace_bytes(0) == 0
    assert clib.gptq_gram_add(fake, 0, fake, 10, ws, big, None) == 2
    assert clib.gptq_gram_add(fake, 64, fake, -1, ws, big, None) == 2
    assert clib.gptq_gram_add(None, 64, fake, 10, ws, big, None) == 1
    assert clib.gptq_gram_add(fake, 64, None, 10, ws, big, None) == 1
    assert clib.gptq_gram_add(fake, 64, mis, 10, ws, big, None) == 1
    assert clib.gptq_gram_add(fake, 64, fake, 10, ws, 16, None) == 3
    assert clib.gptq_gram_add(fake, 64, None, 0, ws, big, None) == 0
    # Act order.
    lam = ctypes.c_double()
    assert clib.gptq_act_order_perm(fake, 0, fake, None) == 2
    assert clib.gptq_act_order_perm(None, 64, fake, None) == 1
    assert clib.gptq_act_order_perm(fake, 64, mis, None) == 1
    assert clib.gptq_fold_permuted(fake, 64, float("nan"), fake, fake, None, None, ctypes.byref(lam), ws, big,
                                   None) == 1
    assert clib.gptq_fold_permuted(fake, 64, 0.01, None, fake, None, None, ctypes.byref(lam), ws, big, None) == 1
    assert clib.gptq_fold_permuted(fake, 64, 0.01, fake, fake, None, None, ctypes.byref(lam), ws, 16, None) == 3
    assert clib.gptq_static_rungs(fake, 4, 48, fake, fake, fake, fake, None) == 2
    assert clib.gptq_static_rungs(fake, 4, 64, fake, fake, None, fake, None) == 1
    assert clib.gptq_q4tp_sweep_act_order(fake, 0, 64, fake, fake, fake, fake, fake, ws, big, None) == 2
    assert clib.gptq_q4tp_sweep_act_order(fake, 4, 64, fake, mis, fake, fake, fake, ws, big, None) == 1
    assert clib.gptq_q4tp_sweep_act_order(fake, 4, 64, fake, fake, fake, fake, fake, ws, 16, None) == 3
    assert clib.gptq_sweep_act_order_workspace_bytes(0, 64) == 0
    assert clib.gptq_quantize_group_act_order(fake, 64, 0.01, fake, 4, fake, fake, fake, None, None, None,
                                              ws, 16, None) == 3
    assert clib.gptq_quantize_group_act_order(fake, 64, float("inf"), fake, 4, fake, fake, fake, None, None,
                                              None, ws, big, None) == 1
    assert clib.gptq_group_act_order_workspace_bytes(4, 0) == 0


def test_wait_hook_arguments(clib):
    # Host-side checks only: nothing here launches a kernel.
    assert clib.gptq_test_set_wait(ctypes.c_ulonglong(20_000_000_000), 0) == 1  # above 10 s
    assert clib.gptq_test_set_wait(ctypes.c_ulonglong(1_000_000), 2) == 1
    assert clib.gptq_test_set_wait(ctypes.c_ulonglong(0), 0) == 0
