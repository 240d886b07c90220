"""The bench's algorithmic flop counts (the roofline's numerator) against an
independent per-entry count (CPU only).

Blocked right-looking Cholesky: entry (i, j) of the lower triangle receives,
through update GEMMs, one multiply-add per column of every block before j's
own block (its own block's columns are the diagonal and panel kernels' work).
Inverse accumulated alongside: entry (c, i), c < i, receives NB multiply-adds
from every step k with c < k + NB <= i.  However the schedule groups the steps
(groups of four, with strip updates between them), the sums must agree exactly.
The sweep: column t of W receives one multiply-add per row for every column of
the blocks before t's block.
"""
import numpy as np
import pytest

import bench


def per_entry_fold(n, NB=128):
    N = (n + NB - 1) // NB * NB
    blk = np.arange(N, dtype=np.int64) // NB
    chol = int(((N - np.arange(N)) * NB * blk).sum())
    # sum over c < i of (blk[i] - blk[c]) = i * blk[i] - sum_{c<i} blk[c]
    before = np.concatenate([[0], np.cumsum(blk)[:-1]])
    inv = int((NB * (np.arange(N) * blk - before)).sum())
    return 2 * (chol + inv)


@pytest.mark.parametrize("n", [128, 256, 384, 512, 640, 896, 1000, 4096, 17408])
@pytest.mark.parametrize("G", [1, 2, 4])
def test_fold_update_flops_per_entry(n, G):
    assert bench.fold_gemm_flops(n, part="all", G=G) == per_entry_fold(n)
    assert (bench.fold_gemm_flops(n, part="trailing", G=G) + bench.fold_gemm_flops(n, part="strip", G=G)
            == per_entry_fold(n))


def test_fold_update_flops_near_textbook():
    # Cholesky n^3/3 + inverse n^3/3; the update GEMMs carry all but the
    # O(n^2 NB) diagonal-block and panel work.
    n = 17408
    got = bench.fold_gemm_flops(n, part="all")
    assert 0.99 < got / (2 * n ** 3 / 3) < 1.0


@pytest.mark.parametrize("rows,n", [(5, 128), (7, 544), (5120, 17408)])
def test_sweep_update_flops_per_entry(rows, n):
    SB = 128
    t = np.arange(n, dtype=np.int64)
    want = 2 * rows * int((SB * (t // SB)).sum())
    assert bench.sweep_gemm_flops(rows, n) == want


def test_hbm_report_arithmetic():
    n, rows = 256, 64
    per_kind = {"build": {"ms_per_step": 0.5, "launches_per_step": 1},
                "sweep_block": {"ms_per_step": 2.0, "launches_per_step": 2},
                "fold_gemm": {"ms_per_step": 9.0, "launches_per_step": 1}}
    rep = bench.hbm_report(per_kind, n, rows, "q4tp", peak_gbs=1000.0)
    assert set(rep) == {"build", "sweep_block"}  # kinds that did not run are left out
    b = n * (n + 1) // 2 * 4 + n * n * 4
    assert rep["build"]["bytes_per_group"] == b
    assert rep["build"]["gbs"] == pytest.approx(b / 0.5e-3 / 1e9)
    assert rep["build"]["frac"] == pytest.approx(rep["build"]["gbs"] / 1000.0)
    sw = rows * n * 4 + n * 128 * 4 + rows * n // 2 + rows * (n // 32) * 5
    assert rep["sweep_block"]["bytes_per_group"] == sw
    q2 = bench.hbm_report(per_kind, n, rows, "q2tp", peak_gbs=None)
    assert q2["sweep_block"]["bytes_per_group"] == sw - rows * n // 2 + rows * n // 4
    assert q2["build"]["frac"] is None
