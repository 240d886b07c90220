"""The bench's reference arm samples the oracle and scales it to seconds per
full group (CPU only, on the small workload): the estimate is the sampled
fold time times (n / n_fold)^3 plus the sampled sweep time times
rows / rows_sweep, for both codecs, and the sample description says so."""
import re

import pytest

import bench
import synth

pytest.importorskip("torch")


@pytest.mark.parametrize("codec", ["q4tp", "q2tp"])
def test_cpu_baseline_sample_scaling(codec):
    cfg = synth.config("tiny")
    est, sample, spent = bench.cpu_baseline_sample(cfg, n_fold=128, rows_sweep=2, codec=codec)
    assert est > 0 and spent > 0
    m = re.match(r"oracle fold at n=128 \(([\d.]+) s, x\(n/128\)\^3\) \+ oracle (\w+) ladder and sweep of 2 rows "
                 r"at n=256 \(([\d.]+) s, x64/2\)", sample)
    assert m and m.group(2) == codec
    # The scaled estimate exceeds what was spent (both factors exceed 1).
    assert est >= spent
