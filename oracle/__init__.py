"""Oracle for the GPTQ fold + q4tp sweep: plain, slow, CPU-only.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and
the benchmark's CPU-baseline leg may import this package.  It shares no code
with the CUDA library (``gptq_post_weight_gb300``) and imports nothing from
it; the library never imports it.

What it follows (pages of the ``cortiq`` project, cited by page title and
item):

* ``cortiq-cli src/gptq.rs``, ``gptq_fold_operator_par``: the host fold.  Dead
  channels (``!(H_ii > 0)``) get a zero row/column and unit diagonal; damping
  ``lambda * max(mean(diag), 1e-12)`` is added to the whole diagonal; a failed
  Cholesky raises lambda (0 -> 1e-4, else x10, stop once > 10); then
  ``L = chol(H_d)``, ``L^-1``, ``H_d^-1 = L^-T L^-1``, ``M = chol(H_d^-1)``,
  ``U = M^T`` -- computed here in f64 and returned as f32 like the page does.
* ``cortiq-cli src/gptq.rs``, ``gptq_quantize_q4tp``: the host q4tp sweep in f32
  (rung rule, ties-even rounding into [-8, 7], ``e = (w - q s) / U_jj`` and the
  full-row update ``w[j+1..] -= e * U[j, j+1..]`` right after each column).
* ``cortiq-engine src/gpu_wgpu/gptq_dev.rs``, ``build_a``: the equilibrated,
  reversed, damped matrix (only to check the library's builder step).
* ``cortiq-cli src/gptq.rs``, the calibration pass (``gram_add_dev``): the
  Hessian accumulator H += X^T X over a window of tokens, packed upper.
* ``cortiq-cli src/gptq.rs``, ``act_order_perm`` / ``permute_sym`` /
  ``gptq_quantize_q4tp_act_order``: act-order with static groups.
* ``cortiq-engine src/gpu_wgpu/gptq_dev.rs``, WGSL ``q2_level`` /
  ``q2tp_group``, and ``cortiq-cli src/gptq.rs``, ``gptq_quantize_q2tp`` with
  ``Q2tpRule::Placed``: the 2-bit "placed" rule (ladder placement, full rung
  search, the lazy-block host sweep).
* ``cortiq-cli src/gptq.rs``, ``q2tp_debias_hessian`` / ``q4tp_debias_hessian``:
  the output debias (per-row slope (W^ H W^T)_rr / (W H W^T)_rr removed
  through the row's f16 lo).

Readings of points the pages leave open are stated where they are used
(``ladder`` for the missing converter ladder, ``nominal_rung`` for the f32
log2, the ``q2tp`` module docstring for the placed ladder).

Every function is pinned by ``tests/test_oracle_*.py`` (closed forms,
hand-computed cases, invariants, brute force); none is "parity unpinned".
"""
from .fold import (  # noqa: F401
    NotSPD,
    fold,
    unpack_upper,
    equilibrated_reversed,
    fold_damping,
)
from .q4tp import (  # noqa: F401
    ladder,
    nominal_rung,
    group_q4tp,
    sweep_q4tp,
    sweep_q4tp_f64,
    dequant_q4tp,
    output_error,
    nibbles_to_codes,
)
from .gram import gram_add, pack_upper  # noqa: F401,E402
from .actorder import (  # noqa: F401,E402
    act_order_perm,
    converter_rungs,
    permute_packed,
    sweep_q4tp_act_order,
    total_cmp_key,
)
from .q2tp import (  # noqa: F401,E402
    q2_level,
    place_scale,
    ladder_q2tp,
    group_q2tp,
    sweep_q2tp,
    sweep_q2tp_f64,
    dequant_q2tp,
    plane_to_codes,
)
from . import debias  # noqa: F401,E402
