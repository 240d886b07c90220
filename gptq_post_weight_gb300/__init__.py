"""GB300 GPTQ fold + q4tp sweep: a C-ABI CUDA library (libgptqfold.so,
declared in include/gptq_fold.h) and its thin ctypes binding (``_lib``).

    from gptq_post_weight_gb300 import _lib
    u, d, hdiag, lam = _lib.fold(h_packed, n, 0.01)
    nib, rungs, scales = _lib.q4tp_sweep(w, u, hdiag, *_lib.ladder(w))
"""
from . import _lib  # noqa: F401
from ._lib import GptqError, load  # noqa: F401
