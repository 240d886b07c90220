"""ctypes binding of libgptqfold.so (include/gptq_fold.h).

Argument marshalling only: every step runs in the library's CUDA kernels.
The wrappers take torch CUDA tensors (device memory and the current stream
come from PyTorch) and raise ``GptqError`` on a non-zero status.  There is
no fallback: without the built library every call fails loudly.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgptqfold.so")

STATUS = {0: "GPTQ_OK", 1: "GPTQ_ERR_ARG", 2: "GPTQ_ERR_SHAPE", 3: "GPTQ_ERR_NOMEM",
          4: "GPTQ_ERR_NOT_SPD", 5: "GPTQ_ERR_CUDA", 6: "GPTQ_ERR_TIMEOUT"}

# name -> (restype, argtypes); the full exported surface of the header.
_P, _I, _D, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_size_t
SIGNATURES = {
    "gptq_status_string": (ctypes.c_char_p, [_I]),
    "gptq_fold_workspace_bytes": (_S, [_I]),
    "gptq_fold": (_I, [_P, _I, _D, _P, _P, _P, _P, _P, _S, _P]),
    "gptq_ladder": (_I, [_P, _I, _I, _P, _P, _P]),
    "gptq_sweep_workspace_bytes": (_S, [_I, _I]),
    "gptq_q4tp_sweep": (_I, [_P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _S, _P]),
    "gptq_q4tp_group": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "gptq_q4tp_sweep_noalloc": (_I, [_P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "gptq_group_workspace_bytes": (_S, [_I, _I]),
    "gptq_quantize_group": (_I, [_P, _I, _D, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _S, _P]),
    "gptq_build_equilibrated": (_I, [_P, _I, _D, _P, _P, _P, _S, _P]),
    "gptq_act_order_perm": (_I, [_P, _I, _P, _P]),
    "gptq_fold_permuted": (_I, [_P, _I, _D, _P, _P, _P, _P, _P, _P, _S, _P]),
    "gptq_static_rungs": (_I, [_P, _I, _I, _P, _P, _P, _P, _P]),
    "gptq_sweep_act_order_workspace_bytes": (_S, [_I, _I]),
    "gptq_q4tp_sweep_act_order": (_I, [_P, _I, _I, _P, _P, _P, _P, _P, _P, _S, _P]),
    "gptq_group_act_order_workspace_bytes": (_S, [_I, _I]),
    "gptq_quantize_group_act_order": (_I, [_P, _I, _D, _P, _I, _P, _P, _P, _P, _P, _P, _P, _S, _P]),
    "gptq_q2tp_place": (_I, [_P, _I, _I, _P, _P, _P, _P, _P]),
    "gptq_q2tp_group": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P]),
    "gptq_q2tp_sweep": (_I, [_P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _S, _P]),
    "gptq_quantize_group_q2tp": (_I, [_P, _I, _D, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _S, _P]),
    "gptq_debias_workspace_bytes": (_S, [_I, _I]),
    "gptq_debias": (_I, [_I, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _S, _P]),
    "gptq_gram_workspace_bytes": (_S, [_I]),
    "gptq_gram_add": (_I, [_P, _I, _P, _I, _P, _S, _P]),
    "gptq_launch_count": (ctypes.c_longlong, []),
    "gptq_kernel_kinds": (_I, []),
    "gptq_kernel_kind_name": (ctypes.c_char_p, [_I]),
    "gptq_profile_select": (None, [ctypes.c_uint]),
    "gptq_profile_start": (_I, [_I]),
    "gptq_profile_stop": (_I, [_P, _P, _I]),
    "gptq_test_set_wait": (_I, [ctypes.c_ulonglong, _I]),
}


class GptqError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__(f"{fn}: {STATUS.get(code, code)}")


_lib = None


def load(path: str = LIB_PATH):
    """Load the library (built by ``gptq_post_weight_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m gptq_post_weight_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _ptr(t):
    """Device address of a CUDA tensor (None -> NULL).  Taken when the
    library call's arguments are built, after every size check."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"tensor arguments must be CUDA tensors, got one on {t.device}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(torch, stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, code):
    if code != 0:
        raise GptqError(fn, code)


def _need(t, name, dtype=None, numel=None, device=None):
    """Raise ValueError unless ``t`` is a contiguous tensor of ``dtype``
    (default float32) with ``numel`` elements on ``device``.  The kernels
    index every buffer by the sizes the call states, so a buffer of another
    size is refused here, before anything is launched (that it lives on the
    GPU is checked by ``_ptr``)."""
    import torch

    dtype = torch.float32 if dtype is None else dtype
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()} (shape {tuple(t.shape)})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the call's data on {device}")


def _matrix(w, name="w", n=None):
    """rows, n of a 2-D float32 matrix (n checked when given)."""
    _need(w, name)
    if w.dim() != 2:
        raise ValueError(f"{name} must be 2-D [rows, n], got shape {tuple(w.shape)}")
    if n is not None and w.shape[1] != n:
        raise ValueError(f"{name} has {w.shape[1]} columns, n = {n}")
    return w.shape[0], w.shape[1]


def _packed(h_packed, n, device=None):
    _need(h_packed, "h_packed", numel=n * (n + 1) // 2 if n > 0 else None, device=device)


def _ws(ws, device):
    import torch

    _need(ws, "ws", dtype=torch.uint8, device=device)


def _check_outs(out, names, sizes, dtypes, device):
    if len(out) != len(names):
        raise ValueError(f"out must hold {len(names)} tensors ({', '.join(names)})")
    for t, nm, k, dt in zip(out, names, sizes, dtypes):
        _need(t, nm, dtype=dt, numel=k, device=device)


def workspace(nbytes: int, device):
    import torch

    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def fold(h_packed, n: int, lam: float = 0.01, ws=None, stream=None, want_d=True):
    """U [n, n], D [n], hdiag [n], lambda_used.  Raises GptqError(NOT_SPD)."""
    import torch

    lib = load()
    _packed(h_packed, n)
    dev = h_packed.device
    u = torch.empty(n, n, dtype=torch.float32, device=dev)
    d = torch.empty(n, dtype=torch.float32, device=dev) if want_d else None
    hd = torch.empty(n, dtype=torch.float32, device=dev)
    need = lib.gptq_fold_workspace_bytes(n)
    if ws is None:
        ws = workspace(need, dev)
    _ws(ws, dev)
    lam_used = ctypes.c_double(0.0)
    code = lib.gptq_fold(_ptr(h_packed), n, float(lam), _ptr(u), _ptr(d), _ptr(hd),
                         ctypes.byref(lam_used), _ptr(ws), ws.numel(), _stream(torch, stream))
    _check("gptq_fold", code)
    return u, d, hd, lam_used.value


def build_equilibrated(h_packed, n: int, lam: float = 0.01):
    import torch

    lib = load()
    _packed(h_packed, n)
    dev = h_packed.device
    a = torch.zeros(n, n, dtype=torch.float32, device=dev)
    d = torch.empty(n, dtype=torch.float32, device=dev)
    ws = workspace(lib.gptq_fold_workspace_bytes(n), dev)
    code = lib.gptq_build_equilibrated(_ptr(h_packed), n, float(lam), _ptr(a), _ptr(d), _ptr(ws),
                                       ws.numel(), _stream(torch))
    _check("gptq_build_equilibrated", code)
    return a, d


def ladder(w):
    import torch

    lib = load()
    rows, n = _matrix(w)
    tab = torch.empty(rows, 32, dtype=torch.float32, device=w.device)
    lost = torch.empty(rows, 2, dtype=torch.float32, device=w.device)
    _check("gptq_ladder", lib.gptq_ladder(_ptr(w), rows, n, _ptr(tab), _ptr(lost), _stream(torch)))
    return tab, lost


def _outs(torch, rows, n, dev, out=None):
    gpr = n // 32
    if out is not None:
        _check_outs(out, ("nibbles", "rungs", "scales"), (rows * n // 2, rows * gpr, rows * gpr),
                    (torch.uint8, torch.uint8, torch.float32), dev)
        return out
    nib = torch.empty(rows * n // 2, dtype=torch.uint8, device=dev)
    rungs = torch.empty(rows * gpr, dtype=torch.uint8, device=dev)
    scales = torch.empty(rows * gpr, dtype=torch.float32, device=dev)
    return nib, rungs, scales


def _sweep_inputs(w, u, hw, tab, lost=None):
    """rows, n after checking W [rows, n], U n*n, hw n, tab rows*32, lost rows*2."""
    rows, n = _matrix(w)
    dev = w.device
    _need(u, "u", numel=n * n, device=dev)
    _need(hw, "hw", numel=n, device=dev)
    _need(tab, "tab", numel=rows * 32, device=dev)
    if lost is not None:
        _need(lost, "lost", numel=rows * 2, device=dev)
    return rows, n


def q4tp_sweep(w, u, hw, tab, lost, ws=None, out=None, stream=None):
    """Sweep W (consumed in place).  Returns (nibbles, rungs, scales)."""
    import torch

    lib = load()
    rows, n = _sweep_inputs(w, u, hw, tab, lost)
    nib, rungs, scales = _outs(torch, rows, n, w.device, out)
    if ws is None:
        ws = workspace(lib.gptq_sweep_workspace_bytes(rows, n), w.device)
    _ws(ws, w.device)
    code = lib.gptq_q4tp_sweep(_ptr(w), rows, n, _ptr(u), _ptr(hw), _ptr(tab), _ptr(lost),
                               _ptr(nib), _ptr(rungs), _ptr(scales), _ptr(ws), ws.numel(),
                               _stream(torch, stream))
    _check("gptq_q4tp_sweep", code)
    return nib, rungs, scales


def q4tp_sweep_noalloc(w, u, hw, tab, lost, out=None, stream=None):
    """gptq_q4tp_sweep_noalloc: the sweep with the library's own static
    scratch instead of a workspace (for callers that cannot allocate device
    memory).  Returns (nibbles, rungs, scales); W is consumed in place."""
    import torch

    lib = load()
    rows, n = _sweep_inputs(w, u, hw, tab, lost)
    nib, rungs, scales = _outs(torch, rows, n, w.device, out)
    code = lib.gptq_q4tp_sweep_noalloc(_ptr(w), rows, n, _ptr(u), _ptr(hw), _ptr(tab), _ptr(lost),
                                       _ptr(nib), _ptr(rungs), _ptr(scales), _stream(torch, stream))
    _check("gptq_q4tp_sweep_noalloc", code)
    return nib, rungs, scales


def _group_inputs(tile, ublk, hw, tab, lost=None):
    """rows after checking tile [rows, 32], ublk 32*32, hw 32, tab rows*32, lost rows*2."""
    rows, c = _matrix(tile, "tile")
    if c != 32:
        raise ValueError(f"tile must be [rows, 32], got shape {tuple(tile.shape)}")
    dev = tile.device
    _need(ublk, "ublk", numel=32 * 32, device=dev)
    _need(hw, "hw", numel=32, device=dev)
    _need(tab, "tab", numel=rows * 32, device=dev)
    if lost is not None:
        _need(lost, "lost", numel=rows * 2, device=dev)
    return rows


def q4tp_group(tile, ublk, hw, tab, lost):
    """The group rule on given tiles: (nibbles [rows,16], rungs, scales, E)."""
    import torch

    lib = load()
    rows = _group_inputs(tile, ublk, hw, tab, lost)
    dev = tile.device
    nib = torch.empty(rows, 16, dtype=torch.uint8, device=dev)
    rungs = torch.empty(rows, dtype=torch.uint8, device=dev)
    scales = torch.empty(rows, dtype=torch.float32, device=dev)
    e = torch.empty(rows, 32, dtype=torch.float32, device=dev)
    code = lib.gptq_q4tp_group(_ptr(tile), rows, _ptr(ublk), _ptr(hw), _ptr(tab), _ptr(lost),
                               _ptr(nib), _ptr(rungs), _ptr(scales), _ptr(e), _stream(torch))
    _check("gptq_q4tp_group", code)
    return nib, rungs, scales, e


def quantize_group(h_packed, n, w, lam=0.01, ws=None, want_u=True, stream=None, out=None, want_aux=True):
    """Fold + ladder + sweep.  Returns dict(nibbles, rungs, scales, tab, lost,
    u, d, hdiag, lam); with want_aux=False, tab, lost, d and hdiag stay in the
    workspace (None here), so that repeated calls on the same buffers pass the
    library the same arguments (its graph replay keys on them)."""
    import torch

    lib = load()
    rows, _ = _matrix(w, n=n)
    dev = w.device
    _packed(h_packed, n, dev)
    nib, rungs, scales = _outs(torch, rows, n, dev, out)
    tab = torch.empty(rows, 32, dtype=torch.float32, device=dev) if want_aux else None
    lost = torch.empty(rows, 2, dtype=torch.float32, device=dev) if want_aux else None
    u = torch.empty(n, n, dtype=torch.float32, device=dev) if want_u else None
    d = torch.empty(n, dtype=torch.float32, device=dev) if want_aux else None
    hd = torch.empty(n, dtype=torch.float32, device=dev) if want_aux else None
    if ws is None:
        ws = workspace(lib.gptq_group_workspace_bytes(rows, n), dev)
    _ws(ws, dev)
    lam_used = ctypes.c_double(0.0)
    code = lib.gptq_quantize_group(_ptr(h_packed), n, float(lam), _ptr(w), rows, _ptr(nib),
                                   _ptr(rungs), _ptr(scales), _ptr(tab), _ptr(lost), _ptr(u),
                                   _ptr(d), _ptr(hd), ctypes.byref(lam_used), _ptr(ws), ws.numel(),
                                   _stream(torch, stream))
    _check("gptq_quantize_group", code)
    return dict(nibbles=nib, rungs=rungs, scales=scales, tab=tab, lost=lost, u=u, d=d, hdiag=hd,
                lam=lam_used.value)


def test_set_wait(wait_ns: int = 0, no_loads: bool = False):
    """gptq_test_set_wait: the device-wait limit in ns (0 = the default 2 s)
    and the test hook that makes the GEMM producers issue no loads."""
    _check("gptq_test_set_wait", load().gptq_test_set_wait(int(wait_ns), 1 if no_loads else 0))


def launch_count() -> int:
    return int(load().gptq_launch_count())


def profile_start(max_launches: int = 100000, kinds=None):
    """Record events for the launches that follow; `kinds`: names to record
    (default all)."""
    lib = load()
    mask = 0xFFFFFFFF
    if kinds is not None:
        names = [lib.gptq_kernel_kind_name(k).decode() for k in range(lib.gptq_kernel_kinds())]
        mask = 0
        for name in kinds:
            mask |= 1 << names.index(name)
    lib.gptq_profile_select(mask)
    _check("gptq_profile_start", lib.gptq_profile_start(int(max_launches)))


def profile_stop():
    """{kind name: (total ms, launches)} for the launches since profile_start."""
    lib = load()
    nk = lib.gptq_kernel_kinds()
    ms = (ctypes.c_double * nk)()
    cnt = (ctypes.c_longlong * nk)()
    r = lib.gptq_profile_stop(ms, cnt, nk)
    if r == -1:
        raise GptqError("gptq_profile_stop", 5)
    out = {lib.gptq_kernel_kind_name(k).decode(): (ms[k], cnt[k]) for k in range(nk)}
    if r == -2:
        out["_truncated"] = (0.0, 1)
    return out


def gram_add(h_packed, x, ws=None, stream=None):
    """H_packed += X^T X in place (X [T, n] f32); returns h_packed."""
    import torch

    lib = load()
    t, n = _matrix(x, "x")
    _packed(h_packed, n, x.device)
    if ws is None:
        ws = workspace(lib.gptq_gram_workspace_bytes(n), x.device)
    _ws(ws, x.device)
    code = lib.gptq_gram_add(_ptr(h_packed), n, _ptr(x), t, _ptr(ws), ws.numel(), _stream(torch, stream))
    _check("gptq_gram_add", code)
    return h_packed


def act_order_perm(hdiag):
    import torch

    lib = load()
    _need(hdiag, "hdiag")
    n = hdiag.numel()
    perm = torch.empty(n, dtype=torch.int32, device=hdiag.device)
    _check("gptq_act_order_perm", lib.gptq_act_order_perm(_ptr(hdiag), n, _ptr(perm), _stream(torch)))
    return perm


def fold_permuted(h_packed, n, perm, lam=0.01):
    """U, D, hdiag (permuted order), lambda_used of H[perm][perm]."""
    import torch

    lib = load()
    _packed(h_packed, n)
    dev = h_packed.device
    _need(perm, "perm", dtype=torch.int32, numel=n, device=dev)
    u = torch.empty(n, n, dtype=torch.float32, device=dev)
    d = torch.empty(n, dtype=torch.float32, device=dev)
    hd = torch.empty(n, dtype=torch.float32, device=dev)
    ws = workspace(lib.gptq_fold_workspace_bytes(n), dev)
    lam_used = ctypes.c_double(0.0)
    code = lib.gptq_fold_permuted(_ptr(h_packed), n, float(lam), _ptr(perm), _ptr(u), _ptr(d), _ptr(hd),
                                  ctypes.byref(lam_used), _ptr(ws), ws.numel(), _stream(torch))
    _check("gptq_fold_permuted", code)
    return u, d, hd, lam_used.value


def static_rungs(w, tab, lost):
    import torch

    lib = load()
    rows, n = _matrix(w)
    _need(tab, "tab", numel=rows * 32, device=w.device)
    _need(lost, "lost", numel=rows * 2, device=w.device)
    rungs = torch.empty(rows * (n // 32), dtype=torch.uint8, device=w.device)
    scales = torch.empty(rows * (n // 32), dtype=torch.float32, device=w.device)
    code = lib.gptq_static_rungs(_ptr(w), rows, n, _ptr(tab), _ptr(lost), _ptr(rungs), _ptr(scales),
                                 _stream(torch))
    _check("gptq_static_rungs", code)
    return rungs, scales


def q4tp_sweep_act_order(w, u, perm, tab, rungs):
    import torch

    lib = load()
    rows, n = _matrix(w)
    dev = w.device
    _need(u, "u", numel=n * n, device=dev)
    _need(perm, "perm", dtype=torch.int32, numel=n, device=dev)
    _need(tab, "tab", numel=rows * 32, device=dev)
    _need(rungs, "rungs", dtype=torch.uint8, numel=rows * (n // 32), device=dev)
    nib = torch.empty(rows * n // 2, dtype=torch.uint8, device=w.device)
    ws = workspace(lib.gptq_sweep_act_order_workspace_bytes(rows, n), w.device)
    code = lib.gptq_q4tp_sweep_act_order(_ptr(w), rows, n, _ptr(u), _ptr(perm), _ptr(tab), _ptr(rungs),
                                         _ptr(nib), _ptr(ws), ws.numel(), _stream(torch))
    _check("gptq_q4tp_sweep_act_order", code)
    return nib


def quantize_group_act_order(h_packed, n, w, lam=0.01, ws=None, want_u=True, stream=None):
    import torch

    lib = load()
    rows, _ = _matrix(w, n=n)
    dev = w.device
    _packed(h_packed, n, dev)
    nib, rungs, scales = _outs(torch, rows, n, dev)
    perm = torch.empty(n, dtype=torch.int32, device=dev)
    u = torch.empty(n, n, dtype=torch.float32, device=dev) if want_u else None
    if ws is None:
        ws = workspace(lib.gptq_group_act_order_workspace_bytes(rows, n), dev)
    _ws(ws, dev)
    lam_used = ctypes.c_double(0.0)
    code = lib.gptq_quantize_group_act_order(_ptr(h_packed), n, float(lam), _ptr(w), rows, _ptr(nib),
                                             _ptr(rungs), _ptr(scales), _ptr(perm), _ptr(u),
                                             ctypes.byref(lam_used), _ptr(ws), ws.numel(),
                                             _stream(torch, stream))
    _check("gptq_quantize_group_act_order", code)
    return dict(nibbles=nib, rungs=rungs, scales=scales, perm=perm, u=u, lam=lam_used.value)


# ------------------------------------------------------------------ q2tp


def q2tp_place(w, hw, want_gscale=False):
    """Placed q2tp ladder of the (dead-zeroed) W: (tab [rows, 32], lost
    [rows, 2], gscale [rows, n/32] or None)."""
    import torch

    lib = load()
    rows, n = _matrix(w)
    _need(hw, "hw", numel=n, device=w.device)
    tab = torch.empty(rows, 32, dtype=torch.float32, device=w.device)
    lost = torch.empty(rows, 2, dtype=torch.float32, device=w.device)
    gs = torch.empty(rows, n // 32, dtype=torch.float32, device=w.device) if want_gscale else None
    _check("gptq_q2tp_place", lib.gptq_q2tp_place(_ptr(w), rows, n, _ptr(hw), _ptr(tab), _ptr(lost),
                                                  _ptr(gs), _stream(torch)))
    return tab, lost, gs


def q2tp_group(tile, ublk, hw, tab):
    """The q2tp group rule on given tiles: (codes [rows, 8] u8, rungs, scales, E)."""
    import torch

    lib = load()
    rows = _group_inputs(tile, ublk, hw, tab)
    dev = tile.device
    codes = torch.empty(rows, 8, dtype=torch.uint8, device=dev)
    rungs = torch.empty(rows, dtype=torch.uint8, device=dev)
    scales = torch.empty(rows, dtype=torch.float32, device=dev)
    e = torch.empty(rows, 32, dtype=torch.float32, device=dev)
    code = lib.gptq_q2tp_group(_ptr(tile), rows, _ptr(ublk), _ptr(hw), _ptr(tab), _ptr(codes),
                               _ptr(rungs), _ptr(scales), _ptr(e), _stream(torch))
    _check("gptq_q2tp_group", code)
    return codes, rungs, scales, e


def _outs_q2(torch, rows, n, dev, out=None):
    gpr = n // 32
    if out is not None:
        _check_outs(out, ("codes", "rungs", "scales"), (rows * n // 4, rows * gpr, rows * gpr),
                    (torch.uint8, torch.uint8, torch.float32), dev)
        return out
    codes = torch.empty(rows * n // 4, dtype=torch.uint8, device=dev)
    rungs = torch.empty(rows * gpr, dtype=torch.uint8, device=dev)
    scales = torch.empty(rows * gpr, dtype=torch.float32, device=dev)
    return codes, rungs, scales


def q2tp_sweep(w, u, hw, tab, ws=None, out=None, stream=None):
    """q2tp sweep of W (consumed in place).  Returns (codes, rungs, scales)."""
    import torch

    lib = load()
    rows, n = _sweep_inputs(w, u, hw, tab)
    codes, rungs, scales = _outs_q2(torch, rows, n, w.device, out)
    if ws is None:
        ws = workspace(lib.gptq_sweep_workspace_bytes(rows, n), w.device)
    _ws(ws, w.device)
    code = lib.gptq_q2tp_sweep(_ptr(w), rows, n, _ptr(u), _ptr(hw), _ptr(tab), _ptr(codes),
                               _ptr(rungs), _ptr(scales), _ptr(ws), ws.numel(), _stream(torch, stream))
    _check("gptq_q2tp_sweep", code)
    return codes, rungs, scales


def quantize_group_q2tp(h_packed, n, w, lam=0.01, ws=None, want_u=True, stream=None, out=None,
                        want_aux=True):
    """Fold + placed ladder + q2tp sweep.  Returns dict(codes, rungs, scales,
    tab, lost, u, d, hdiag, lam); want_aux as for quantize_group."""
    import torch

    lib = load()
    rows, _ = _matrix(w, n=n)
    dev = w.device
    _packed(h_packed, n, dev)
    codes, rungs, scales = _outs_q2(torch, rows, n, dev, out)
    tab = torch.empty(rows, 32, dtype=torch.float32, device=dev) if want_aux else None
    lost = torch.empty(rows, 2, dtype=torch.float32, device=dev) if want_aux else None
    u = torch.empty(n, n, dtype=torch.float32, device=dev) if want_u else None
    d = torch.empty(n, dtype=torch.float32, device=dev) if want_aux else None
    hd = torch.empty(n, dtype=torch.float32, device=dev) if want_aux else None
    if ws is None:
        ws = workspace(lib.gptq_group_workspace_bytes(rows, n), dev)
    _ws(ws, dev)
    lam_used = ctypes.c_double(0.0)
    code = lib.gptq_quantize_group_q2tp(_ptr(h_packed), n, float(lam), _ptr(w), rows, _ptr(codes),
                                        _ptr(rungs), _ptr(scales), _ptr(tab), _ptr(lost), _ptr(u),
                                        _ptr(d), _ptr(hd), ctypes.byref(lam_used), _ptr(ws),
                                        ws.numel(), _stream(torch, stream))
    _check("gptq_quantize_group_q2tp", code)
    return dict(codes=codes, rungs=rungs, scales=scales, tab=tab, lost=lost, u=u, d=d, hdiag=hd,
                lam=lam_used.value)


def debias(bits, w, h_packed, codes, rungs, tab, lost, scales, ws=None, want_num_den=False, stream=None):
    """Output debias (in place on tab, lost, scales).  Returns num_den [rows, 2]
    f64 or None."""
    import torch

    lib = load()
    rows, n = _matrix(w)
    dev = w.device
    _packed(h_packed, n, dev)
    if int(bits) in (2, 4):
        gpr = n // 32
        _need(codes, "codes", dtype=torch.uint8, numel=rows * n * int(bits) // 8, device=dev)
        _need(rungs, "rungs", dtype=torch.uint8, numel=rows * gpr, device=dev)
        _need(tab, "tab", numel=rows * 32, device=dev)
        _need(lost, "lost", numel=rows * 2, device=dev)
        _need(scales, "scales", numel=rows * gpr, device=dev)
    nd = torch.empty(rows, 2, dtype=torch.float64, device=w.device) if want_num_den else None
    if ws is None:
        ws = workspace(lib.gptq_debias_workspace_bytes(rows, n), w.device)
    _ws(ws, dev)
    code = lib.gptq_debias(int(bits), _ptr(w), rows, n, _ptr(h_packed), _ptr(codes), _ptr(rungs), _ptr(tab),
                           _ptr(lost), _ptr(scales), _ptr(nd), _ptr(ws), ws.numel(), _stream(torch, stream))
    _check("gptq_debias", code)
    return nd
