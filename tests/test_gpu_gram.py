"""Device Gram accumulation H += X^T X (packed upper) against the f64 oracle.

Tolerance: relative Frobenius error 1e-5.  Each product is taken with the
3xTF32 split (about 2^-21 relative) and summed in f32 over a chunk of up to
4096 tokens, then chunk sums are added in f32; for the shapes below that
bounds the error near 1e-7 relative to ||H||_F, so 1e-5 leaves a wide margin
while still catching any dropped chunk, tile or transposition.
"""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def activations(t, n, seed):
    rng = np.random.default_rng(seed)
    scale = np.exp(rng.standard_normal(n))
    scale[::37] *= 30.0
    scale[5] = 0.0  # a channel that never fires
    x = rng.standard_normal((t, n)) * scale
    return x.astype(np.float32)


@pytest.mark.parametrize("n,t", [(200, 1000), (256, 32), (333, 9000), (1000, 5000)])
def test_gram_add_matches_oracle(lib, n, t):
    from gptq_post_weight_gb300 import _lib

    x = activations(t, n, n + t)
    h0 = np.random.default_rng(1).standard_normal(n * (n + 1) // 2).astype(np.float32)
    hp = torch.from_numpy(h0.copy()).cuda()
    _lib.gram_add(hp, torch.from_numpy(x).cuda())
    want = oracle.gram_add(h0, x)
    got = hp.cpu().numpy()
    assert rel_fro(got, want) <= 1e-5, rel_fro(got, want)
    # the dead channel's row stays as it was
    r = 5
    off = r * (2 * n - r + 1) // 2
    np.testing.assert_allclose(got[off:off + n - r], h0[off:off + n - r], rtol=0, atol=0)


def test_gram_two_windows_equal_one(lib):
    from gptq_post_weight_gb300 import _lib

    n, t = 300, 3000
    x = activations(t, n, 7)
    a = torch.zeros(n * (n + 1) // 2, device="cuda")
    b = torch.zeros_like(a)
    _lib.gram_add(a, torch.from_numpy(x).cuda())
    _lib.gram_add(b, torch.from_numpy(x[:1234]).cuda())
    _lib.gram_add(b, torch.from_numpy(x[1234:]).cuda())
    assert rel_fro(b.cpu().numpy(), a.cpu().numpy()) <= 1e-6


def test_gram_then_fold_chain(lib):
    """Accumulated on the device, the Hessian folds to the oracle's operator
    of the same (oracle-accumulated) Hessian."""
    from gptq_post_weight_gb300 import _lib

    n, t = 384, 2048
    x = activations(t, n, 9)
    hp = torch.zeros(n * (n + 1) // 2, device="cuda")
    _lib.gram_add(hp, torch.from_numpy(x).cuda())
    u, d, hd, lam = _lib.fold(hp, n, 0.01)
    uo = oracle.fold(oracle.gram_add(np.zeros(n * (n + 1) // 2), x).astype(np.float32), n, 0.01)[0]
    assert rel_fro(u.cpu().numpy(), uo) <= 1e-4


@pytest.mark.slow
def test_gram_full_width(lib):
    """A 4096-token window at the n = 17408 width."""
    from gptq_post_weight_gb300 import _lib

    n, t = 17408, 4096
    x = activations(t, n, 11)
    hp = torch.zeros(n * (n + 1) // 2, device="cuda")
    _lib.gram_add(hp, torch.from_numpy(x).cuda())
    want = oracle.gram_add(np.zeros(n * (n + 1) // 2), x)
    assert rel_fro(hp.cpu().numpy(), want) <= 1e-5
