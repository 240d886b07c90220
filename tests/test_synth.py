"""The seeded input generator draws what its recipe says (CPU only).

Both sides of every parity check consume these bytes, so the recipe itself
is pinned here: the channel plan (dead and outlier channels, lognormal
scales), the packed-upper layout of H, the structure H must have (symmetric,
dead rows and columns zero, diagonal near the squared channel scale, rank at
most T), the weight distribution, and determinism per seed.
"""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")


def small(**kw):
    return synth.config("tiny", **kw)


def test_channel_plan():
    cfg = small()
    scale, outl, dead = synth.channel_plan(cfg)
    assert len(dead) == cfg.n_dead and len(outl) == cfg.n_outlier
    assert not set(dead.tolist()) & set(outl.tolist())
    assert torch.all(scale[dead] == 0)
    live = torch.ones(cfg.n, dtype=torch.bool)
    live[dead] = False
    live[outl] = False
    # Ordinary channels: lognormal(0, sigma).  Outliers: 100x such a draw,
    # i.e. log-scale 4.6 higher on average (not above every ordinary channel).
    lg = torch.log(scale[live].double())
    assert abs(lg.mean().item()) < 0.3 and abs(lg.std().item() - cfg.sigma) < 0.2
    assert torch.log(scale[outl].double()).mean().item() > lg.mean().item() + 3.0


def test_pack_upper_layout():
    n = 7
    h = torch.arange(n * n, dtype=torch.float32).reshape(n, n)
    p = synth.pack_upper(h)
    assert p.numel() == n * (n + 1) // 2
    for r in range(n):
        off = r * (2 * n - r + 1) // 2
        assert torch.equal(p[off : off + n - r], h[r, r:])


def test_hessian_structure():
    cfg = small(T=4096)
    x = synth.make_x(cfg)
    h = synth.make_h(cfg)
    scale, outl, dead = synth.channel_plan(cfg)
    assert torch.equal(h, h.T)
    assert torch.all(h[dead] == 0) and torch.all(h[:, dead] == 0)
    # E[x^2] = 1 per unit-scale sample: H_ii / scale_i^2 is a chi-square mean over T.
    live = scale > 0
    ratio = (torch.diagonal(h)[live] / scale[live] ** 2).double()
    assert torch.all((ratio - 1).abs() < 6 * np.sqrt(2 / cfg.T))
    # H is X X^T / T of the same draw.
    ref = (x.double() @ x.double().T) / cfg.T
    assert torch.allclose(h.double(), ref, rtol=1e-4, atol=1e-6 * ref.abs().max().item())
    hp = synth.make_h_packed(cfg)
    assert torch.equal(hp, synth.pack_upper(h))


def test_rank_deficient():
    cfg = synth.rank_deficient(small())
    assert cfg.T == cfg.n // 2
    h = synth.make_h(cfg).double()
    ev = torch.linalg.eigvalsh(h)
    # At most T nonzero eigenvalues: the lowest n - T are round-off.
    assert ev[: cfg.n - cfg.T].abs().max().item() <= 1e-5 * ev[-1].item()
    assert ev[cfg.n - cfg.T :].min().item() > 0


def test_weights_and_determinism():
    cfg = small()
    w = synth.make_w(cfg)
    assert w.shape == (cfg.rows, cfg.n) and w.dtype == torch.float32
    assert abs(w.double().std().item() / cfg.w_std - 1) < 0.02
    assert abs(w.double().mean().item()) < 4 * cfg.w_std / np.sqrt(w.numel())
    hp1, w1 = synth.make_problem(cfg)
    hp2, w2 = synth.make_problem(cfg)
    assert torch.equal(hp1, hp2) and torch.equal(w1, w2)
    hp3, w3 = synth.make_problem(small(seed=1))
    assert not torch.equal(w1, w3) and not torch.equal(hp1, hp3)
