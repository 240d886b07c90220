"""Pins for the oracle Gram accumulation (CPU only): brute force over tokens
(sum of outer products, element by element), the packed layout against the
fold page's row-offset formula, chunked accumulation, and a closed form."""
import numpy as np

import oracle


def test_bruteforce_outer_products():
    rng = np.random.default_rng(0)
    t, n = 7, 5
    x = rng.standard_normal((t, n))
    hp0 = rng.standard_normal(n * (n + 1) // 2)
    got = oracle.gram_add(hp0, x)
    k = 0
    for a in range(n):
        for b in range(a, n):
            want = hp0[k] + sum(x[s, a] * x[s, b] for s in range(t))
            assert abs(got[k] - want) < 1e-12
            # offset formula of the packed layout: row a starts at a(2n-a+1)/2
            assert k == a * (2 * n - a + 1) // 2 + (b - a)
            k += 1


def test_chunks_add_up():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((100, 12)).astype(np.float32)
    one = oracle.gram_add(np.zeros(78), x)
    two = oracle.gram_add(oracle.gram_add(np.zeros(78), x[:37]), x[37:])
    np.testing.assert_allclose(two, one, rtol=1e-12, atol=1e-12)


def test_orthogonal_columns_give_diagonal():
    # Columns of X orthogonal with norms c_i: H = diag(c_i^2).
    q, _ = np.linalg.qr(np.random.default_rng(2).standard_normal((16, 6)))
    c = np.array([1.0, 2.0, 0.5, 3.0, 0.0, 1.5])
    x = q * c
    hp = oracle.gram_add(np.zeros(21), x)
    h = oracle.unpack_upper(hp.astype(np.float32), 6)
    np.testing.assert_allclose(h, np.diag(c ** 2), atol=1e-6)
