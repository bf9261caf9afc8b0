"""The identity the sibling-recursive acceptance kernel evaluates (CPU only, numpy).

After k rejected siblings the target becomes r_k = norm([r_{k-1} - q]+) (hncyxsy.com
sections 2.1-2.2, applied once per candidate), starting from r_0 = p.  The kernel keeps
r_k as [p - c_k q]+ / n_k with c_0 = 0, n_0 = 1, c_k = c_{k-1} + n_{k-1},
n_k = sum [p - c_k q]+, and keeps (c, n) unchanged when that sum is zero.  The test
iterates the definition and checks the closed form against it, including the empty case.
"""
import numpy as np
import pytest


def _iterate(p, q, k):
    r = p.copy()
    for _ in range(k):
        w = np.maximum(r - q, 0.0)
        if w.sum() > 0.0:
            r = w / w.sum()
    return r


def _closed(p, q, k):
    c, n = 0.0, 1.0
    for _ in range(k):
        c1 = c + n
        tot = np.maximum(p - c1 * q, 0.0).sum()
        if tot > 0.0:
            c, n = c1, tot
    return np.maximum(p - c * q, 0.0) / n


@pytest.mark.parametrize("V,k,seed", [(16, 1, 0), (16, 3, 1), (1000, 5, 2), (64, 8, 3)])
def test_closed_form_equals_iterated_residual(V, k, seed):
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.full(V, 0.5))
    q = rng.dirichlet(np.full(V, 0.5))
    a, b = _iterate(p, q, k), _closed(p, q, k)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-15)
    assert abs(b.sum() - 1.0) < 1e-12


def test_empty_residual_keeps_the_previous_one():
    # q dominates p everywhere after one step: [r_1 - q]+ has no mass, r stays r_1
    p = np.array([0.6, 0.4, 0.0, 0.0])
    q = np.array([0.5, 0.5, 0.0, 0.0])
    r1 = _iterate(p, q, 1)
    assert np.allclose(r1, [1.0, 0.0, 0.0, 0.0])
    assert np.allclose(_iterate(p, q, 3), r1)
    assert np.allclose(_closed(p, q, 3), r1)


def test_a_wrong_coefficient_is_caught():
    # the tempting c_k = k (subtract q once per rejection, unnormalised) differs
    rng = np.random.default_rng(9)
    p = rng.dirichlet(np.full(32, 0.5))
    q = rng.dirichlet(np.full(32, 0.5))
    w = np.maximum(p - 2.0 * q, 0.0)
    assert not np.allclose(w / w.sum(), _iterate(p, q, 2))
