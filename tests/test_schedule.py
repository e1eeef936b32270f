"""The per-step minimax schedule of the coupled iteration (host only, through
the C ABI): each step's polynomial T_k must map the interval [lo_k, 1] holding
M_k's spectrum into [lo_(k+1), 1] with its top at 1, stay positive without
folding, and the composed steps must take every m in [lo_0, 1] to 1 while the
product of the T_k reaches m^(-1/p).  Checked by dense float64 evaluation of
the scalar model, independent of how the schedule was optimised."""
import numpy as np
import pytest

import shampoo_roots_gb300 as sr

L0 = 1e-6 / (1.01 * (1 + 1024 * 1e-6))      # the start interval of a d = 1024 root, eps = 1e-6


def _grid(lo):
    return np.unique(np.concatenate([np.geomspace(lo, 1.0, 20001), np.linspace(lo, 1.0, 20001)]))


def _T(a, b, c, m):
    return a - b * m + c * m * m


@pytest.mark.parametrize("p,degree", [(4, 1), (4, 2), (2, 1), (2, 2)])
def test_each_step_maps_its_interval_into_the_next(p, degree):
    a, b, c, lo = sr.precond_step_schedule(p, L0, 0.3, degree)
    assert len(a) >= 5
    if degree == 1:
        assert all(x == 0.0 for x in c)
    for k in range(len(a)):
        m = _grid(lo[k])
        t = _T(a[k], b[k], c[k], m)
        g = m * t ** p
        assert t.min() > 0
        assert t.min() >= 0.3 * t.max() * (1 - 1e-9)             # no fold past the cap
        assert g.max() <= 1 + 1e-9 and g.max() >= 1 - 1e-6       # the top lands at 1
        nxt = lo[k + 1] if k + 1 < len(a) else None
        if nxt is not None:
            assert g.min() >= nxt * (1 - 1e-9)                    # the new bottom is a true bound
            assert g.min() <= nxt * (1 + 1e-4)                    # and a tight one
            assert nxt > lo[k]
    assert 1 - lo[-1] < 1e-3


@pytest.mark.parametrize("p,degree", [(4, 1), (4, 2), (2, 1)])
def test_composed_steps_reach_the_inverse_root(p, degree):
    """m_(k+1) = m_k T_k(m_k)^p from every m_0 in [lo_0, 1] ends at 1, and
    x = prod T_k(m_k) ends at m_0^(-1/p) (the scalar coupled iteration,
    M = X^p M_0)."""
    a, b, c, lo = sr.precond_step_schedule(p, L0, 0.3, degree)
    m0 = _grid(lo[0])
    m, x = m0.copy(), np.ones_like(m0)
    for k in range(len(a)):
        t = _T(a[k], b[k], c[k], m)
        x *= t
        m *= t ** p
    # classical Newton steps finish what the schedule leaves (as the library does)
    for _ in range(3):
        t = ((p + 1) - m) / p
        x *= t
        m *= t ** p
    assert np.max(np.abs(m - 1)) < 1e-9
    assert np.max(np.abs(x * m0 ** (1.0 / p) - 1)) < 1e-9


def test_quadratic_steps_need_fewer_products_at_p4():
    """Products per iteration: 4 (linear T) or 5 (quadratic T) at p = 4."""
    lin = sr.precond_step_schedule(4, L0, 0.3, 1)[0]
    quad = sr.precond_step_schedule(4, L0, 0.3, 2)[0]
    assert len(lin) == 10 and len(quad) == 7
    assert 5 * len(quad) < 4 * len(lin)


def test_schedule_rejects_bad_arguments():
    lib = sr.load()
    import ctypes
    arr = [(ctypes.c_double * 4)() for _ in range(4)]
    n = ctypes.c_int()
    assert lib.precond_step_schedule(3, L0, 0.3, 1, 4, *arr, ctypes.byref(n)) == sr.EINVAL
    assert lib.precond_step_schedule(4, 0.0, 0.3, 1, 4, *arr, ctypes.byref(n)) == sr.EINVAL
    assert lib.precond_step_schedule(4, L0, 1.0, 1, 4, *arr, ctypes.byref(n)) == sr.EINVAL
    assert lib.precond_step_schedule(4, L0, 0.3, 3, 4, *arr, ctypes.byref(n)) == sr.EINVAL
    assert lib.precond_step_schedule(4, L0, 0.3, 2, 4, *arr, ctypes.byref(n)) == sr.OK
    assert n.value == 4
