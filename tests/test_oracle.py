"""CPU tests of the float64 oracle: its pins, and proof that the pins catch
plausible mistakes planted in a copy of the oracle (on the CPU only)."""
import types

import numpy as np
import pytest

import oracle.roots as R
import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(R)


def _impl(**over):
    ns = types.SimpleNamespace(**{k: getattr(R, k) for k in
                                  ("gram_ema", "trace_normalise", "inv_root_eigh", "precondition",
                                   "lambda_max_bound", "coupled_newton_schulz")})
    for k, v in over.items():
        setattr(ns, k, v)
    ns.inv_root = lambda A, eps, power: ns.inv_root_eigh(ns.trace_normalise(A), eps, power)
    return ns


def _eigh_root(transform):
    def f(A_hat, eps, power):
        lam, Q = np.linalg.eigh(np.asarray(A_hat, dtype=np.float64))
        return (Q * transform(lam, eps, power)[None, :]) @ Q.T
    return f


def _ns(mut):
    def f(A, p, tol=1e-12, max_iter=100, scale=None):
        A = np.asarray(A, dtype=np.float64)
        d = A.shape[0]
        c = 1.01 * R.lambda_max_bound(A) if scale is None else scale
        I = np.eye(d)
        M, X = A / c, I.copy()
        k = 0
        while k < max_iter and np.linalg.norm(M - I) > tol:
            T = mut(M, I, p)
            X = X @ T
            M = np.linalg.matrix_power(T, p) @ M
            k += 1
        return 0.5 * (X + X.T) * c ** (-1.0 / p), k, []
    return f


def _ws_only(A):
    A = np.asarray(A, dtype=np.float64)
    n = A.shape[0]
    mu = np.trace(A) / n
    s2 = max(np.sum(A * A) / n - mu * mu, 0.0)
    return mu + np.sqrt(s2)            # missing sqrt(n - 1)


MUTANTS = {
    "eps dropped": dict(inv_root_eigh=_eigh_root(lambda l, e, p: np.maximum(l, 1e-300) ** p)),
    "power sign flipped": dict(inv_root_eigh=_eigh_root(lambda l, e, p: (l + e) ** (-p))),
    "eps multiplied": dict(inv_root_eigh=_eigh_root(lambda l, e, p: (l * (1 + e)) ** p)),
    "power halved": dict(inv_root_eigh=_eigh_root(lambda l, e, p: (l + e) ** (p / 2))),
    "EMA without (1-beta)": dict(gram_ema=lambda L, Rr, G, b: (b * L + G @ G.T, b * Rr + G.T @ G)),
    "EMA left/right swapped": dict(gram_ema=lambda L, Rr, G, b: (b * L + (1 - b) * G.T @ G,
                                                               b * Rr + (1 - b) * G @ G.T)),
    "EMA beta on new term": dict(gram_ema=lambda L, Rr, G, b: ((1 - b) * L + b * G @ G.T,
                                                             (1 - b) * Rr + b * G.T @ G)),
    "rescale by Frobenius": dict(trace_normalise=lambda A: np.asarray(A) / np.linalg.norm(A)),
    "rescale by dimension": dict(trace_normalise=lambda A: np.asarray(A) / np.asarray(A).shape[0]),
    "apply sides swapped": dict(precondition=lambda XL, G, XR: XR @ np.asarray(G) @ XL),
    "apply one-sided": dict(precondition=lambda XL, G, XR: XL @ np.asarray(G)),
    "bound without sqrt(n-1)": dict(lambda_max_bound=_ws_only),
    "bound without abs": dict(lambda_max_bound=lambda A: float(np.max((np.asarray(A) @ np.asarray(A).sum(1))
                                                                      / np.asarray(A).sum(1)))),
    "iteration sign of M": dict(coupled_newton_schulz=_ns(lambda M, I, p: ((p + 1) * I + M) / p)),
    "iteration wrong affine": dict(coupled_newton_schulz=_ns(lambda M, I, p: (p * I - M) / (p - 1))),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    fails = P.failures(_impl(**MUTANTS[name]))
    assert fails, f"no pin caught the planted mistake '{name}'"


def test_oracle_step_small():
    """Whole step on a tiny case: shapes, EMA state kept, X^4 A_reg = I."""
    rng = np.random.default_rng(0)
    st = R.OracleState([(6, 4), (3, 5)])
    for _ in range(2):
        G = [rng.standard_normal((6, 4)), rng.standard_normal((3, 5))]
        U, XL, XR = R.precond_step(st, G, 0.9, 1e-3, -0.25)
    assert U[0].shape == (6, 4) and U[1].shape == (3, 5)
    for L, X in ((st.L[0], XL[0]), (st.R[1], XR[1])):
        Areg = L / np.trace(L) + 1e-3 * np.eye(L.shape[0])
        P._close(np.linalg.matrix_power(X, 4) @ Areg, np.eye(L.shape[0]), 1e-10, "X^4 A = I")


def test_scalar_model_counts():
    # p = 4 counts of the scalar model used for the iteration cap
    assert R.scalar_iterations(1e-6, 4, 1e-7) == 20
    assert R.scalar_iterations(1e-4, 4, 1e-7) == 14
    assert R.scalar_iterations(1e-8, 4, 1e-7) == 25
