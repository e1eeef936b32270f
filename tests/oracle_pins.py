"""Pins of the float64 oracle against things other than itself.

Each ``pin_*`` function takes an implementation namespace ``impl`` exposing
``gram_ema``, ``trace_normalise``, ``inv_root_eigh``, ``precondition``,
``inv_root``, ``lambda_max_bound`` and ``coupled_newton_schulz`` (the oracle
module, or a copy with a planted mistake) and raises AssertionError when the
implementation disagrees with:

* closed forms (diagonal matrices, the 2 x 2 spectral formula, the EMA sum,
  a rank-one EMA, unit trace, Q diag(lam) Q^T with known lam);
* invariants of the exact root (X^(-1/power) A_reg = I, symmetry, X A = A X);
* brute force (a cyclic Jacobi eigensolver written here, d <= 8);
* the pages: the Appendix D algorithm box of "Online KL Shampoo" at p = 2 and
  its iteration count (section 2.2).
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.max(np.abs(a - b)) / max(1.0, np.max(np.abs(b)))
    assert err <= tol, f"{what}: max rel err {err:.3e} > {tol:.1e}"


def haar_q(d, seed):
    rng = np.random.default_rng(seed)
    q, r = np.linalg.qr(rng.standard_normal((d, d)))
    return q * np.sign(np.diagonal(r))[None, :]


# ---------------------------------------------------------------- roots
def pin_diagonal(impl):
    a = np.array([4.0, 1.0, 0.25, 1e-3, 0.0])
    for power in (-0.25, -0.5):
        for eps in (1e-6, 1e-2):
            X = impl.inv_root(np.diag(a), eps, power)
            want = np.diag((a / a.sum() + eps) ** power)
            _close(X, want, 1e-12, f"diagonal p={power} eps={eps}")


def _f2x2(A, f):
    a, b, c = A[0, 0], A[0, 1], A[1, 1]
    mid = 0.5 * (a + c)
    rad = math.sqrt((0.5 * (a - c)) ** 2 + b * b)
    lp, lm = mid + rad, mid - rad
    I = np.eye(2)
    if rad == 0.0:
        return f(lp) * I
    return (f(lp) * (A - lm * I) - f(lm) * (A - lp * I)) / (lp - lm)


def pin_two_by_two(impl):
    cases = [np.array([[2.0, 0.5], [0.5, 1.0]]), np.array([[1.0, -0.9], [-0.9, 1.0]]),
             np.array([[3.0, 0.0], [0.0, 3.0]]), np.array([[1e-4, 2e-5], [2e-5, 1.0]])]
    for A in cases:
        for power in (-0.25, -0.5):
            eps = 1e-6
            Ah = A / np.trace(A)
            want = _f2x2(Ah, lambda l: (l + eps) ** power)
            _close(impl.inv_root(A, eps, power), want, 1e-10, f"2x2 {A.tolist()} p={power}")


def pin_known_spectrum(impl):
    d = 24
    Q = haar_q(d, 7)
    lam = 10.0 ** np.linspace(-8, 0, d)
    A = (Q * lam[None, :]) @ Q.T
    A = 0.5 * (A + A.T)
    for power in (-0.25, -0.5):
        eps = 1e-6
        want = (Q * ((lam / lam.sum() + eps) ** power)[None, :]) @ Q.T
        _close(impl.inv_root(A, eps, power), want, 1e-9, f"Q diag(lam) Q^T p={power}")


def pin_root_invariants(impl):
    d = 16
    rng = np.random.default_rng(3)
    B = rng.standard_normal((d, 5))
    A = B @ B.T                      # rank 5: eps carries the null space
    for power in (-0.25, -0.5):
        eps = 1e-3
        X = impl.inv_root(A, eps, power)
        Areg = A / np.trace(A) + eps * np.eye(d)
        p = int(round(-1.0 / power))
        _close(np.linalg.matrix_power(X, p) @ Areg, np.eye(d), 1e-10, f"X^{p} A = I")
        _close(X, X.T, 1e-13, "X symmetric")
        _close(X @ Areg, Areg @ X, 1e-12, "X commutes with A")


def jacobi_eigh(A, sweeps=60):
    """Cyclic Jacobi eigenvalue algorithm (pure Python loops; small d)."""
    A = [list(map(float, row)) for row in np.asarray(A)]
    d = len(A)
    V = [[1.0 if i == j else 0.0 for j in range(d)] for i in range(d)]
    for _ in range(sweeps):
        off = sum(A[i][j] ** 2 for i in range(d) for j in range(d) if i != j)
        if off < 1e-30:
            break
        for p in range(d - 1):
            for q in range(p + 1, d):
                if abs(A[p][q]) < 1e-300:
                    continue
                theta = (A[q][q] - A[p][p]) / (2.0 * A[p][q])
                t = (1.0 if theta >= 0 else -1.0) / (abs(theta) + math.sqrt(theta * theta + 1.0))
                c = 1.0 / math.sqrt(t * t + 1.0)
                s = t * c
                for k in range(d):
                    akp, akq = A[k][p], A[k][q]
                    A[k][p] = c * akp - s * akq
                    A[k][q] = s * akp + c * akq
                for k in range(d):
                    apk, aqk = A[p][k], A[q][k]
                    A[p][k] = c * apk - s * aqk
                    A[q][k] = s * apk + c * aqk
                for k in range(d):
                    vkp, vkq = V[k][p], V[k][q]
                    V[k][p] = c * vkp - s * vkq
                    V[k][q] = s * vkp + c * vkq
    return np.array([A[i][i] for i in range(d)]), np.array(V)


def pin_jacobi(impl):
    rng = np.random.default_rng(11)
    for d in (2, 3, 5, 8):
        B = rng.standard_normal((d, d))
        A = B @ B.T + 0.1 * np.eye(d)
        Ah = A / np.trace(A)
        lam, V = jacobi_eigh(Ah)
        for power in (-0.25, -0.5):
            eps = 1e-4
            want = (V * ((lam + eps) ** power)[None, :]) @ V.T
            _close(impl.inv_root_eigh(Ah, eps, power), want, 1e-10, f"Jacobi d={d} p={power}")


def pin_trace(impl):
    rng = np.random.default_rng(5)
    B = rng.standard_normal((9, 4))
    A = B @ B.T
    Ah = impl.trace_normalise(A)
    assert abs(np.trace(Ah) - 1.0) < 1e-14, "unit trace"
    _close(Ah * np.trace(A), A, 1e-14, "rescale is a scalar multiple")


# ---------------------------------------------------------------- EMA
def pin_ema_scalar(impl):
    beta = 0.9
    gs = [1.5, -0.25, 2.0, 0.0, -3.0]
    L = np.zeros((1, 1))
    R = np.zeros((1, 1))
    for t, g in enumerate(gs):
        L, R = impl.gram_ema(L, R, np.array([[g]]), beta)
        want = sum((1 - beta) * beta ** (t - s) * gs[s] ** 2 for s in range(t + 1))
        _close(L, [[want]], 1e-14, "1x1 EMA left")
        _close(R, [[want]], 1e-14, "1x1 EMA right")


def pin_ema_rank_one(impl):
    beta = 0.95
    rng = np.random.default_rng(2)
    u = rng.standard_normal(6)
    u /= np.linalg.norm(u)
    v = rng.standard_normal(4)
    v /= np.linalg.norm(v)
    a = [0.5, 2.0, -1.0]
    L = np.zeros((6, 6))
    R = np.zeros((4, 4))
    for t in range(3):
        L, R = impl.gram_ema(L, R, a[t] * np.outer(u, v), beta)
    w = sum((1 - beta) * beta ** (2 - s) * a[s] ** 2 for s in range(3))
    _close(L, w * np.outer(u, u), 1e-14, "rank-one EMA left (G G^T)")
    _close(R, w * np.outer(v, v), 1e-14, "rank-one EMA right (G^T G)")


# ---------------------------------------------------------------- apply
def pin_apply(impl):
    rng = np.random.default_rng(9)
    m, n = 5, 3
    G = rng.standard_normal((m, n))
    XL = np.diag(np.arange(1.0, m + 1))
    XR = np.diag([10.0, 100.0, 1000.0])
    U = impl.precondition(XL, G, XR)
    want = np.arange(1.0, m + 1)[:, None] * G * np.array([10.0, 100.0, 1000.0])[None, :]
    _close(U, want, 1e-14, "diagonal two-sided apply scales rows by X_L and columns by X_R")


# ---------------------------------------------------------------- bound
def pin_lambda_bound(impl):
    rng = np.random.default_rng(4)
    for d in (2, 7, 30):
        for _ in range(5):
            B = rng.standard_normal((d, d))
            A = B @ B.T
            lmax = np.linalg.eigvalsh(A)[-1]
            bnd = impl.lambda_max_bound(A)
            assert bnd >= lmax * (1 - 1e-12), f"bound {bnd} below lambda_max {lmax}"
    for c in (0.5, 3.0):
        bnd = impl.lambda_max_bound(c * np.eye(6))
        assert abs(bnd - c) < 1e-12, f"bound of {c} I is {bnd}"
    # a diagonal matrix: Minc's bound is exact (max entry), Wolkowicz-Styan is not
    bnd = impl.lambda_max_bound(np.diag([1.0, 2.0, 3.0]))
    assert abs(bnd - 3.0) < 1e-12, f"bound of diag(1,2,3) is {bnd}"


# ---------------------------------------------------------------- iteration
def page_box_inverse_sqrt(S, steps):
    """The Appendix D algorithm box with the classical coefficients
    (a, b) = (3/2, -1/2): Y0 = S/L, Z0 = I, P = Z Y, Q = a I + b P,
    Y <- Y Q, Z <- Q Z, return sym(Z)/sqrt(L); L = 1.01 x bound."""
    d = S.shape[0]
    I = np.eye(d)
    from oracle.roots import lambda_max_bound  # the bound is pinned separately
    Lc = 1.01 * lambda_max_bound(S)
    Y, Z = S / Lc, I.copy()
    for _ in range(steps):
        P = Z @ Y
        Q = 1.5 * I - 0.5 * P
        Y, Z = Y @ Q, Q @ Z
    return 0.5 * (Z + Z.T) / math.sqrt(Lc)


def pin_iteration_p2_is_page_box(impl):
    Q = haar_q(10, 21)
    lam = 10.0 ** np.linspace(-3, 0, 10)
    S = (Q * lam[None, :]) @ Q.T
    for steps in (1, 3, 8):
        X, _, _ = impl.coupled_newton_schulz(S, 2, tol=0.0, max_iter=steps)
        _close(X, page_box_inverse_sqrt(S, steps), 1e-12, f"p=2 iteration == page box ({steps} steps)")


def pin_iteration_converges_to_root(impl):
    Q = haar_q(12, 8)
    lam = 10.0 ** np.linspace(-6, 0, 12)
    A = (Q * lam[None, :]) @ Q.T
    A = 0.5 * (A + A.T)
    for p in (2, 4):
        X, k, _ = impl.coupled_newton_schulz(A, p, tol=1e-13, max_iter=80)
        want = (Q * (lam ** (-1.0 / p))[None, :]) @ Q.T
        _close(X, want, 1e-9, f"coupled iteration p={p} reaches A^(-1/{p})")


def load_iteration_golden():
    rows = []
    with open(os.path.join(GOLDEN, "coupled_ns_iterations.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            p, m0, tol, iters = line.split()[:4]
            rows.append((int(p), float(m0), float(tol), int(iters)))
    return rows


def pin_iteration_count(impl):
    for p, m0, tol, iters in load_iteration_golden():
        # one eigenvalue m0 (1x1 matrix, scale fixed to 1): matrix iteration == scalar model
        _, k, _ = impl.coupled_newton_schulz(np.array([[m0]]), p, tol=tol, max_iter=200, scale=1.0)
        assert k == iters, f"p={p} m0={m0}: {k} iterations, pages say {iters}"


ALL_PINS = [pin_diagonal, pin_two_by_two, pin_known_spectrum, pin_root_invariants, pin_jacobi,
            pin_trace, pin_ema_scalar, pin_ema_rank_one, pin_apply, pin_lambda_bound,
            pin_iteration_p2_is_page_box, pin_iteration_converges_to_root, pin_iteration_count]


def failures(impl):
    out = []
    for pin in ALL_PINS:
        try:
            pin(impl)
        except AssertionError as e:
            out.append((pin.__name__, str(e)))
        except Exception as e:  # a mutant may also crash
            out.append((pin.__name__, f"{type(e).__name__}: {e}"))
    return out
