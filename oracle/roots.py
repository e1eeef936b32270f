"""Plain float64 CPU oracle for the matrix-preconditioner step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run this module.  The CUDA
library never calls it, and it shares no code with the CUDA path.

What it computes (per weight matrix G, m x n, row-major), following
"Sharding EMA-Gram eigensolves" (Marin research note), section Background:

1. Gram EMAs:  L <- beta L + (1 - beta) G G^T,   R <- beta R + (1 - beta) G^T G
   (the left Gram averages the gradient times its transpose, the right Gram
   the reverse product).
2. Rescale each Gram to unit trace:  A_hat = L / tr(L).
3. Eigendecompose A_hat = Q diag(lam) Q^T (LAPACK ``eigh``), add the
   regulariser eps to the eigenvalues, raise to ``power`` (-1/4 for the
   quarter power, -1/2 for the inverse square root of "Online KL Shampoo"
   section 2) and reconstruct X = Q diag((lam + eps)**power) Q^T.
4. Apply both sides:  U = X_L G X_R.

This is a plain definition: the GPU method reaches the same result through a
matmul-only iteration; the oracle does not.  Everything runs in float64; the
inputs are upcast exactly from their fp32 / bf16 storage values.

Also here, each following its passage:
* ``lambda_max_bound``: the O(n^2) upper bound on the largest eigenvalue used
  to scale the iteration's start ("Online KL Shampoo", Appendix D: the minimum
  of the Wolkowicz-Styan bound and the Minc row-sum bound).
* ``coupled_newton_schulz``: the coupled Newton-Schulz inverse p-th root
  iteration in float64 ("Online KL Shampoo", section 2.2 and the Appendix D
  algorithm box for p = 2; the p-th-root generalisation X <- X T,
  M <- T^p M, T = ((p+1) I - M) / p is Guo & Higham 2006, which reduces to the
  page's (a, b) = (3/2, -1/2) step at p = 2).  A debug reference for the
  iteration, not the parity target.
* ``scalar_iterations``: the scalar model of that iteration on one eigenvalue,
  used to bound the iteration count (section 2.2 puts the classical
  iteration at about 21 steps).

Readings of points the pages leave open:
* the rescaling of the Grams before the root (Background) = divide by the
  trace (unit trace).
* the regulariser is added to the eigenvalues of the rescaled Gram, with no
  clamp of tiny negative eigenvalues; lam + eps <= 0 raises.
* the EMA state is stored raw; rescaling applies to a copy at each update.
* G is m x n, L = G G^T is m x m and R = G^T G is n x n.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np


# --------------------------------------------------------------------------
# step 1: Gram EMAs
# --------------------------------------------------------------------------
def gram_ema(L: np.ndarray, R: np.ndarray, G: np.ndarray, beta: float) -> Tuple[np.ndarray, np.ndarray]:
    """EMA of the left and right Grams ("Sharding EMA-Gram eigensolves", Background)."""
    G = np.asarray(G, dtype=np.float64)
    L_new = beta * L + (1.0 - beta) * (G @ G.T)
    R_new = beta * R + (1.0 - beta) * (G.T @ G)
    return L_new, R_new


# --------------------------------------------------------------------------
# step 2: rescale
# --------------------------------------------------------------------------
def trace_normalise(A: np.ndarray) -> np.ndarray:
    """A / tr(A): the Gram rescaled to unit trace (the reading taken of the
    rescaling step of "Sharding EMA-Gram eigensolves", Background)."""
    A = np.asarray(A, dtype=np.float64)
    t = np.trace(A)
    if not np.isfinite(t) or t <= 0.0:
        raise ValueError(f"trace must be positive and finite, got {t}")
    return A / t


# --------------------------------------------------------------------------
# step 3: eigendecomposition root
# --------------------------------------------------------------------------
def inv_root_eigh(A_hat: np.ndarray, eps: float, power: float) -> np.ndarray:
    """Q diag((lam + eps)**power) Q^T of a symmetric matrix ("Sharding EMA-Gram
    eigensolves", Background: decompose, add a small regulariser to the
    eigenvalues, raise to the power, reconstruct)."""
    A_hat = np.asarray(A_hat, dtype=np.float64)
    lam, Q = np.linalg.eigh(A_hat)
    shifted = lam + eps
    if np.any(shifted <= 0.0):
        raise ValueError("an eigenvalue plus eps is not positive")
    f = shifted ** power
    return (Q * f[None, :]) @ Q.T


# --------------------------------------------------------------------------
# step 4: two-sided apply
# --------------------------------------------------------------------------
def precondition(X_L: np.ndarray, G: np.ndarray, X_R: np.ndarray) -> np.ndarray:
    """U = X_L G X_R: both powers applied to the gradient to form the update
    ("Sharding EMA-Gram eigensolves", Background)."""
    return X_L @ np.asarray(G, dtype=np.float64) @ X_R


# --------------------------------------------------------------------------
# whole step and whole root
# --------------------------------------------------------------------------
class OracleState:
    """float64 EMA state for a list of matrices, starting from zero Grams."""

    def __init__(self, shapes: Sequence[Tuple[int, int]]):
        self.shapes = [tuple(s) for s in shapes]
        self.L = [np.zeros((m, m)) for m, _ in self.shapes]
        self.R = [np.zeros((n, n)) for _, n in self.shapes]


def precond_step(state: OracleState, grads: Sequence[np.ndarray], beta: float, eps: float,
                 power: float):
    """One preconditioner step for every matrix.  Returns (U, X_L, X_R) lists."""
    U, XL, XR = [], [], []
    for i, G in enumerate(grads):
        state.L[i], state.R[i] = gram_ema(state.L[i], state.R[i], G, beta)
        xl = inv_root_eigh(trace_normalise(state.L[i]), eps, power)
        xr = inv_root_eigh(trace_normalise(state.R[i]), eps, power)
        XL.append(xl)
        XR.append(xr)
        U.append(precondition(xl, G, xr))
    return U, XL, XR


def inv_root(A: np.ndarray, eps: float, power: float) -> np.ndarray:
    """Root of a given SPD matrix through the same rescale + regularise + eigh
    path (no EMA, no gradient); eps is therefore relative to the trace."""
    return inv_root_eigh(trace_normalise(A), eps, power)


# --------------------------------------------------------------------------
# scaling bound ("Online KL Shampoo", Appendix D helper)
# --------------------------------------------------------------------------
def lambda_max_bound(A: np.ndarray) -> float:
    """Upper bound on the largest eigenvalue of a symmetric matrix, O(n^2):
    min(Wolkowicz-Styan, Minc).

    Wolkowicz-Styan: with mu = tr(A)/n and s^2 = ||A||_F^2 / n - mu^2,
    lam_max <= mu + s sqrt(n - 1).
    Minc: with row sums r = |A| 1 (floored at 1e-12), lam_max <= max_i (|A| r)_i / r_i.
    """
    A = np.asarray(A, dtype=np.float64)
    n = A.shape[0]
    mu = np.trace(A) / n
    s2 = max(np.sum(A * A) / n - mu * mu, 0.0)
    ws = mu + np.sqrt(s2) * np.sqrt(n - 1)
    absA = np.abs(A)
    r = np.maximum(absA.sum(axis=1), 1e-12)
    minc = np.max((absA @ r) / r)
    return float(min(ws, minc))


# --------------------------------------------------------------------------
# coupled Newton-Schulz (debug reference for the iteration, float64)
# --------------------------------------------------------------------------
def coupled_newton_schulz(A_hat_reg: np.ndarray, p: int, tol: float = 1e-12, max_iter: int = 100,
                          scale: float | None = None):
    """Inverse p-th root of an SPD matrix by the coupled iteration.

    c = 1.01 * lambda_max_bound (the start's scale), M_0 = A / c, X_0 = I;
    repeat  T = ((p+1) I - M) / p,  X <- X T,  M <- T^p M  until
    ||M - I||_F <= tol; return sym(X) * c**(-1/p).
    Returns (X, iterations, residual history).
    """
    A = np.asarray(A_hat_reg, dtype=np.float64)
    d = A.shape[0]
    c = 1.01 * lambda_max_bound(A) if scale is None else scale
    I = np.eye(d)
    M = A / c
    X = I.copy()
    hist = []
    k = 0
    while k < max_iter:
        r = np.linalg.norm(M - I)
        hist.append(r)
        if r <= tol:
            break
        T = ((p + 1) * I - M) / p
        X = X @ T
        M = np.linalg.matrix_power(T, p) @ M
        k += 1
    X = 0.5 * (X + X.T) * c ** (-1.0 / p)
    return X, k, hist


def scalar_iterations(m0: float, p: int, tol: float) -> int:
    """Iterations of the scalar map m <- m ((p+1-m)/p)^p from m0 until |m - 1| < tol."""
    m = float(m0)
    k = 0
    while abs(m - 1.0) >= tol:
        m = m * ((p + 1 - m) / p) ** p
        k += 1
        if k > 10000:
            raise RuntimeError("scalar iteration did not converge")
    return k


def rel_fro(a: np.ndarray, b: np.ndarray) -> float:
    """||a - b||_F / ||b||_F (the parity measure)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))
