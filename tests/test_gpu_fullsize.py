"""GPU parity at the workloads' full sizes, on sampled matrices: the whole
stack runs on the GPU exactly as bench.py times it, and the float64 oracle
recomputes a sample of its matrices (one of each shape class) from the same
gradients, step by step."""
import numpy as np
import pytest

from gpu_common import TOL
from oracle import roots as oracle
from workloads import synth

pytestmark = pytest.mark.gpu


def _stack_parity(index, steps, power, sample=None, opts=None):
    import torch
    import shampoo_roots_gb300 as sr
    w = synth.workload(index)
    shapes = list(w.shapes)
    if sample is None:
        sample = sorted({shapes.index(s) for s in set(shapes)})     # first matrix of each shape class
    dev = torch.device("cuda")
    L = [torch.zeros((m, m), device=dev) for m, _ in shapes]
    R = [torch.zeros((n, n), device=dev) for _, n in shapes]
    out = [torch.empty((m, n), device=dev) for m, n in shapes]
    st = oracle.OracleState([shapes[i] for i in sample])
    pc = sr.Preconditioner(0, **(opts or {}))
    worst = {"U": 0.0, "XL": 0.0, "XR": 0.0}
    for s in range(steps):
        grads = synth.torch_gradients_for_step(w, s, dev)
        sr.precond_step(pc.h, grads, L, R, w.beta, w.eps, power, out=out)
        _, _, status, _ = sr.precond_get_stats(pc.h, 2 * len(shapes))
        assert all(x == 0 for x in status), (s, status)
        G = [grads[i].float().cpu().numpy().astype(np.float64) for i in sample]
        Uo, XLo, XRo = oracle.precond_step(st, G, w.beta, w.eps, power)
        for k, i in enumerate(sample):
            m, n = shapes[i]
            xl = torch.empty((m, m), device=dev)
            xr = torch.empty((n, n), device=dev)
            sr.precond_get_root(pc.h, 2 * i, xl)
            sr.precond_get_root(pc.h, 2 * i + 1, xr)
            worst["U"] = max(worst["U"], oracle.rel_fro(out[i].cpu().numpy(), Uo[k]))
            worst["XL"] = max(worst["XL"], oracle.rel_fro(xl.cpu().numpy(), XLo[k]))
            worst["XR"] = max(worst["XR"], oracle.rel_fro(xr.cpu().numpy(), XRo[k]))
    pc.close()
    print(f"workload {w.name} power {power}: worst relative Frobenius errors {worst}")
    assert max(worst.values()) <= TOL, worst
    return worst


def test_stack_quarter_power_full_size():
    """24-layer d=1024 stack, bf16 gradients, power -1/4, 10 EMA steps."""
    _stack_parity(1, 10, -0.25)


def test_stack_inverse_sqrt_full_size():
    """Same stack, power -1/2, 10 EMA steps."""
    _stack_parity(2, 10, -0.5)


def test_wide_6144_full_size():
    """16 fp32 gradients of 6144^2 and 16 of 6144x3072 (alpha -0.5), power -1/4,
    4 EMA steps; the oracle recomputes one matrix of each shape at every step:
    matrix 0 (6144^2, both Grams full-rank 6144^2) and matrix 16 (6144x3072,
    its rank-deficient 6144^2 left and full-rank 3072^2 right Grams)."""
    _stack_parity(4, 4, -0.25, sample=[0, 16])


@pytest.mark.parametrize("power", [-0.25, -0.5])
def test_spd64_2048_full_size(power):
    """64 SPD 2048^2 matrices with log-uniform spectra on [1e-8, 1], eps 1e-6
    relative to the trace; roots of all 64, oracle on 4 of them."""
    _spd_parity(power)


def _spd_parity(power, opts=None):
    import torch
    import shampoo_roots_gb300 as sr
    w = synth.workload(3)
    dev = torch.device("cuda")
    A = synth.torch_spd_inputs(w, dev)
    X = [torch.empty_like(a) for a in A]
    pc = sr.Preconditioner(0, **(opts or {}))
    sr.precond_inv_root(pc.h, A, X, w.eps, power)
    _, _, status, _ = sr.precond_get_stats(pc.h, len(A))
    pc.close()
    assert all(s == 0 for s in status), status
    errs = {}
    for i in (0, 21, 42, 63):
        a = A[i].cpu().numpy().astype(np.float64)
        errs[i] = oracle.rel_fro(X[i].cpu().numpy(), oracle.inv_root(a, w.eps, power))
    print(f"workload {w.name} power {power}: relative Frobenius errors {errs}")
    for i, err in errs.items():
        assert err <= TOL, (i, err)
    return errs
