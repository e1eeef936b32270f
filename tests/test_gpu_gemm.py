"""GPU check of the GEMM core through the C ABI self-test entry point: the
tcgen05 digit GEMM (three bf16 digits per operand with a power-of-two scale per
row and 128-column block, exact digit products, 128-wide K chunks summed in
fp32) and the fp64 engine's GEMM (double-float products on the fp32 pipes)
against float64 numpy, on ragged shapes that span several tiles and chunks and
on rows whose magnitudes differ by many orders."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

SHAPES = [(128, 128, 128), (200, 72, 300), (1000, 130, 1024), (256, 384, 4096), (17, 5, 3), (130, 260, 129)]


def _operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    A = rng.standard_normal((M, K))
    B = rng.standard_normal((N, K))
    # rows (and, through B, columns of C) scaled over 12 orders of magnitude, and
    # blocks of columns scaled apart, so the per-(row, block) scales matter
    A *= 10.0 ** rng.uniform(-6, 6, size=(M, 1))
    B *= 10.0 ** rng.uniform(-3, 3, size=(N, 1))
    colscale = 10.0 ** rng.uniform(-4, 4, size=(1, (K + 127) // 128))
    A *= np.repeat(colscale, 128, axis=1)[:, :K]
    return A.astype(np.float32), B.astype(np.float32)


@pytest.mark.parametrize("engine", [1, 2])
@pytest.mark.parametrize("shape", SHAPES)
def test_gemm_selftest_against_float64(engine, shape):
    import torch
    import shampoo_roots_gb300 as sr
    M, N, K = shape
    A, B = _operands(M, N, K, seed=M * 7 + N * 3 + K)
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    # bound: the digits hold each operand to 2^-27 of its (row, block) scale, which
    # is at most twice the block's largest magnitude; products and sums add a few
    # units of 2^-24 of the chunk sums of |a| |b|
    absprod = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64)).T
    pc = sr.Preconditioner(0)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    C = torch.empty((M, N), device="cuda")
    sr.precond_gemm_selftest(pc.h, engine, dA, dB, C, passes=3)
    pc.close()
    got = C.cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    tol = (2.0 ** -20 if engine == 2 else 2.0 ** -22) * absprod + 2.0 ** -23 * np.abs(ref)
    worst = float(np.max(err / np.maximum(tol, 1e-300)))
    print(f"engine {engine} {shape}: worst error / bound {worst:.3f}")
    assert worst <= 1.0, worst
