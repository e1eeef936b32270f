"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and
the float64 oracle on the same seeded inputs."""
import numpy as np

from oracle import roots as oracle
from workloads import synth

TOL = 1e-3          # relative Frobenius error bound (fp32 path)


def to_dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.to(dtype) if dtype is not None else t


def run_steps(shapes, grads_per_step, dtype, beta, eps, power, engine=0, small_dim=None, check_roots=True,
              extra_opts=None):
    """Run len(grads_per_step) steps on the GPU and in the oracle; return the
    worst relative Frobenius errors (U, X_L, X_R) and the last stats."""
    import torch
    import shampoo_roots_gb300 as sr
    tdt = torch.bfloat16 if dtype == synth.BF16 else torch.float32
    opts = dict(extra_opts or {})
    if small_dim is not None:
        opts["small_dim"] = small_dim
    pc = sr.Preconditioner(0, engine=engine, **opts)
    L = [torch.zeros((m, m), device="cuda") for m, _ in shapes]
    R = [torch.zeros((n, n), device="cuda") for _, n in shapes]
    st = oracle.OracleState(shapes)
    worst = {"U": 0.0, "XL": 0.0, "XR": 0.0}
    stats = None
    for G in grads_per_step:
        g = [to_dev(x).to(tdt) for x in G]
        out = [torch.empty(x.shape, device="cuda") for x in G]
        sr.precond_step(pc.h, g, L, R, beta, eps, power, out=out)
        stats = sr.precond_get_stats(pc.h, 2 * len(shapes))
        Uo, XLo, XRo = oracle.precond_step(st, [x.astype(np.float64) for x in G], beta, eps, power)
        for i, (m, n) in enumerate(shapes):
            worst["U"] = max(worst["U"], oracle.rel_fro(out[i].cpu().numpy(), Uo[i]))
            if check_roots:
                xl = torch.empty((m, m), device="cuda")
                xr = torch.empty((n, n), device="cuda")
                sr.precond_get_root(pc.h, 2 * i, xl)
                sr.precond_get_root(pc.h, 2 * i + 1, xr)
                worst["XL"] = max(worst["XL"], oracle.rel_fro(xl.cpu().numpy(), XLo[i]))
                worst["XR"] = max(worst["XR"], oracle.rel_fro(xr.cpu().numpy(), XRo[i]))
    pc.close()
    return worst, stats
