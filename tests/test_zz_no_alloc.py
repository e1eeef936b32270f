"""The allocation-free inverse root (precond_inv_root_noalloc) against the
handle-based precond_inv_root, through the C ABI.

It serves callers that cannot allocate device memory when they need a root
(allocator hooks, host callbacks, runtimes with a fixed memory budget), so
it runs on a fixed scratch array; this file is collected last so that a
failure here never hides the other tests."""
import numpy as np
import pytest

from gpu_common import TOL
from oracle import roots as oracle
from workloads import synth

pytestmark = pytest.mark.gpu


def test_no_alloc_matches_handle_path_on_two_calls_in_a_row():
    import torch
    import shampoo_roots_gb300 as sr
    mats = [synth.spd(200, synth.rng_for(11, 0, 0)), synth.spd(256, synth.rng_for(11, 0, 1))]
    pc = sr.Preconditioner(0, engine=1)
    for power in (-0.25, -0.5):
        for a in mats:                      # two calls in a row share the scratch
            A = torch.from_numpy(a).cuda()
            X_ref = torch.empty_like(A)
            sr.precond_inv_root(pc.h, [A], [X_ref], 1e-6, power)
            X = torch.full_like(A, float("nan"))
            code, status = sr.precond_inv_root_noalloc(A, X, 1e-6, power)
            assert code == sr.OK and status == sr.OK
            err = oracle.rel_fro(X.cpu().numpy(), X_ref.cpu().numpy())
            assert err <= TOL, err
            assert oracle.rel_fro(X.cpu().numpy(), oracle.inv_root(a.astype(np.float64), 1e-6, power)) <= TOL
    pc.close()


def test_no_alloc_rejects_sizes_beyond_the_scratch():
    import torch
    import shampoo_roots_gb300 as sr
    A = torch.eye(sr.NOALLOC_MAX_D + 1, device="cuda")
    X = torch.empty_like(A)
    code, _ = sr.precond_inv_root_noalloc(A, X, 1e-6, -0.25, raw=True)
    assert code == sr.EINVAL
