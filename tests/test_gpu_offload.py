"""Offloaded EMA state on a GPU ("Online KL Shampoo", zero-delay CPU offload):
pinned host state streamed through two device buffers on a copy stream, around
the library's steps on the caller's stream, against the same steps on
device-resident state, bit for bit, for the full and the packed layouts."""
import pytest

from gpu_common import to_dev
from workloads import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("packed", [0, 1])
def test_offloaded_state_matches_resident_state(packed):
    import torch
    import shampoo_roots_gb300 as sr
    from shampoo_roots_gb300 import offload
    shapes = [(256, 128), (300, 130), (130, 300), (96, 64)]
    groups = [[0], [1, 2], [3]]
    resident = sr.Preconditioner(0, packed_state=packed)
    streamed = sr.Preconditioner(0, packed_state=packed)

    def dev_state(d):
        t = torch.zeros(d * (d + 1) // 2 if packed else d * d, device="cuda")
        return t if packed else t.view(d, d)

    L = [dev_state(m) for m, _ in shapes]
    R = [dev_state(n) for _, n in shapes]
    off = offload.OffloadedState(shapes, "cuda", packed=bool(packed), groups=groups)
    step = offload.library_step(streamed.h, 0.95, 1e-6, -0.25)
    for s in range(3):
        G = [to_dev(synth.gradient(m, n, -0.7, synth.rng_for(41, s, i), synth.F32)) for i, (m, n) in enumerate(shapes)]
        got = off.step(G, step)
        want = [None] * len(shapes)
        for g in groups:                    # the same plans: one call per group
            out = [torch.empty(shapes[i], device="cuda") for i in g]
            sr.precond_step(resident.h, [G[i] for i in g], [L[i] for i in g], [R[i] for i in g],
                            0.95, 1e-6, -0.25, out=out)
            for i, o in zip(g, out):
                want[i] = o
        torch.cuda.synchronize()
        for a, b in zip(got, want):
            assert torch.equal(a, b)
    off.synchronize()
    torch.cuda.synchronize()
    for a, b in zip(off.L + off.R, L + R):
        assert torch.equal(a, b.cpu())
    assert all(x.is_pinned() for x in off.L + off.R)
    resident.close()
    streamed.close()
