"""EMA state kept in host memory and streamed through the device in groups
("Online KL Shampoo", zero-delay CPU offload), on CPU: the pages' break-even
dimension, the grouping, steps over offloaded state against steps over
resident state, bit for bit, for full and packed layouts and several group
splits, and two gloo ranks whose owners keep their state offloaded against one
process.  The step here is an fp32 EMA with float64-oracle roots; on a GPU it
is the library's step (``offload.library_step``)."""
import math

import numpy as np
import pytest
import torch

from oracle import roots as O
from shampoo_roots_gb300 import offload

SHAPES = [(12, 8), (10, 10), (6, 14), (16, 4), (9, 9)]
BETA, EPS, POWER = 0.9, 1e-6, -0.25


def test_break_even_matches_the_pages():
    # H100: 989 TFLOP/s fp16, 60 GEMMs per step, 3 d^2 fp32 state elements, 64 GB/s PCIe Gen5 x16;
    # the pages conclude that the transfer hides behind the GEMMs for d >= 1546
    d = offload.break_even_dim(989e12, 60, 3, 4, 64e9)
    assert math.ceil(d) == 1546
    # the model scales as rate / link bandwidth
    assert offload.break_even_dim(2 * 989e12, 60, 3, 4, 64e9) == pytest.approx(2 * d)
    assert offload.break_even_dim(989e12, 60, 3, 4, 640e9) == pytest.approx(d / 10)


def test_default_groups_respect_the_budget():
    shapes = [(100, 50)] * 5 + [(400, 400)] + [(10, 10)] * 3
    per = [4 * (offload.state_numel(m, False) + offload.state_numel(n, False)) for m, n in shapes]
    groups = offload.default_groups(shapes, False, 120_000)
    assert sorted(i for g in groups for i in g) == list(range(len(shapes)))
    assert all(g == list(range(g[0], g[-1] + 1)) for g in groups)            # consecutive
    for g in groups:
        assert len(g) == 1 or sum(per[i] for i in g) <= 120_000           # a lone matrix may exceed it
    assert [5] in groups                                                  # the 400^2 one stands alone
    assert offload.default_groups(shapes, True, 1 << 40) == [list(range(len(shapes)))]


def test_groups_must_cover_every_matrix_once():
    for bad in ([[0, 1], [1, 2, 3, 4]], [[0, 1, 2]], [[0, 1, 2, 3, 4], []]):
        with pytest.raises(ValueError):
            offload.OffloadedState(SHAPES, "cpu", groups=bad)


def _full(x, d, packed):
    if not packed:
        return x.double()
    A = np.zeros((d, d))
    A[np.triu_indices(d)] = x.numpy()
    return torch.from_numpy(A + np.triu(A, 1).T)


def _store(dst, A, packed):
    d = A.shape[0]
    if packed:
        dst.copy_(torch.from_numpy(A.numpy()[np.triu_indices(d)]).float())
    else:
        dst.copy_(A.float())


def _ema_step(packed):
    """fp32 EMA state updated in place, float64-oracle roots, fp32 update."""

    def run(idx, grads, L, R):
        out = []
        for g, l, r in zip(grads, L, R):
            m, n = g.shape
            G = g.double()
            Lf = BETA * _full(l, m, packed) + (1 - BETA) * (G @ G.T)
            Rf = BETA * _full(r, n, packed) + (1 - BETA) * (G.T @ G)
            _store(l, Lf, packed)
            _store(r, Rf, packed)
            XL = O.inv_root(_full(l, m, packed).numpy(), EPS, POWER)
            XR = O.inv_root(_full(r, n, packed).numpy(), EPS, POWER)
            out.append(torch.from_numpy(XL @ G.numpy() @ XR).float())
        return out

    return run


def _grads(step):
    rng = np.random.default_rng([3, step])
    return [torch.from_numpy(rng.standard_normal(s).astype(np.float32)) for s in SHAPES]


@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("groups", [None, [[0], [1], [2], [3], [4]], [[0, 2], [1], [3, 4]], [[4, 3, 2, 1, 0]]])
def test_offloaded_steps_match_resident_state(packed, groups):
    fn = _ema_step(packed)
    off = offload.OffloadedState(SHAPES, "cpu", packed=packed, groups=groups)
    numel = [(offload.state_numel(m, packed), offload.state_numel(n, packed)) for m, n in SHAPES]
    L = [torch.zeros(a) if packed else torch.zeros(m, m) for (a, _), (m, _n) in zip(numel, SHAPES)]
    R = [torch.zeros(b) if packed else torch.zeros(n, n) for (_, b), (_m, n) in zip(numel, SHAPES)]
    for step in range(3):
        g = _grads(step)
        got = off.step(g, fn)
        want = fn(list(range(len(SHAPES))), g, L, R)
        for a, b in zip(got, want):
            assert torch.equal(a, b)
    off.synchronize()
    for a, b in zip(off.L + off.R, L + R):
        assert torch.equal(a, b)


def test_owner_compute_adapter():
    fn = _ema_step(False)
    off = offload.OffloadedState(SHAPES[:2], "cpu", groups=[[0], [1]])
    run = off.compute(fn)
    g = _grads(0)[:2]
    u = run([4, 1], g)                      # the owner's global indices; the state is the owner's own
    assert [tuple(x.shape) for x in u] == [SHAPES[0], SHAPES[1]]
    with pytest.raises(ValueError):
        run([4], g[:1])


def test_the_tests_see_a_shared_buffer(monkeypatch):
    """A planted mistake in the schedule: every group in one device buffer.  The
    second group's upload then lands on the first group's state before its step,
    and the comparison with resident state catches it."""
    fn = _ema_step(False)
    off = offload.OffloadedState(SHAPES, "cpu", groups=[[0], [1], [2], [3], [4]])
    real = offload.OffloadedState._views
    monkeypatch.setattr(offload.OffloadedState, "_views", lambda self, b, g: real(self, 0, g))
    L = [torch.zeros(m, m) for m, _ in SHAPES]
    R = [torch.zeros(n, n) for _, n in SHAPES]
    caught = False
    for step in range(2):                   # the second step starts from non-zero state
        g = _grads(step)
        want = fn(list(range(len(SHAPES))), g, L, R)
        try:
            got = off.step(g, fn)
        except ValueError:                  # the mixed-up state is not even positive definite
            caught = True
            break
        if not all(torch.equal(a, b) for a, b in zip(got, want)):
            caught = True
            break
    assert caught


def _free_port():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _local_grads(rank, step):
    rng = np.random.default_rng([5, rank, step])
    return [rng.standard_normal(s).astype(np.float32) for s in SHAPES]


def _owner_rank(rank, world, port, q):
    import os
    import torch.distributed as dist
    from shampoo_roots_gb300 import sharding
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        plan = sharding.OwnerSharding(SHAPES, rank, world)
        off = offload.OffloadedState([SHAPES[i] for i in plan.mine], "cpu", packed=True,
                                     groups=[[j] for j in range(len(plan.mine))])
        run = off.compute(_ema_step(True))
        outs = []
        for step in range(2):
            grads = [torch.from_numpy(g) for g in _local_grads(rank, step)]
            outs.append([u.numpy().copy() for u in plan.step(grads, run)])
        q.put((rank, plan.owners, outs))
    finally:
        dist.destroy_process_group()


def test_owners_with_offloaded_state_match_a_single_process():
    """Two gloo ranks, each owner keeping its matrices' packed state offloaded:
    the same updates as one process stepping every matrix on resident state."""
    import torch.multiprocessing as mp
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_owner_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][1] == res[1][1] and set(res[0][1]) == {0, 1}
    fn = _ema_step(True)
    L = [torch.zeros(offload.state_numel(m, True)) for m, _ in SHAPES]
    R = [torch.zeros(offload.state_numel(n, True)) for _, n in SHAPES]
    for step in range(2):
        g0, g1 = _local_grads(0, step), _local_grads(1, step)
        avg = [torch.from_numpy(((a + b) / np.float32(world)).astype(np.float32)) for a, b in zip(g0, g1)]
        want = fn(list(range(len(SHAPES))), avg, L, R)
        for rank in range(world):
            for i, u in enumerate(want):
                assert np.array_equal(res[rank][2][step][i], u.numpy()), (rank, step, i)
