"""Owner sharding across data-parallel ranks, on CPU: the LPT owner plan
against brute force and Graham's bound, and two gloo ranks running the
reduce -> owner step -> broadcast exchange against a single-process step, bit
for bit ("Sharding EMA-Gram eigensolves", matrix-sharded layout; "Online KL
Shampoo", Appendix G).  The owner's step here is the float64 oracle; on GPUs it
is the library's step (``sharding.library_compute``)."""
import itertools
import os
import socket

import numpy as np
import pytest

from shampoo_roots_gb300 import sharding

SHAPES = [(64, 32), (32, 64), (48, 48), (16, 80), (80, 16), (40, 24)]
BETA, EPS, POWER = 0.95, 1e-6, -0.25


def _brute_force(costs, world):
    return min(sharding.makespan(costs, o, world) for o in itertools.product(range(world), repeat=len(costs)))


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("seed", range(6))
def test_lpt_within_grahams_bound(world, seed):
    rng = np.random.default_rng(seed)
    costs = list(rng.uniform(1, 100, size=7))
    owners = sharding.lpt_owners(costs, world)
    assert sorted(set(owners)) <= list(range(world))
    opt = _brute_force(costs, world)
    assert sharding.makespan(costs, owners, world) <= (4 / 3 - 1 / (3 * world)) * opt + 1e-9


def test_lpt_known_cases():
    assert sharding.lpt_owners([5, 4, 3, 3, 3], 2) == [0, 1, 1, 0, 1]     # loads 8 / 10 (optimum 9: LPT is not exact)
    assert sharding.lpt_owners([1, 1, 1, 1], 4) == [0, 1, 2, 3]
    assert sharding.lpt_owners([3, 3], 1) == [0, 0]
    with pytest.raises(ValueError):
        sharding.lpt_owners([1], 0)


def test_lpt_balances_the_wide_stack():
    shapes = [(6144, 6144)] * 16 + [(6144, 3072)] * 16
    costs = [sharding.matrix_cost(m, n) for m, n in shapes]
    for world in (2, 4, 8):
        owners = sharding.lpt_owners(costs, world)
        loads = [sum(c for c, r in zip(costs, owners) if r == k) for k in range(world)]
        assert max(loads) <= (4 / 3) * sum(costs) / world
        assert len(set(owners)) == world


def test_cost_model():
    assert sharding.matrix_cost(2, 3, iters=1) == 8 + 27 + 2 * 3 * 5
    assert sharding.matrix_cost(4096, 1024) == sharding.matrix_cost(1024, 4096)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _local_grads(rank, step):
    from workloads import synth
    rng = np.random.default_rng([7, rank, step])
    return [synth.gradient(m, n, -0.7, rng, synth.F32).astype(np.float32) for m, n in SHAPES]


def _oracle_compute(state, shapes):
    import torch
    from oracle import roots as O

    def compute(idx, grads):
        st = O.OracleState([shapes[i] for i in idx])
        st.L, st.R = [state[i][0] for i in idx], [state[i][1] for i in idx]
        U, _, _ = O.precond_step(st, [g.numpy().astype(np.float64) for g in grads], BETA, EPS, POWER)
        for j, i in enumerate(idx):
            state[i] = (st.L[j], st.R[j])
        return [torch.from_numpy(u.astype(np.float32)) for u in U]
    return compute


def _rank(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        plan = sharding.OwnerSharding(SHAPES, rank, world)
        state = {i: (np.zeros((m, m)), np.zeros((n, n))) for i, (m, n) in enumerate(SHAPES) if plan.owners[i] == rank}
        outs = []
        for step in range(2):
            grads = [torch.from_numpy(g) for g in _local_grads(rank, step)]
            U = plan.step(grads, _oracle_compute(state, SHAPES))
            outs.append([u.numpy().copy() for u in U])
        q.put((rank, plan.owners, sorted(state), outs))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_match_a_single_process_bit_for_bit():
    import torch.multiprocessing as mp
    from oracle import roots as O
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    owners = res[0][1]
    assert res[1][1] == owners
    assert set(owners) == {0, 1}
    # each rank kept the state of exactly the matrices it owns
    assert res[0][2] == [i for i, r in enumerate(owners) if r == 0]
    assert res[1][2] == [i for i, r in enumerate(owners) if r == 1]
    # single process: the same fp32 average of both ranks' gradients, the same oracle step on all matrices
    st = O.OracleState(SHAPES)
    for step in range(2):
        g0, g1 = _local_grads(0, step), _local_grads(1, step)
        avg = [((a + b) / np.float32(world)).astype(np.float32) for a, b in zip(g0, g1)]
        U, _, _ = O.precond_step(st, [g.astype(np.float64) for g in avg], BETA, EPS, POWER)
        for rank in range(world):
            for i, u in enumerate(U):
                got = res[rank][3][step][i]
                assert got.dtype == np.float32
                assert np.array_equal(got, u.astype(np.float32)), (rank, step, i)
