"""GPU parity: the CUDA path through the C ABI against the float64 oracle,
element by element (relative Frobenius error <= 1e-3 on the fp32 path)."""
import numpy as np
import pytest

from gpu_common import TOL, run_steps, to_dev
from oracle import roots as oracle
from workloads import synth

pytestmark = pytest.mark.gpu


def test_single_256x128_full_size():
    w = synth.workload(0)
    G = synth.gradients_for_step(w, 0)
    worst, (it, res, status, scale) = run_steps(list(w.shapes), [G], w.dtype, w.beta, w.eps, -0.25)
    print(f"workload {w.name}: worst relative Frobenius errors {worst}, iterations {it}")
    assert all(s == 0 for s in status), status
    assert max(worst.values()) <= TOL, worst
    # start scale c = 1.01 x the bound of the oracle's rescaled, regularised Gram
    st = oracle.OracleState(list(w.shapes))
    Lo, Ro = oracle.gram_ema(st.L[0], st.R[0], G[0].astype(np.float64), w.beta)
    for k, A in enumerate((Lo, Ro)):
        Ah = oracle.trace_normalise(A) + w.eps * np.eye(A.shape[0])
        assert abs(scale[k] / (1.01 * oracle.lambda_max_bound(Ah)) - 1) < 1e-5


@pytest.mark.parametrize("engine", [1, 2])
@pytest.mark.parametrize("power", [-0.25, -0.5])
def test_ragged_shapes_both_engines(engine, power):
    """Sizes that leave ragged tiles in both engines (tile 64 / 128 x 256)."""
    shapes = [(300, 130), (130, 300), (257, 257)]
    rng = [synth.rng_for(9, 0, i) for i in range(3)]
    G = [synth.gradient(m, n, -0.7, rng[i], synth.F32) for i, (m, n) in enumerate(shapes)]
    worst, (it, res, status, _) = run_steps(shapes, [G], synth.F32, 0.95, 1e-6, power, engine=engine)
    assert all(s == 0 for s in status), status
    assert max(worst.values()) <= TOL, worst


def test_stack_bf16_scaled_quarter():
    """The 24-layer d=1024 stack recipe at 1/4 size (2 layers), 3 EMA steps:
    256^2 Grams on the fp64 engine, 1024^2 on the tcgen05 engine."""
    w = synth.scaled(synth.workload(1), 4)
    shapes = list(w.shapes[:12])
    steps = [[synth.gradient(m, n, w.alpha, synth.rng_for(1, s, i), w.dtype) for i, (m, n) in enumerate(shapes)]
             for s in range(3)]
    worst, (it, res, status, _) = run_steps(shapes, steps, w.dtype, w.beta, w.eps, -0.25)
    assert all(s == 0 for s in status), status
    assert max(worst.values()) <= TOL, worst


@pytest.mark.parametrize("power", [-0.25, -0.5])
def test_spd_inv_root_tcgen05(power):
    """Conditioning-stress recipe (log-uniform spectrum on [1e-8, 1]) at d=1024."""
    import torch
    import shampoo_roots_gb300 as sr
    A = [synth.spd(1024, synth.rng_for(3, 0, i)) for i in range(3)]
    pc = sr.Preconditioner(0)
    X = [torch.empty_like(to_dev(a)) for a in A]
    sr.precond_inv_root(pc.h, [to_dev(a) for a in A], X, 1e-6, power)
    it, res, status, _ = sr.precond_get_stats(pc.h, len(A))
    pc.close()
    assert all(s == 0 for s in status), status
    for a, x in zip(A, X):
        err = oracle.rel_fro(x.cpu().numpy(), oracle.inv_root(a.astype(np.float64), 1e-6, power))
        assert err <= TOL, err


def test_nonfinite_gradient_flags_and_keeps_state():
    import torch
    import shampoo_roots_gb300 as sr
    pc = sr.Preconditioner(0)
    g = torch.randn(64, 32, device="cuda")
    g[3, 5] = float("nan")
    L = torch.full((64, 64), 0.5, device="cuda")
    R = torch.full((32, 32), 0.25, device="cuda")
    out = torch.full((64, 32), 7.0, device="cuda")
    sr.precond_step(pc.h, [g], [L], [R], 0.9, 1e-6, -0.25, out=[out])
    it, res, status, _ = sr.precond_get_stats(pc.h, 2)
    pc.close()
    assert status == [sr.ENONFINITE, sr.ENONFINITE]
    assert torch.all(L == 0.5) and torch.all(R == 0.25)
    assert torch.all(out == 7.0)


def test_iteration_cap_reports_notconv_and_writes():
    import torch
    import shampoo_roots_gb300 as sr
    pc = sr.Preconditioner(0, max_iter=1)
    g = to_dev(synth.gradients_for_step(synth.workload(0), 0)[0])
    L = torch.zeros(256, 256, device="cuda")
    R = torch.zeros(128, 128, device="cuda")
    out = torch.full((256, 128), float("nan"), device="cuda")
    sr.precond_step(pc.h, [g], [L], [R], 0.95, 1e-6, -0.25, out=[out])
    it, res, status, _ = sr.precond_get_stats(pc.h, 2)
    pc.close()
    assert status == [sr.ENOTCONV, sr.ENOTCONV] and it == [1, 1]
    assert torch.isfinite(out).all()


def test_resume_matches_straight_run():
    """Run 3 steps, copy the state out and back, run 3 more: identical bits to 6 straight steps."""
    import torch
    import shampoo_roots_gb300 as sr
    shapes = [(96, 160), (600, 520)]
    grads = [[to_dev(synth.gradient(m, n, -0.7, synth.rng_for(7, s, i), synth.F32)) for i, (m, n) in
              enumerate(shapes)] for s in range(6)]

    def run(steps, L, R, pc):
        outs = []
        for G in steps:
            o = [torch.empty_like(x) for x in G]
            sr.precond_step(pc.h, [x.clone() for x in G], L, R, 0.95, 1e-6, -0.25, out=o)
            outs.append(o)
        torch.cuda.synchronize()
        return outs

    pc = sr.Preconditioner(0)
    L = [torch.zeros(m, m, device="cuda") for m, _ in shapes]
    R = [torch.zeros(n, n, device="cuda") for _, n in shapes]
    straight = run(grads, L, R, pc)
    L2 = [torch.zeros(m, m, device="cuda") for m, _ in shapes]
    R2 = [torch.zeros(n, n, device="cuda") for _, n in shapes]
    run(grads[:3], L2, R2, pc)
    saved = [x.cpu() for x in L2 + R2]
    pc.close()
    pc = sr.Preconditioner(0)
    L3 = [s.cuda() for s in saved[:2]]
    R3 = [s.cuda() for s in saved[2:]]
    resumed = run(grads[3:], L3, R3, pc)
    pc.close()
    for a, b in zip(straight[3:], resumed):
        for x, y in zip(a, b):
            assert torch.equal(x, y)
    for x, y in zip(L + R, L3 + R3):
        assert torch.equal(x, y)


def test_bf16_in_place_output():
    import torch
    import shampoo_roots_gb300 as sr
    shapes = [(128, 96)]
    G = [synth.gradient(128, 96, -0.7, synth.rng_for(5, 0, 0), synth.BF16)]
    g = to_dev(G[0]).to(torch.bfloat16)
    pc = sr.Preconditioner(0)
    L = torch.zeros(128, 128, device="cuda")
    R = torch.zeros(96, 96, device="cuda")
    sr.precond_step(pc.h, [g], [L], [R], 0.95, 1e-6, -0.5)
    pc.close()
    st = oracle.OracleState(shapes)
    Uo, _, _ = oracle.precond_step(st, [G[0].astype(np.float64)], 0.95, 1e-6, -0.5)
    want = synth.round_to_bf16(Uo[0])
    got = g.float().cpu().numpy()
    # in-place bf16 output: the fp32 U (relative error ~1e-5 of max |U|) rounded
    # once; near a rounding boundary that is one bf16 step from the rounded oracle
    ulp = np.abs(want) * 2.0 ** -7
    assert np.all(np.abs(got - want) <= ulp + 1e-4 * np.abs(Uo[0]).max())
    assert oracle.rel_fro(got, Uo[0]) <= 2.0 ** -8


@pytest.mark.gpu
@pytest.mark.parametrize("engine", [1, 2])
def test_graph_replay_matches_direct_launches(engine):
    """The graph path replays one capture per plan with fresh pointer tables and
    runs the Gram, start, iteration and finish stages of these small plans on
    forked streams (with and without the graph): it must give bit-identical
    results to direct launches on one stream while the caller's tensors move,
    the plan changes and comes back, and the caller uses a non-default stream."""
    import torch
    import shampoo_roots_gb300 as sr
    rng = np.random.default_rng(11)
    # the first plan comes back while cached, and again after five other plans
    # have evicted it (the handle keeps four)
    plans = [[(200, 72), (64, 136)], [(96, 40)], [(200, 72), (64, 136)], [(200, 72), (64, 136)],
             [(40, 24)], [(48, 24)], [(56, 24)], [(64, 24)], [(72, 24)], [(200, 72), (64, 136)]]
    results = {}
    # (graph, branches): direct launches on one stream, graph replay with the stages on
    # forked streams, and direct launches on forked streams
    for use_graph, branches in ((0, 0), (1, 1), (0, 1)):
        pc = sr.Preconditioner(0, engine=engine, small_dim=0 if engine == 2 else 512, use_graph=use_graph,
                               branches=branches)
        rng = np.random.default_rng(11)
        side = torch.cuda.Stream()
        state = {}
        outs = []
        launches0 = sr.precond_launch_count(pc.h)
        with torch.cuda.stream(side):
            for shapes in plans:
                key = tuple(shapes)
                if key not in state:
                    state[key] = ([torch.zeros((m, m), device="cuda") for m, _ in shapes],
                                  [torch.zeros((n, n), device="cuda") for _, n in shapes])
                L, R = state[key]
                g = [torch.from_numpy(synth.gradient(m, n, 1.0, rng, synth.F32)).cuda() for m, n in shapes]
                out = [torch.empty((m, n), device="cuda") for m, n in shapes]
                sr.precond_step(pc.h, g, L, R, 0.9, 1e-6, -0.25, out=out, stream=side)
                outs.append([o.cpu() for o in out])
        torch.cuda.synchronize()
        results[(use_graph, branches)] = (outs, sr.precond_launch_count(pc.h) - launches0,
                                          sr.precond_get_stats(pc.h, 4))
        pc.close()
    o0, n0, s0 = results[(0, 0)]
    for key in ((1, 1), (0, 1)):
        o1, n1, s1 = results[key]
        assert n0 == n1 > 0
        for a, b in zip(o0, o1):
            for x, y in zip(a, b):
                assert torch.equal(x, y)
        assert s0[0] == s1[0] and s0[2] == s1[2]


@pytest.mark.gpu
@pytest.mark.parametrize("engine", [1, 2])
def test_tiny_and_degenerate_shapes(engine):
    """Sides of 1, 2, 3 and 17 (single-element Grams, rank-1 Grams, tiles that
    are almost all padding), two EMA steps, both engines.

    eps is 1e-4 here: the EMA state is fp32 by contract, and its rounding moves
    the zero eigenvalues of a rank-1 d = 3 Gram by about 2^-24 of its trace.
    Against eps = 1e-6 that alone changes (lambda + eps)^(-1/4) by about 1.5 %
    in the directions where X is largest, whatever computes the root.  With
    large d the perturbation spreads over many directions and the workloads
    meet the bar at eps = 1e-6."""
    shapes = [(1, 5), (3, 1), (2, 2), (17, 33)]
    steps = []
    for s in range(2):
        rng = [synth.rng_for(11, s, i) for i in range(len(shapes))]
        steps.append([synth.gradient(m, n, -0.5, rng[i], synth.F32) for i, (m, n) in enumerate(shapes)])
    worst, (it, res, status, _) = run_steps(shapes, steps, synth.F32, 0.9, 1e-4, -0.25, engine=engine)
    assert all(s == 0 for s in status), status
    assert max(worst.values()) <= TOL, worst


@pytest.mark.gpu
@pytest.mark.parametrize("engine", [0, 1])
def test_tiny_and_degenerate_shapes_root_of_the_fp32_state(engine):
    """The same tiny and rank-deficient shapes at the workloads' eps = 1e-6,
    through the default engine choice (these sides are all <= 64, so the fp64
    engine) and the fp64 engine forced.

    Here the oracle roots the GPU's own fp32 EMA state (read back after each
    step and upcast exactly), so the state's rounding, which the caller's fp32
    layout fixes, is not part of the comparison: what is compared is the root
    of the Gram the step actually held ("Sharding EMA-Gram eigensolves",
    Background: rescale, add eps to the eigenvalues, raise to the power,
    reconstruct), element by element, and the update built from it.  A rank-1
    Gram of side 3 has eigenvalues 1e-6 below entries of order 1: its root needs
    the start matrix to about 2^-30, which the fp64 engine (and its fp64 start)
    gives and the tcgen05 engine's 27-bit digits do not; that engine is checked
    on these shapes at eps = 1e-4 above."""
    import torch
    import shampoo_roots_gb300 as sr
    shapes = [(1, 5), (3, 1), (2, 2), (17, 33)]
    eps, power, beta = 1e-6, -0.25, 0.9
    pc = sr.Preconditioner(0, engine=engine)
    L = [torch.zeros((m, m), device="cuda") for m, _ in shapes]
    R = [torch.zeros((n, n), device="cuda") for _, n in shapes]
    worst = {"U": 0.0, "XL": 0.0, "XR": 0.0}
    for s in range(2):
        G = [synth.gradient(m, n, -0.5, synth.rng_for(11, s, i), synth.F32) for i, (m, n) in enumerate(shapes)]
        g = [to_dev(x) for x in G]
        out = [torch.empty(x.shape, device="cuda") for x in G]
        sr.precond_step(pc.h, g, L, R, beta, eps, power, out=out)
        _, _, status, _ = sr.precond_get_stats(pc.h, 2 * len(shapes))
        assert all(x == 0 for x in status), (s, status)
        for i, (m, n) in enumerate(shapes):
            xl = torch.empty((m, m), device="cuda")
            xr = torch.empty((n, n), device="cuda")
            sr.precond_get_root(pc.h, 2 * i, xl)
            sr.precond_get_root(pc.h, 2 * i + 1, xr)
            xlo = oracle.inv_root_eigh(oracle.trace_normalise(L[i].cpu().numpy().astype(np.float64)), eps, power)
            xro = oracle.inv_root_eigh(oracle.trace_normalise(R[i].cpu().numpy().astype(np.float64)), eps, power)
            uo = oracle.precondition(xlo, G[i].astype(np.float64), xro)
            worst["XL"] = max(worst["XL"], oracle.rel_fro(xl.cpu().numpy(), xlo))
            worst["XR"] = max(worst["XR"], oracle.rel_fro(xr.cpu().numpy(), xro))
            worst["U"] = max(worst["U"], oracle.rel_fro(out[i].cpu().numpy(), uo))
    pc.close()
    print(f"engine {engine}: worst relative Frobenius errors against the root of the fp32 state {worst}")
    assert max(worst.values()) <= TOL, worst


@pytest.mark.gpu
def test_zero_gradient_from_zero_state_is_flagged():
    """An all-zero gradient on zero state leaves Grams of trace 0, whose unit-trace
    rescaling is undefined: both roots report ENONFINITE, the output is not
    written, and the state holds the (zero) EMA."""
    import torch
    import shampoo_roots_gb300 as sr
    pc = sr.Preconditioner(0)
    g = torch.zeros(48, 24, device="cuda")
    L = torch.zeros(48, 48, device="cuda")
    R = torch.zeros(24, 24, device="cuda")
    out = torch.full((48, 24), 3.0, device="cuda")
    sr.precond_step(pc.h, [g], [L], [R], 0.9, 1e-6, -0.25, out=[out])
    _, _, status, _ = sr.precond_get_stats(pc.h, 2)
    pc.close()
    assert status == [sr.ENONFINITE, sr.ENONFINITE]
    assert torch.all(out == 3.0)
    assert torch.all(L == 0) and torch.all(R == 0)


@pytest.mark.gpu
def test_two_handles_on_two_streams_match_their_solo_runs():
    """Two handles used at the same time on two streams (one per thread of a
    training job, say) share nothing: each gives bit-identical results to the
    same calls made alone."""
    import torch
    import shampoo_roots_gb300 as sr
    shapes = [[(160, 96), (96, 160)], [(256, 64)]]
    rngs = [synth.rng_for(13, 0, i) for i in range(3)]
    grads = [[torch.from_numpy(synth.gradient(m, n, -0.7, rngs[j + 2 * k], synth.F32)).cuda()
              for j, (m, n) in enumerate(sh)] for k, sh in enumerate(shapes)]

    def run(concurrent):
        hs = [sr.Preconditioner(0) for _ in shapes]
        streams = [torch.cuda.Stream() for _ in shapes]
        state = [([torch.zeros((m, m), device="cuda") for m, _ in sh],
                  [torch.zeros((n, n), device="cuda") for _, n in sh]) for sh in shapes]
        outs = [[torch.empty((m, n), device="cuda") for m, n in sh] for sh in shapes]
        for step in range(3):
            for k in range(len(shapes)):
                with torch.cuda.stream(streams[k]):
                    sr.precond_step(hs[k].h, grads[k], state[k][0], state[k][1], 0.9, 1e-6, -0.25, out=outs[k],
                                    stream=streams[k])
                if not concurrent:
                    torch.cuda.synchronize()
        torch.cuda.synchronize()
        res = [[o.cpu() for o in ok] for ok in outs]
        for h in hs:
            h.close()
        return res

    solo, both = run(False), run(True)
    for a, b in zip(solo, both):
        for x, y in zip(a, b):
            assert torch.equal(x, y)


@pytest.mark.gpu
def test_many_small_matrices_in_one_call():
    """300 gradients of four small shapes in one call (large batch dimensions
    in every grid, long pointer tables), two EMA steps, against the oracle on
    every matrix."""
    shapes = [(32, 16), (16, 48), (40, 40), (24, 8)] * 75
    steps = []
    for s in range(2):
        steps.append([synth.gradient(m, n, -0.5, synth.rng_for(17, s, i), synth.F32)
                      for i, (m, n) in enumerate(shapes)])
    worst, (it, res, status, _) = run_steps(shapes, steps, synth.F32, 0.9, 1e-4, -0.25, check_roots=False)
    assert all(s == 0 for s in status), status
    assert worst["U"] <= TOL, worst


def _pack_upper(a):
    """Row-by-row packing of the upper triangle of a square array (the library's layout)."""
    d = a.shape[0]
    return np.concatenate([a[r, r:] for r in range(d)])


@pytest.mark.parametrize("engine", [1, 2])
def test_packed_state_matches_full_state_bit_for_bit(engine):
    """PRECOND_OPT_PACKED_STATE ("Online KL Shampoo", Appendix F, packed
    symmetric state): the EMA state is the upper triangle packed row by row.
    The full state is kept exactly symmetric, so three steps with either layout
    give identical updates and roots, the packed state equals the full state's
    upper triangle, and both meet the oracle."""
    import torch
    import shampoo_roots_gb300 as sr
    shapes = [(40, 24), (17, 33)] if engine == 1 else [(300, 130), (130, 300), (257, 257), (96, 64)]
    steps = [[synth.gradient(m, n, -0.7, synth.rng_for(23, s, i), synth.F32) for i, (m, n) in enumerate(shapes)]
             for s in range(3)]

    def run(packed):
        pc = sr.Preconditioner(0, engine=engine, packed_state=packed)
        if packed:
            L = [torch.zeros(m * (m + 1) // 2, device="cuda") for m, _ in shapes]
            R = [torch.zeros(n * (n + 1) // 2, device="cuda") for _, n in shapes]
        else:
            L = [torch.zeros((m, m), device="cuda") for m, _ in shapes]
            R = [torch.zeros((n, n), device="cuda") for _, n in shapes]
        outs, roots = [], []
        for G in steps:
            out = [torch.empty((m, n), device="cuda") for m, n in shapes]
            sr.precond_step(pc.h, [to_dev(g) for g in G], L, R, 0.95, 1e-6, -0.25, out=out)
            outs.append([o.cpu().numpy() for o in out])
            rr = []
            for i, (m, n) in enumerate(shapes):
                xl, xr = torch.empty((m, m), device="cuda"), torch.empty((n, n), device="cuda")
                sr.precond_get_root(pc.h, 2 * i, xl)
                sr.precond_get_root(pc.h, 2 * i + 1, xr)
                rr.append((xl.cpu().numpy(), xr.cpu().numpy()))
            roots.append(rr)
        _, _, status, _ = sr.precond_get_stats(pc.h, 2 * len(shapes))
        state = ([x.cpu().numpy() for x in L], [x.cpu().numpy() for x in R])
        pc.close()
        return outs, roots, state, status

    fo, fr, (fL, fR), fs = run(0)
    po, pr, (pL, pR), ps = run(1)
    assert all(s == 0 for s in fs) and all(s == 0 for s in ps), (fs, ps)
    for a, b in zip(fL + fR, pL + pR):
        assert np.array_equal(a, a.T)                  # the full state is exactly symmetric
        assert np.array_equal(_pack_upper(a), b)
    for s in range(len(steps)):
        for i in range(len(shapes)):
            assert np.array_equal(fo[s][i], po[s][i]), (s, i)
            assert np.array_equal(fr[s][i][0], pr[s][i][0]) and np.array_equal(fr[s][i][1], pr[s][i][1])
    st = oracle.OracleState(shapes)
    for s, G in enumerate(steps):
        Uo, XLo, XRo = oracle.precond_step(st, [g.astype(np.float64) for g in G], 0.95, 1e-6, -0.25)
        for i in range(len(shapes)):
            assert oracle.rel_fro(po[s][i], Uo[i]) <= TOL
            assert oracle.rel_fro(pr[s][i][0], XLo[i]) <= TOL and oracle.rel_fro(pr[s][i][1], XRo[i]) <= TOL


def test_timing_modes_give_identical_results():
    """PRECOND_OPT_TIMING = 1 (an event around every iteration-stage GEMM) and
    2 (per-stage events only) give the same update bit for bit; mode 2 reports
    no per-launch time but the same launches and issued work."""
    import torch
    import shampoo_roots_gb300 as sr
    shapes = [(256, 128), (300, 130)]
    G = [synth.gradient(m, n, -0.7, synth.rng_for(29, 0, i), synth.F32) for i, (m, n) in enumerate(shapes)]
    res = {}
    for mode in (1, 2):
        pc = sr.Preconditioner(0, timing=mode)
        L = [torch.zeros((m, m), device="cuda") for m, _ in shapes]
        R = [torch.zeros((n, n), device="cuda") for _, n in shapes]
        out = [torch.empty((m, n), device="cuda") for m, n in shapes]
        sr.precond_step(pc.h, [to_dev(g) for g in G], L, R, 0.95, 1e-6, -0.25, out=out)
        ms, launches, flops = sr.precond_get_timing(pc.h)
        gms, gn, gis = sr.precond_get_gemm_timing(pc.h)
        res[mode] = ([o.cpu() for o in out], ms, launches, flops, gms, gn, gis)
        pc.close()
    for a, b in zip(res[1][0], res[2][0]):
        assert torch.equal(a, b)
    for mode in (1, 2):
        assert all(x > 0 for x in res[mode][1]), res[mode][1]
    assert res[1][4] > 0 and res[2][4] == -1.0
    assert res[1][5] == res[2][5] == res[1][2] > 0
    assert res[1][6] == res[2][6] > 0 and res[1][3] == res[2][3] > 0


def test_tile_split_gives_identical_results():
    """PRECOND_OPT_TILE_SPLIT = 1, 2, 4: small products spread each tile over that
    many CTAs, each writing a share of its outputs; the update, the roots and
    the iteration counts are the same bit for bit (full and packed state), and
    the split run still meets the oracle."""
    import torch
    import shampoo_roots_gb300 as sr
    shapes = [(256, 128), (300, 130), (384, 200)]
    G = [synth.gradient(m, n, -0.7, synth.rng_for(31, 0, i), synth.F32) for i, (m, n) in enumerate(shapes)]
    for packed in (0, 1):
        res = {}
        for split in (1, 2, 4):
            pc = sr.Preconditioner(0, tile_split=split, packed_state=packed, engine=2)
            side = (lambda d: d * (d + 1) // 2) if packed else (lambda d: d * d)
            L = [torch.zeros(side(m), device="cuda") for m, _ in shapes]
            R = [torch.zeros(side(n), device="cuda") for _, n in shapes]
            if not packed:
                L = [x.view(m, m) for x, (m, _) in zip(L, shapes)]
                R = [x.view(n, n) for x, (_, n) in zip(R, shapes)]
            out = [torch.empty((m, n), device="cuda") for m, n in shapes]
            sr.precond_step(pc.h, [to_dev(g) for g in G], L, R, 0.95, 1e-6, -0.25, out=out)
            torch.cuda.synchronize()
            iters = sr.precond_get_stats(pc.h, 2 * len(shapes))[0]
            roots = []
            for i, (m, n) in enumerate(shapes):
                xl, xr = torch.empty((m, m), device="cuda"), torch.empty((n, n), device="cuda")
                sr.precond_get_root(pc.h, 2 * i, xl)
                sr.precond_get_root(pc.h, 2 * i + 1, xr)
                roots += [xl.cpu(), xr.cpu()]
            res[split] = ([o.cpu() for o in out], [x.cpu() for x in L + R] + roots, list(iters))
            pc.close()
        for split in (2, 4):
            for a, b in zip(res[1][0] + res[1][1], res[split][0] + res[split][1]):
                assert torch.equal(a, b), (packed, split)
            assert res[1][2] == res[split][2]
    st = oracle.OracleState(shapes)
    Uo, _, _ = oracle.precond_step(st, [g.astype(np.float64) for g in G], 0.95, 1e-6, -0.25)
    for u, uo in zip(res[4][0], Uo):
        assert oracle.rel_fro(u.double().numpy(), uo) <= TOL
