"""Benchmark of the matrix-preconditioner step on GB300.

A step = one call of the whole hot path (Gram EMAs, statistics and bound,
coupled Newton-Schulz roots, two-sided apply) over one batch of synthetic
gradients.  The default workload is the largest one that fits one GPU, the
wide stack: 16 fp32 gradients of 6144 x 6144 and 16 of 6144 x 3072
(s_i ~ i^-0.5), fp32 Grams, power -1/4: 32 weight matrices, 64 roots
(48 of side 6144, 16 of side 3072).  `--workload N` selects the others.

Prints ONE JSON line (rank 0).  `value` is whole-job throughput in
preconditioner steps per second (1000 / ms_per_step per GPU, summed over
ranks); `tflops_algorithmic` is the step's algorithmic FLOPs (2mnk per logical
GEMM, iterations actually executed) over its time; `e2e` is the throughput
with the gradients copied from pinned host memory and the update copied back
inside the timed region.  `--impl reference` times the float64 CPU oracle on
whole preconditioner steps of the same workload (as many as fit a few
minutes, at least one) and says how many it ran.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "preconditioner step ms and TFLOP/s (% GB300 tensor peak) vs CPU oracle"
WORKLOAD_INDEX = 4          # default: the wide stack (16 x 6144^2 + 16 x 6144x3072), power -1/4


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of every rank's x: a job's time is its slowest rank's."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, steps: int, elapsed: float) -> float:
    """Whole-job preconditioner steps per second: every rank ran `steps` steps
    of its own stack (weak scaling) within `elapsed` seconds."""
    return world * steps / elapsed


def rank_step_seed(rank: int, step: int) -> int:
    """Gradient-draw index of a rank's step: ranks draw disjoint batches."""
    return 1000 * rank + step


# DRAM traffic of the dominant kernel, from ncu captures (dram__bytes_read.sum +
# dram__bytes_write.sum) of one whole iteration (E, X', D, F, M') of a small
# case per root class: 2 roots of 6144^2 and 8 of 3072^2 (the wide stack), 5 of
# 4096^2 and 64 of 1024^2 (the 24-layer stack), each 2300-2600 tiles of
# 128 x 128 (as many tiles in flight per SM as at full size).  Bytes
# per output element and product, averaged over the iteration; the bench scales
# them by the elements each root class computed in the step.  The algorithmic
# bytes are 6 B of digits per element for each distinct operand read and 6 B
# written (the element-wise input is the A operand, taken from the operand
# ring: no extra read), 14.4 B on average over an iteration.  Valid only for
# the kernel sources the captures were taken on (their SHA-1s), the default
# options and the quadratic p = 4 steps (4 products in the first iteration, 5
# after).
TRAFFIC_CAPTURES = {
    1: {"bytes_per_element": {4096: 26.32, 1024: 14.93}, "algorithmic_bytes_per_element": 14.4,
        "power": -0.25,
        "sources": {"gemm_tc.cuh": "e2e7297b0c5888ec741d4361631d99f23c44111e",
                    "engine.cuh": "23828dc074daf405d0bc22da5e5d8ffca1abbfdb",
                    "common.cuh": "bde15094817cdd9be373c93fc049db220e42550e"}},
    4: {"bytes_per_element": {6144: 35.82, 3072: 19.06}, "algorithmic_bytes_per_element": 14.4,
        "power": -0.25,
        "sources": {"gemm_tc.cuh": "e2e7297b0c5888ec741d4361631d99f23c44111e",
                    "engine.cuh": "23828dc074daf405d0bc22da5e5d8ffca1abbfdb",
                    "common.cuh": "bde15094817cdd9be373c93fc049db220e42550e"}},
}


# options that change how the products run, not which products run or their operands
LAUNCH_ONLY_OPTS = ("tile_split", "branches", "use_graph", "packed_state")


def captured_traffic(workload: int, power: float, opts, root_dims, root_iters, launches: float):
    """(traffic, algorithmic bytes) per launch of the dominant kernel over the
    step's launch mix, or (None, None) when no capture covers this run or the
    kernel changed since."""
    import hashlib
    cap = TRAFFIC_CAPTURES.get(workload)
    if cap is None or opts or power != cap["power"] or not launches:
        return None, None
    for name, digest in cap["sources"].items():
        with open(os.path.join(ROOT, "shampoo_roots_gb300", "csrc", name), "rb") as f:
            if hashlib.sha1(f.read()).hexdigest() != digest:
                return None, None
    measured = 0.0
    for d, k in zip(root_dims, root_iters):
        if d not in cap["bytes_per_element"] or k < 1:
            return None, None
        products = 4 + 5 * (k - 1)
        measured += products * d * d * cap["bytes_per_element"][d]
    algorithmic = iteration_bytes(power, opts, root_dims, root_iters)
    return measured / launches, algorithmic / launches


def iteration_bytes(power: float, opts, root_dims, root_iters):
    """Algorithmic DRAM bytes of the step's iteration-stage products with the
    default options: 6 B of digits per element for each distinct operand read
    and 6 B written.  p = 4 takes quadratic steps (4 products in the first
    iteration: 3 with one operand and M' with two, 13.5 B per element on
    average; 5 after, 14.4 B); p = 2 takes linear steps (D = M M and M', then X'
    too: 30 B, then 48 B per element and iteration).  None for options that
    change the products (engine, step degree, classical steps, tolerances);
    options that change only how they run leave the bytes as they are."""
    if any(k not in LAUNCH_ONLY_OPTS for k in opts):
        return None
    total = 0.0
    for d, k in zip(root_dims, root_iters):
        if k < 1:
            continue
        if power == -0.25:
            total += (54.0 + 72.0 * (k - 1)) * d * d
        elif power == -0.5:
            total += (30.0 + 48.0 * (k - 1)) * d * d
        else:
            return None
    return total


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def step_flops_outside_roots(shapes):
    """Algorithmic FLOPs of the Gram EMAs and the apply (2mnk per product)."""
    f = 0.0
    for m, n in shapes:
        f += 2.0 * m * m * n + 2.0 * n * n * m      # L = G G^T, R = G^T G
        f += 2.0 * m * n * n + 2.0 * m * m * n      # V = G X_R, U = X_L V
    return f


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            # wait (at most 3 s) for the sampler's first line, so that a short region
            # still has the sample taken as it starts
            t0 = time.time()
            while time.time() - t0 < 3.0 and os.path.getsize(self.path) == 0:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if not self.path or not os.path.exists(self.path):
            return out
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return out
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        out.update(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(mx) if mx else None,
                   reasons=reasons, samples=len(rows))
        return out


def oracle_sample(w, seconds_budget=20.0):
    """Time the float64 oracle on one matrix of each shape class of the stack
    (one EMA step from zero Grams) and extrapolate to the whole stack.
    Returns (oracle seconds per full step, sample description, cores)."""
    import numpy as np
    from oracle import roots as oracle
    from workloads import synth
    classes = {}
    for i, s in enumerate(w.shapes):
        classes.setdefault(s, []).append(i)
    per_class = {}
    t_used = 0.0
    for shape, idx in classes.items():
        G = synth.gradients_for_step(w, 0, [idx[0]])[0].astype(np.float64)
        st = oracle.OracleState([shape])
        t0 = time.perf_counter()
        oracle.precond_step(st, [G], w.beta, w.eps, w.powers[0])
        dt = time.perf_counter() - t0
        per_class[shape] = (dt, len(idx))
        t_used += dt
        if t_used > seconds_budget:
            break
    total = sum(dt * cnt for dt, cnt in per_class.values())
    # classes not sampled within the budget are extrapolated by d^3
    for shape, idx in classes.items():
        if shape not in per_class:
            ref_shape, (dt, _) = next(iter(per_class.items()))
            scale = (max(shape) / max(ref_shape)) ** 3
            total += dt * scale * len(idx)
    desc = ("one matrix of each shape class " + ", ".join(f"{m}x{n}" for (m, n) in per_class) +
            f" (one EMA step, {t_used:.1f} s), extrapolated to all {len(w.shapes)} matrices")
    return total, desc, os.cpu_count()


def oracle_sample_spd(w, power, n=2):
    """Time the oracle on `n` of the SPD matrices; extrapolate to all of them."""
    import numpy as np
    from oracle import roots as oracle
    from workloads import synth
    A = synth.spd_inputs(w, matrices=range(n))
    t0 = time.perf_counter()
    for a in A:
        oracle.inv_root(a.astype(np.float64), w.eps, power)
    dt = time.perf_counter() - t0
    return dt / n * w.count, f"{n} of the {w.count} SPD {w.dims[0]}^2 matrices ({dt:.1f} s), extrapolated", os.cpu_count()


# The arithmetic of the path: fp32 values; every product on bf16 tensor cores as
# exact products of three 9-bit bf16 digits under a power-of-two scale per (row,
# 128-column block), six digit products per K step accumulated in tensor memory
# over one 128-wide K block and summed across blocks in fp32 registers; fp32
# storage between products.
DTYPE = "fp32 (exact bf16x3 digit products)"
DTYPE_NOTE = ("fp32 matrices; products as exact bf16 digit products on tensor cores (3 digits of 9 bits "
              "per (row, 128-column block) scale, six digit products per K step, per-block sums in fp32), "
              "about 2^-26 relative to the block scales")
SM_COUNT = 152
BF16_FLOPS_PER_CLK_SM = 8192.0     # dense bf16 tensor-core rate per SM and clock (2 x 4096 FMA)

REFERENCE_BUDGET_S = 300.0     # reference arm: time budget for whole oracle steps

L2_NOTE = ("inputs larger than L2 (129 MB): the state and input matrices of every workload but the "
           "single 256x128 one, which flushes L2 with a 256 MB write between timed steps")


def synth_workload(index):
    from workloads import synth
    return synth.workload(index)


def parse_opts(args):
    return {k: float(v) for k, v in (o.split("=", 1) for o in args.opt)}


def workload_config(w, power, opts):
    """The `config` object of both arms' JSON lines (identical for the same run)."""
    nroots = 2 * w.count if w.kind == "step" else w.count
    return {"workload": w.name, "matrices": w.count, "roots": nroots, "grad_dtype": w.dtype,
            "power": power, "beta": w.beta if w.kind == "step" else None, "eps": w.eps,
            "options": opts, "l2": L2_NOTE}


def _reference_inputs(w):
    """Inputs of one step of workload `w` for the reference arm, drawn on the host
    with the torch backend of the same recipe (fp32 QR).  Step workloads draw one
    gradient per shape class and pass it for every matrix of that class: the
    oracle's work does not depend on the values, and the float64 draws of the
    largest stacks would otherwise take minutes.  Returns float64 arrays."""
    import numpy as np
    from workloads import synth
    if w.kind == "step":
        first = {}
        for i, s in enumerate(w.shapes):
            first.setdefault(s, i)
        drawn = dict(zip(first.keys(), synth.torch_gradients_for_step(w, 0, "cpu", matrices=list(first.values()))))
        return [drawn[s].float().numpy().astype(np.float64) for s in w.shapes]
    return [a.numpy().astype(np.float64) for a in synth.torch_spd_inputs(w, "cpu")]


def run_reference(args):
    """Reference arm: the float64 CPU oracle, as it stands, on whole steps of the
    workload.  Small workloads run the requested warm-up and timed steps; when one
    oracle step takes long (the largest stacks need minutes), the arm runs as many
    whole steps as fit REFERENCE_BUDGET_S (at least one, no warm-up: the oracle
    has nothing to warm up) and reports the counts it actually ran."""
    from oracle import roots as oracle
    from workloads import synth
    w = synth.workload(args.workload)
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    power = args.power if args.power is not None else w.powers[0]
    inputs = _reference_inputs(w)
    state = [None]

    def one_step():
        t0 = time.perf_counter()
        if w.kind == "step":
            if state[0] is None:
                state[0] = oracle.OracleState(list(w.shapes))
            oracle.precond_step(state[0], inputs, w.beta, w.eps, power)
        else:
            for a in inputs:
                oracle.inv_root(a, w.eps, power)
        return time.perf_counter() - t0

    first = one_step()                 # a whole step; decides how many more fit
    warm_run, timed = 0, []
    if first * (args.warmup + args.steps) <= REFERENCE_BUDGET_S:
        warm_run = 1
        for _ in range(args.warmup - 1):
            one_step()
            warm_run += 1
        for _ in range(args.steps):
            timed.append(one_step())
    else:
        timed.append(first)
        used = first
        while len(timed) < args.steps and used + first <= REFERENCE_BUDGET_S:
            timed.append(one_step())
            used += timed[-1]
    per_step = statistics.median(timed)
    value = 1.0 / per_step
    sample = (f"{len(timed)} whole oracle step(s) of all {w.count} matrices "
              f"(EMA state carried from step to step; the same inputs every step"
              f"{', one drawn gradient per shape class' if w.kind == 'step' else ''}), "
              f"{warm_run} warm-up step(s); timed {sum(timed):.1f} s")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "preconditioner steps/s",
            "n_gpus": args.gpus, "steps": len(timed), "warmup": warm_run,
            "requested": {"steps": args.steps, "warmup": args.warmup},
            "ms_per_step": per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "extrapolated": False,
            "config": workload_config(w, power, parse_opts(args)),
            "cpu_baseline": {"value": value, "unit": "preconditioner steps/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "preconditioner steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def profile_small(args):
    """A small case for ncu captures: inverse quarter roots of a few SPD
    matrices of the conditioning-stress recipe (default 4 of 2048^2; a few GB
    on the device at most)."""
    import dataclasses
    import torch
    import shampoo_roots_gb300 as sr
    from workloads import synth
    w = synth.workload(3)
    dev = torch.device("cuda")
    if args.profile_dim == 2048 and args.profile_count == 4:
        A = [torch.from_numpy(a).to(dev) for a in synth.spd_inputs(w, matrices=range(4))]
    else:
        wp = dataclasses.replace(w, dims=(args.profile_dim,) * args.profile_count)
        A = synth.torch_spd_inputs(wp, dev)
    X = [torch.empty_like(a) for a in A]
    pc = sr.Preconditioner(0)
    for _ in range(args.warmup + args.steps):
        sr.precond_inv_root(pc.h, A, X, w.eps, -0.25)
    torch.cuda.synchronize()
    it, _, status, _ = sr.precond_get_stats(pc.h, len(A))
    pc.close()
    print(json.dumps({"profile_small": True, "iterations": it, "status": status}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--workload", type=int, default=WORKLOAD_INDEX,
                    help="0 single 256x128, 1 stack p=-1/4 (default), 2 stack p=-1/2, 3 SPD 64x2048^2, 4 wide 6144")
    ap.add_argument("--power", type=float, default=None, help="override the workload's power")
    ap.add_argument("--opt", action="append", default=[], metavar="KEY=VALUE",
                    help="handle option (PRECOND_OPT_KEY, lower case), e.g. tol=1e-5")
    ap.add_argument("--profile-dim", type=int, default=2048, help="profiling case: matrix side")
    ap.add_argument("--profile-count", type=int, default=4, help="profiling case: number of matrices")
    ap.add_argument("--profile-small", action="store_true",
                    help="profiling case: roots of 4 SPD 2048^2 matrices, no JSON line")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.profile_small:
        return profile_small(args)

    import torch
    import shampoo_roots_gb300 as sr
    from workloads import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    w = synth.workload(args.workload)
    power = args.power if args.power is not None else w.powers[0]
    opts = parse_opts(args)
    # per-stage CUDA events only: an event node between every pair of GEMMs in the captured
    # graph would cost the small workloads a third of their step
    pc = sr.Preconditioner(local, timing=2, **opts)
    if w.kind == "step":
        shapes = list(w.shapes)
        nroots = 2 * len(shapes)
        # two distinct gradient batches (ranks draw from their own seeds: weak scaling)
        pools = [synth.torch_gradients_for_step(w, rank_step_seed(rank, s), dev) for s in range(2)]
        L = [torch.zeros((m, m), device=dev) for m, _ in shapes]
        R = [torch.zeros((n, n), device=dev) for _, n in shapes]
        out = [torch.empty((m, n), device=dev) for m, n in shapes]

        def step(i):
            sr.precond_step(pc.h, pools[i % 2], L, R, w.beta, w.eps, power, out=out, stream=stream)
    else:
        shapes = []
        nroots = w.count
        A = synth.torch_spd_inputs(w, dev)
        Xo = [torch.empty_like(a) for a in A]

        def step(i):
            sr.precond_inv_root(pc.h, A, Xo, w.eps, power, stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # ---------------- timed region (device-resident inputs)
    launches0 = sr.precond_launch_count(pc.h)
    # workloads whose data fit in L2 (the single 256x128 matrix) get an L2 flush
    # (a 256 MB write) between timed steps, outside the steps' events
    flush = torch.empty((64 << 20,), device=dev) if w.index == 0 else None
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with Clocks(local) as clk:
        barrier()
        # the steps go back to back (no host synchronisation between them); the library's
        # per-stage events and counters then describe the last step, which stands for every
        # step of the region (same shapes, same iteration counts)
        for i in range(args.steps):
            if flush is not None:
                flush.zero_()
            evs[i][0].record(stream)
            step(i)
            evs[i][1].record(stream)
        barrier()
        ms, nl, fl = sr.precond_get_timing(pc.h)
        _, gn, gis = sr.precond_get_gemm_timing(pc.h)
        it, _, _, _ = sr.precond_get_stats(pc.h, nroots)
    stage_ms = [x * args.steps for x in ms]
    root_flops = fl * args.steps
    issued_flops = gis * args.steps
    gemm_ms = ms[2] * args.steps        # the iteration stage: its GEMM launches (and the quadratic steps' shift)
    gemm_n = gn * args.steps
    iters_seen = [statistics.mean(it)]
    last_iters = list(it)
    elapsed = sum(a.elapsed_time(b) for a, b in evs) / 1e3
    gpu_launches = sr.precond_launch_count(pc.h) - launches0
    elapsed = max_over_ranks(elapsed, dist, dev)
    step_flops = step_flops_outside_roots(shapes) + root_flops / args.steps
    value = job_rate(world, args.steps, elapsed)               # preconditioner steps per second, whole job
    tflops = world * step_flops * args.steps / elapsed / 1e12
    ms_per_step = elapsed / args.steps * 1e3

    # ---------------- end to end: pinned host gradients in, update out, inside the timed region.
    # As a training loop would: step i+1's gradients go up and step i's update comes
    # down on copy streams of their own while step i computes (two device buffers each).
    e2e = None
    if not args.no_e2e and w.kind == "step":
        host_g = [[g.cpu().pin_memory() for g in pool] for pool in pools]
        host_u = [torch.empty((m, n), dtype=torch.float32).pin_memory() for m, n in shapes]
        dev_g = [[torch.empty_like(g) for g in pools[0]] for _ in range(2)]
        dev_u = [out, [torch.empty_like(o) for o in out]]
        h2d = sum(g.numel() * g.element_size() for g in host_g[0])
        d2h = sum(u.numel() * u.element_size() for u in host_u)
        cs_in, cs_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event()
        ev_h = [ev() for _ in range(args.steps)]      # step i's gradients are on the device
        ev_c = [ev() for _ in range(args.steps)]      # step i computed
        ev_d = [ev() for _ in range(args.steps)]      # step i's update is on the host

        def upload(i):
            with torch.cuda.stream(cs_in):
                for dg, hg in zip(dev_g[i % 2], host_g[i % 2]):
                    dg.copy_(hg, non_blocking=True)
                ev_h[i].record(cs_in)

        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cs_in)
        upload(0)
        for i in range(args.steps):
            stream.wait_event(ev_h[i])
            if i >= 2:
                stream.wait_event(ev_d[i - 2])          # dev_u[i % 2] has been copied out
            sr.precond_step(pc.h, dev_g[i % 2], L, R, w.beta, w.eps, power, out=dev_u[i % 2], stream=stream)
            ev_c[i].record(stream)
            if i + 1 < args.steps:
                if i >= 1:
                    cs_in.wait_event(ev_c[i - 1])       # dev_g[(i + 1) % 2] was read by step i - 1
                upload(i + 1)
            cs_out.wait_event(ev_c[i])
            with torch.cuda.stream(cs_out):
                for hu, o in zip(host_u, dev_u[i % 2]):
                    hu.copy_(o, non_blocking=True)
                ev_d[i].record(cs_out)
        cs_in.wait_event(ev_d[args.steps - 1])
        e1.record(cs_in)
        barrier()
        t_e2e = e0.elapsed_time(e1) / 1e3
        t_e2e = max_over_ranks(t_e2e, dist, dev)
        e2e = {"value": job_rate(world, args.steps, t_e2e), "unit": "preconditioner steps/s",
               "ms_per_step": t_e2e / args.steps * 1e3, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "overlap": "next step's upload and last step's download on copy streams during compute"}
        if flush is not None:
            e2e["l2"] = "steps back to back with no L2 flush between them (the device-timed steps flush)"

    peaks = load_peaks()
    # dominant kernel: the tcgen05 GEMM of the iteration stage (timed inside a long step -> sustained peak).
    # Its time is the iteration stage's (CUDA events on the launching stream around the stage): the
    # stage holds those GEMM launches and, for quadratic steps, one small shift kernel per root class,
    # so the per-launch time is an upper bound and the rates lower bounds.
    achieved = (root_flops / (gemm_ms / 1e3) / 1e12) if gemm_ms > 0 else None
    peak = peaks["bf16_tflops_sustained"]
    # issued: tiles actually run (upper triangles of symmetric products) x 6 bf16 digit products,
    # counted once per CTA that computed them (a launch of few tiles repeats each on up to 4 CTAs)
    issued = (issued_flops / (gemm_ms / 1e3) / 1e12) if gemm_ms > 0 else None
    root_dims = [d for m, n in shapes for d in (m, n)] if w.kind == "step" else list(w.dims)
    traffic, traffic_alg = captured_traffic(w.index, power, opts, root_dims, last_iters,
                                            gemm_n / args.steps if args.steps else 0)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": (achieved / peak) if achieved else None, "traffic": traffic,
                "traffic_algorithmic": traffic_alg,
                "kernel": "gemm_tc_kernel (iteration-stage products)",
                "launch_time": "iteration-stage events / its GEMM launches",
                "peak_kind": f"bf16 dense, sustained ({peaks['source']})",
                "issued_tflops": issued, "issued_frac": (issued / peak) if issued else None,
                "avg_launch_ms": gemm_ms / gemm_n if gemm_n else None}
    # the same products seen from HBM: algorithmic bytes over the iteration stage's time (the
    # latency-bound small workloads are far from both roofs)
    alg_bytes = iteration_bytes(power, opts, root_dims, last_iters)
    if alg_bytes is not None and gemm_ms > 0:
        gbs = alg_bytes / (gemm_ms / args.steps / 1e3) / 1e9
        roofline["hbm_view"] = {"achieved_algorithmic_gbs": gbs, "peak_gbs": peaks["hbm_gbs"],
                                "frac": gbs / peaks["hbm_gbs"], "bytes_per_step": alg_bytes}
    clk_summary = clk.summary()
    if clk_summary.get("sm_mhz") and achieved:
        # secondary view: against the tensor cores' nominal dense bf16 rate at the
        # sampled median SM clock (the measured peak above is a torch.matmul rate)
        nominal = SM_COUNT * BF16_FLOPS_PER_CLK_SM * clk_summary["sm_mhz"] * 1e6 / 1e12
        roofline["nominal_at_clock"] = {"peak": nominal, "sm_mhz": clk_summary["sm_mhz"],
                                        "frac_algorithmic": achieved / nominal,
                                        "frac_issued": (issued / nominal) if issued else None}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        if w.kind == "step":
            t_oracle, desc, cores = oracle_sample(w)
        else:
            t_oracle, desc, cores = oracle_sample_spd(w, power)
        cpu = {"value": 1.0 / t_oracle, "unit": "preconditioner steps/s", "cores": cores, "kind": "oracle",
               "sample": desc, "ms_per_step_extrapolated": t_oracle * 1e3}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "preconditioner steps/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": DTYPE, "data": "synthetic",
                "config": workload_config(w, power, opts),
                "mean_iterations": statistics.mean(iters_seen) if iters_seen else None,
                "numerics": DTYPE_NOTE,
                "tflops_algorithmic": tflops,
                "pct_tensor_peak": tflops / peaks["bf16_tflops"],
                "stages_ms_per_step": {k: v / args.steps for k, v in zip(
                    ("prep_gram", "bound_start", "iterations", "finish_apply"), stage_ms)},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": gpu_launches,
                "clocks": clk_summary}
        print(json.dumps(line), flush=True)
    pc.close()
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
