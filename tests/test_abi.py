"""CPU tests of the C ABI: the library loads, exports every declared entry
point, and its host-side validation / planning behaves as documented.  No
GPU work: a host-only handle (cuda_device = -1) validates and plans only."""
import ctypes
import os
import re

import pytest

import shampoo_roots_gb300 as sr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "precond.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(precond_\w+)\s*\(", src)))


def test_exports_every_declared_symbol():
    lib = sr.load()
    names = declared_functions()
    assert len(names) >= 10, names
    for n in names:
        assert hasattr(lib, n), f"missing export {n}"


def test_error_strings():
    for code in (sr.OK, sr.EINVAL, sr.ENOMEM, sr.ECUDA, sr.ENODEV, sr.ENOTCONV, sr.ENONFINITE):
        assert sr.error_string(code) and sr.error_string(code) != "unknown status"
    assert sr.error_string(-99) == "unknown status"


def test_create_arguments():
    lib = sr.load()
    assert lib.precond_create(None, -1) == sr.EINVAL
    h = ctypes.c_void_p()
    assert lib.precond_create(ctypes.byref(h), -2) == sr.EINVAL
    assert lib.precond_create(ctypes.byref(h), -1) == sr.OK
    assert h.value
    assert lib.precond_destroy(h) == sr.OK
    assert lib.precond_destroy(None) == sr.OK


class Host:
    """A host-only handle and raw calls with fake (never dereferenced) device pointers."""

    def __init__(self):
        self.lib = sr.load()
        self.h = sr.precond_create(-1)
        self._next = 0x10000

    def fake(self):
        self._next += 0x1000000
        return self._next

    def step(self, shapes, dtype=sr.F32, beta=0.95, eps=1e-6, power=-0.25, L=None, R=None, out=False,
             grads=None, count=None):
        n = len(shapes)
        g = grads if grads is not None else [self.fake() for _ in range(n)]
        Ls = L if L is not None else [self.fake() for _ in range(n)]
        Rs = R if R is not None else [self.fake() for _ in range(n)]
        arr = lambda xs: (ctypes.c_void_p * max(len(xs), 1))(*xs)
        sh = (ctypes.c_int64 * max(2 * n, 1))(*[v for s in shapes for v in s])
        outs = arr([self.fake() for _ in range(n)]) if out else None
        return self.lib.precond_step(self.h, n if count is None else count, arr(g), dtype, sh, arr(Ls), arr(Rs),
                                     ctypes.c_float(beta), ctypes.c_float(eps), ctypes.c_float(power), outs, None)

    def inv_root(self, dims, eps=1e-6, power=-0.5, same=False):
        n = len(dims)
        A = [self.fake() for _ in range(n)]
        X = list(A) if same else [self.fake() for _ in range(n)]
        arr = lambda xs: (ctypes.c_void_p * n)(*xs)
        return self.lib.precond_inv_root(self.h, n, arr(A), (ctypes.c_int64 * n)(*dims), ctypes.c_float(eps),
                                         ctypes.c_float(power), arr(X), None)

    def close(self):
        sr.precond_destroy(self.h)


@pytest.fixture
def host():
    h = Host()
    yield h
    h.close()


def test_valid_step_reaches_device_stage(host):
    assert host.step([(256, 128)]) == sr.ENODEV
    assert host.step([(1024, 4096), (4096, 1024), (3, 5)], dtype=sr.BF16, power=-0.5, out=True) == sr.ENODEV


@pytest.mark.parametrize("kw", [
    dict(power=-0.3), dict(power=0.25), dict(power=-1.0),
    dict(eps=0.0), dict(eps=-1e-6), dict(eps=float("nan")), dict(eps=float("inf")),
    dict(beta=1.0), dict(beta=-0.1), dict(beta=float("nan")),
    dict(dtype=7),
])
def test_step_rejects_bad_scalars(host, kw):
    assert host.step([(8, 4)], **kw) == sr.EINVAL


def test_step_rejects_bad_shapes_and_pointers(host):
    assert host.step([(0, 4)]) == sr.EINVAL
    assert host.step([(4, -1)]) == sr.EINVAL
    assert host.step([(4, 4)], count=0) == sr.EINVAL
    assert host.step([(4, 4)], grads=[0]) == sr.EINVAL
    assert host.step([(4, 4)], L=[0]) == sr.EINVAL
    p = host.fake()
    assert host.step([(4, 4)], L=[p], R=[p]) == sr.EINVAL            # L aliases R
    q = host.fake()
    assert host.step([(4, 4), (4, 4)], L=[q, host.fake()], R=[host.fake(), q]) == sr.EINVAL
    assert host.lib.precond_step(None, 1, None, 0, None, None, None, ctypes.c_float(0.9),
                                 ctypes.c_float(1e-6), ctypes.c_float(-0.25), None, None) == sr.EINVAL


def test_inv_root_validation(host):
    assert host.inv_root([2048] * 3) == sr.ENODEV
    assert host.inv_root([16], power=-0.25) == sr.ENODEV
    assert host.inv_root([0]) == sr.EINVAL
    assert host.inv_root([16], eps=0.0) == sr.EINVAL
    assert host.inv_root([16], power=0.5) == sr.EINVAL
    assert host.inv_root([16], same=True) == sr.EINVAL


def test_workspace_limit_gives_enomem(host):
    sr.precond_set_option(host.h, sr.OPT_WORKSPACE_MAX, 1 << 20)
    assert host.step([(4096, 4096)]) == sr.ENOMEM
    assert host.inv_root([2048]) == sr.ENOMEM
    assert host.step([(16, 8)]) == sr.ENODEV     # small plan fits in 1 MiB
    sr.precond_set_option(host.h, sr.OPT_WORKSPACE_MAX, 0)
    assert host.step([(4096, 4096)]) == sr.ENODEV


def test_options(host):
    lib = sr.load()
    assert lib.precond_set_option(host.h, 999, 1.0) == sr.EINVAL
    assert lib.precond_set_option(host.h, sr.OPT_TOL, 0.0) == sr.EINVAL
    assert lib.precond_set_option(host.h, sr.OPT_TOL, 1e-6) == sr.OK
    assert lib.precond_set_option(host.h, sr.OPT_MAX_ITER, 2.5) == sr.EINVAL
    assert lib.precond_set_option(host.h, sr.OPT_MAX_ITER, 30) == sr.OK
    assert lib.precond_set_option(host.h, sr.OPT_ENGINE, 3) == sr.EINVAL
    assert lib.precond_set_option(host.h, sr.OPT_ENGINE, 2) == sr.OK
    assert lib.precond_set_option(host.h, sr.OPT_MIN_ITER, 0) == sr.EINVAL
    for v in (0, 3, 8, 2.5):
        assert lib.precond_set_option(host.h, sr.OPT_TILE_SPLIT, v) == sr.EINVAL
    for v in (1, 2, 4):
        assert lib.precond_set_option(host.h, sr.OPT_TILE_SPLIT, v) == sr.OK
    assert lib.precond_set_option(None, sr.OPT_TOL, 1e-5) == sr.EINVAL


def test_host_handle_has_no_stats(host):
    lib = sr.load()
    assert lib.precond_get_stats(host.h, 2, None, None, None, None) == sr.ENODEV
    assert lib.precond_get_root(host.h, 0, ctypes.c_void_p(host.fake()), None) == sr.ENODEV
    assert lib.precond_launch_count(host.h) == 0


def test_option_keys_match_header():
    """Every PRECOND_OPT_* key of the header has the same value in the binding."""
    import re
    import shampoo_roots_gb300 as sr
    text = open(os.path.join(ROOT, "include", "precond.h")).read()
    keys = dict(re.findall(r"#define PRECOND_OPT_(\w+)\s+(\d+)", text))
    assert len(keys) >= 11
    for name, val in keys.items():
        assert getattr(sr, "OPT_" + name) == int(val), name


def test_bench_traffic_is_dropped_when_the_kernel_changes(monkeypatch):
    """bench.py scales the captured DRAM traffic by the elements each root class
    computed, and reports it only for the kernel sources it was captured on,
    with the default options and the captured power."""
    import hashlib
    import bench
    cap = dict(bench.TRAFFIC_CAPTURES[4])
    current = {}
    for name in cap["sources"]:
        with open(os.path.join(ROOT, "shampoo_roots_gb300", "csrc", name), "rb") as f:
            current[name] = hashlib.sha1(f.read()).hexdigest()
    monkeypatch.setitem(bench.TRAFFIC_CAPTURES, 4, dict(cap, sources=current))
    dims, iters = [6144] * 48 + [3072] * 16, [6] * 64
    t, a = bench.captured_traffic(4, -0.25, {}, dims, iters, 92)
    assert t is not None and t > a > 0
    # 48 x 6144^2 + 16 x 3072^2 elements, 29 products each at 6 iterations, over 92 launches
    assert a == pytest.approx((54 + 72 * 5) * (48 * 6144 ** 2 + 16 * 3072 ** 2) / 92)
    b = cap["bytes_per_element"]
    assert t == pytest.approx(29 * (48 * 6144 ** 2 * b[6144] + 16 * 3072 ** 2 * b[3072]) / 92)
    assert bench.captured_traffic(4, -0.5, {}, dims, iters, 92) == (None, None)
    assert bench.captured_traffic(4, -0.25, {"tol": 1e-5}, dims, iters, 92) == (None, None)
    # the HBM view's algorithmic bytes ignore options that only change how the products run
    assert bench.iteration_bytes(-0.25, {"tile_split": 1, "branches": 0}, dims, iters) == \
        bench.iteration_bytes(-0.25, {}, dims, iters) > 0
    assert bench.iteration_bytes(-0.25, {"step_degree": 1}, dims, iters) is None
    assert bench.captured_traffic(0, -0.25, {}, [256, 128], [6, 6], 96) == (None, None)
    monkeypatch.setitem(bench.TRAFFIC_CAPTURES, 4, dict(cap, sources=dict(current, **{"gemm_tc.cuh": "0" * 40})))
    assert bench.captured_traffic(4, -0.25, {}, dims, iters, 92) == (None, None)


def test_workspace_is_planned_on_a_host_only_handle(host):
    assert sr.precond_get_workspace(host.h) == (0, 0)
    assert host.step([(256, 128)]) == sr.ENODEV
    one, held = sr.precond_get_workspace(host.h)
    assert one > 0 and held == 0
    # the digit planes of both roots dominate: 3 bf16 digits per element of X (2), M (2), D and F
    assert one >= 6 * 6 * (256 * 256 + 128 * 128)
    assert host.step([(256, 128)] * 4) == sr.ENODEV
    four, _ = sr.precond_get_workspace(host.h)
    assert 3 * one < four <= 4 * one
    assert host.step([(8, 4)], eps=0.0) == sr.EINVAL          # a rejected call leaves the figure alone
    assert sr.precond_get_workspace(host.h)[0] == four
    assert host.lib.precond_get_workspace(None, None, None) == sr.EINVAL


def test_packed_state_option(host):
    assert sr.precond_set_option(host.h, sr.OPT_PACKED_STATE, 1) is None
    assert host.lib.precond_set_option(host.h, sr.OPT_PACKED_STATE, ctypes.c_double(2.0)) == sr.EINVAL
    assert host.step([(256, 128)]) == sr.ENODEV          # plans and validates with packed state


def test_tile_split_sizes_the_hand_over_scratch(host):
    """A plan of few tiles reserves hand-over slots for up to PRECOND_OPT_TILE_SPLIT
    CTAs per tile: two 128 x 128 fp32 slots per CTA in each of the plan's scratch
    regions (the call's stream and the two branch streams of each tcgen05 root
    class).  The plan bounds a product's tiles by the full square: 2 x 2 for the
    256^2 products of the single 256x128 gradient, so the split of 4 reserves
    16 CTAs' slots instead of 4."""
    slot_bytes = 2 * 128 * 128 * 4
    regions = 1 + 2 * 2                    # root classes 256 and 128, both on the tcgen05 engine
    sizes = {}
    for split in (1, 2, 4):
        assert sr.precond_set_option(host.h, sr.OPT_TILE_SPLIT, split) is None
        assert host.step([(256, 128)]) == sr.ENODEV
        sizes[split] = sr.precond_get_workspace(host.h)[0]
    assert sizes[2] - sizes[1] == regions * (8 - 4) * slot_bytes
    assert sizes[4] - sizes[1] == regions * (16 - 4) * slot_bytes
    # a plan whose products already fill the GPU reserves one CTA per SM whatever the split
    big = {}
    for split in (1, 4):
        sr.precond_set_option(host.h, sr.OPT_TILE_SPLIT, split)
        assert host.step([(4096, 4096)]) == sr.ENODEV
        big[split] = sr.precond_get_workspace(host.h)[0]
    assert big[1] == big[4]
