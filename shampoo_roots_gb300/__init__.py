"""Python binding of libprecond (ctypes).

Argument marshalling only: every step of the preconditioner runs in the CUDA
library.  The names follow the C ABI of include/precond.h.  torch tensors are
accepted wherever the C ABI takes device pointers; torch supplies device
memory and streams, nothing else.  If the library is not built, every call
raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libprecond.so")

OK, EINVAL, ENOMEM, ECUDA, ENODEV, ENOTCONV, ENONFINITE = 0, -1, -2, -3, -4, -5, -6
F32, BF16 = 0, 1
OPT_TOL, OPT_MAX_ITER, OPT_MIN_ITER, OPT_ENGINE, OPT_SMALL_DIM, OPT_WORKSPACE_MAX, OPT_TIMING, OPT_USE_GRAPH, \
    OPT_CLASSICAL, OPT_FOLD, OPT_BRANCHES, OPT_STEP_DEGREE, OPT_PACKED_STATE, OPT_TILE_SPLIT = range(1, 15)

_lib = None


class PrecondError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {error_string(code)} ({code})")


def load():
    """Load libprecond.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with shampoo_roots_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
    L.precond_create.argtypes = [ctypes.POINTER(vp), i32]
    L.precond_destroy.argtypes = [vp]
    L.precond_step.argtypes = [vp, i32, ctypes.POINTER(vp), i32, ctypes.POINTER(i64), ctypes.POINTER(vp),
                               ctypes.POINTER(vp), f32, f32, f32, ctypes.POINTER(vp), vp]
    L.precond_inv_root.argtypes = [vp, i32, ctypes.POINTER(vp), ctypes.POINTER(i64), f32, f32,
                                   ctypes.POINTER(vp), vp]
    L.precond_get_stats.argtypes = [vp, i32, ctypes.POINTER(i32), ctypes.POINTER(f32), ctypes.POINTER(i32),
                                    ctypes.POINTER(f32)]
    L.precond_set_option.argtypes = [vp, i32, f64]
    L.precond_get_timing.argtypes = [vp, ctypes.POINTER(f64), ctypes.POINTER(i64), ctypes.POINTER(f64)]
    L.precond_launch_count.argtypes = [vp]
    L.precond_get_gemm_timing.argtypes = [vp, ctypes.POINTER(f64), ctypes.POINTER(i64), ctypes.POINTER(f64)]
    L.precond_get_workspace.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    L.precond_launch_count.restype = i64
    L.precond_get_root.argtypes = [vp, i32, vp, vp]
    L.precond_debug_plane.argtypes = [vp, i32, i32, vp, vp]
    L.precond_inv_root_noalloc.argtypes = [vp, i64, f32, f32, vp, vp, ctypes.POINTER(i32)]
    L.precond_gemm_selftest.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, i32, vp]
    L.precond_step_schedule.argtypes = [i32, f64, f64, i32, i32, ctypes.POINTER(f64), ctypes.POINTER(f64),
                                        ctypes.POINTER(f64), ctypes.POINTER(f64), ctypes.POINTER(i32)]
    L.precond_error_string.argtypes = [i32]
    L.precond_error_string.restype = ctypes.c_char_p
    for name in ("precond_create", "precond_destroy", "precond_step", "precond_inv_root", "precond_get_stats",
                 "precond_set_option", "precond_get_timing", "precond_get_root", "precond_gemm_selftest",
                 "precond_debug_plane", "precond_get_gemm_timing", "precond_get_workspace",
                 "precond_inv_root_noalloc", "precond_step_schedule"):
        getattr(L, name).restype = i32
    _lib = L
    return L


def error_string(code: int) -> str:
    return load().precond_error_string(int(code)).decode()


precond_error_string = error_string


def precond_step_schedule(p: int, l0: float, fold: float = 0.3, degree: int = 2, max_steps: int = 60):
    """The iteration's per-step minimax schedule: lists (alpha, beta, gamma, lo)
    of T_k(m) = alpha_k - beta_k m + gamma_k m^2 and each step's interval bottom."""
    arrs = [(ctypes.c_double * max_steps)() for _ in range(4)]
    n = ctypes.c_int()
    _check(load().precond_step_schedule(int(p), float(l0), float(fold), int(degree), int(max_steps), *arrs,
                                        ctypes.byref(n)), "precond_step_schedule")
    return tuple([a[i] for i in range(n.value)] for a in arrs)


def _check(code: int, what: str) -> int:
    if code != OK:
        raise PrecondError(code, what)
    return code


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _ptr_array(xs):
    arr = (ctypes.c_void_p * len(xs))()
    for i, x in enumerate(xs):
        arr[i] = _ptr(x)
    return arr


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def precond_create(cuda_device: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(load().precond_create(ctypes.byref(h), int(cuda_device)), "precond_create")
    return h.value


def precond_destroy(h) -> None:
    _check(load().precond_destroy(h), "precond_destroy")


def precond_set_option(h, key: int, value: float) -> None:
    _check(load().precond_set_option(h, int(key), float(value)), "precond_set_option")


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"gradients must be float32 or bfloat16, got {t.dtype}")


def precond_step(h, grads: Sequence, L: Sequence, R: Sequence, beta: float, eps: float, power: float,
                 out: Optional[Sequence] = None, stream=None, raw: bool = False) -> int:
    """One preconditioner step (see include/precond.h).  ``grads``, ``L``,
    ``R`` and ``out`` are CUDA tensors (contiguous; fp32 state and outputs)."""
    n = len(grads)
    if n == 0 or len(L) != n or len(R) != n or (out is not None and len(out) != n):
        raise ValueError("grads, L, R (and out) must have the same non-zero length")
    dt = _dtype_code(grads[0])
    shapes = (ctypes.c_int64 * (2 * n))()
    for i, g in enumerate(grads):
        if g.dim() != 2 or not g.is_contiguous() or _dtype_code(g) != dt:
            raise ValueError("every gradient must be a contiguous 2-D tensor of one dtype")
        shapes[2 * i], shapes[2 * i + 1] = g.shape
    for t in list(L) + list(R) + list(out or []):
        if not t.is_contiguous():
            raise ValueError("state and output tensors must be contiguous")
    outs = _ptr_array(out) if out is not None else None
    code = load().precond_step(h, n, _ptr_array(grads), dt, shapes, _ptr_array(L), _ptr_array(R),
                               float(beta), float(eps), float(power), outs, _stream(stream))
    return code if raw else _check(code, "precond_step")


def precond_inv_root(h, A: Sequence, X: Sequence, eps: float, power: float, stream=None, raw: bool = False) -> int:
    n = len(A)
    if n == 0 or len(X) != n:
        raise ValueError("A and X must have the same non-zero length")
    dims = (ctypes.c_int64 * n)()
    for i, a in enumerate(A):
        if a.dim() != 2 or a.shape[0] != a.shape[1] or not a.is_contiguous():
            raise ValueError("every A must be a contiguous square matrix")
        dims[i] = a.shape[0]
    code = load().precond_inv_root(h, n, _ptr_array(A), dims, float(eps), float(power), _ptr_array(X),
                                   _stream(stream))
    return code if raw else _check(code, "precond_inv_root")


def precond_get_stats(h, nroots: int):
    """Returns (iters, resid, status, scale) lists of the last call's roots."""
    it = (ctypes.c_int * nroots)()
    rs = (ctypes.c_float * nroots)()
    stt = (ctypes.c_int * nroots)()
    sc = (ctypes.c_float * nroots)()
    _check(load().precond_get_stats(h, nroots, it, rs, stt, sc), "precond_get_stats")
    return list(it), list(rs), list(stt), list(sc)


def precond_get_timing(h):
    ms = (ctypes.c_double * 4)()
    nl = ctypes.c_int64()
    fl = ctypes.c_double()
    _check(load().precond_get_timing(h, ms, ctypes.byref(nl), ctypes.byref(fl)), "precond_get_timing")
    return list(ms), nl.value, fl.value


def precond_get_gemm_timing(h):
    """(milliseconds, launches, issued bf16 MMA FLOPs) of the last call's iteration-stage GEMMs."""
    ms = ctypes.c_double()
    n = ctypes.c_int64()
    fl = ctypes.c_double()
    _check(load().precond_get_gemm_timing(h, ctypes.byref(ms), ctypes.byref(n), ctypes.byref(fl)),
           "precond_get_gemm_timing")
    return ms.value, n.value, fl.value


def precond_get_workspace(h):
    """(planned bytes of the last validated call, device bytes held now)."""
    planned, held = ctypes.c_int64(), ctypes.c_int64()
    _check(load().precond_get_workspace(h, ctypes.byref(planned), ctypes.byref(held)), "precond_get_workspace")
    return planned.value, held.value


def precond_launch_count(h) -> int:
    return int(load().precond_launch_count(h))


def precond_get_root(h, r: int, dst, stream=None) -> None:
    _check(load().precond_get_root(h, int(r), _ptr(dst), _stream(stream)), "precond_get_root")


def precond_debug_plane(h, r: int, which: int, dst, stream=None) -> None:
    _check(load().precond_debug_plane(h, int(r), int(which), _ptr(dst), _stream(stream)), "precond_debug_plane")


NOALLOC_MAX_D = 256


def precond_inv_root_noalloc(A, X, eps: float, power: float, stream=None, raw: bool = False):
    """Allocation-free inverse root of one d x d matrix (d <= NOALLOC_MAX_D);
    returns (return code, per-root status)."""
    if A.dim() != 2 or A.shape[0] != A.shape[1] or not A.is_contiguous() or not X.is_contiguous():
        raise ValueError("A must be a contiguous square matrix and X contiguous")
    st = ctypes.c_int(0)
    code = load().precond_inv_root_noalloc(_ptr(A), int(A.shape[0]), float(eps), float(power), _ptr(X),
                                           _stream(stream), ctypes.byref(st))
    if not raw:
        _check(code, "precond_inv_root_noalloc")
    return code, st.value


def precond_gemm_selftest(h, engine: int, A, B, C, passes: int = 3, stream=None) -> None:
    M, K = A.shape
    N = B.shape[0]
    _check(load().precond_gemm_selftest(h, int(engine), M, N, K, _ptr(A), _ptr(B), _ptr(C), int(passes),
                                        _stream(stream)), "precond_gemm_selftest")


class Preconditioner:
    """Owns a handle (and, optionally, the fp32 EMA state of a list of shapes)."""

    def __init__(self, device: int = 0, **options):
        self.h = precond_create(device)
        self.device = device
        for k, v in options.items():
            precond_set_option(self.h, globals()["OPT_" + k.upper()], v)

    def set_option(self, key: str, value: float) -> None:
        precond_set_option(self.h, globals()["OPT_" + key.upper()], value)

    def close(self) -> None:
        if self.h:
            precond_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
