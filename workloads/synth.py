"""Seeded synthetic inputs for the matrix-preconditioner step.

This module only draws inputs. It holds none of the preconditioner's
arithmetic (no Gram, no normalisation, no root, no apply), so the CPU oracle
and the CUDA path can both consume what it produces without sharing code.

Recipe (the pages train on the Delphi 447M recipe and wide transformer
stacks; no dataset or weight is used here, these synthetic stacks stand in):

* gradients  G = U . diag(s) . V^T  with U, V Haar-distributed orthonormal
  factors (QR of a standard Gaussian matrix, signs fixed so diag(R) > 0,
  Mezzadri 2007), s_i = i**alpha for i = 1..min(m, n); built in float64 and
  rounded (round-to-nearest-even) to the storage dtype (fp32 or bf16);
* SPD stress matrices  A = Q . diag(lam) . Q^T  with Haar Q and
  log10(lam) ~ U(-8, 0), stored as fp32.

Seeds: ``numpy.random.default_rng(SeedSequence([config, step, matrix]))``;
the single-gradient case uses ``default_rng(0)`` exactly.  A torch backend
draws the same recipe on a CUDA device (fp32 QR) for the large stacks, where
a host float64 QR per matrix per step would dominate the set-up time.
"""
from __future__ import annotations

import dataclasses
from typing import List, Sequence, Tuple

import numpy as np

F32 = "f32"
BF16 = "bf16"


# --------------------------------------------------------------------------
# storage rounding (input preparation, not part of the method)
# --------------------------------------------------------------------------
def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float values to bfloat16 (nearest, ties to even); return float32."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = ((u + 0x7FFF + lsb) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).reshape(f.shape)


def bf16_bits(x_rounded_f32: np.ndarray) -> np.ndarray:
    """uint16 payload of values that are already exact bf16 numbers."""
    return (np.ascontiguousarray(x_rounded_f32, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == F32:
        return np.asarray(x, dtype=np.float32)
    if dtype == BF16:
        return round_to_bf16(x)
    raise ValueError(f"unknown storage dtype {dtype!r}")


# --------------------------------------------------------------------------
# numpy backend (float64 draws)
# --------------------------------------------------------------------------
def haar(n: int, k: int, rng: np.random.Generator) -> np.ndarray:
    """n x k matrix with Haar-distributed orthonormal columns (k <= n)."""
    z = rng.standard_normal((n, k))
    q, r = np.linalg.qr(z)
    sgn = np.sign(np.diagonal(r))
    sgn[sgn == 0] = 1.0
    return q * sgn[None, :]


def gradient(m: int, n: int, alpha: float, rng: np.random.Generator, dtype: str) -> np.ndarray:
    """G = U diag(s) V^T, s_i = i**alpha, rounded to ``dtype``; returned as float32 values."""
    r = min(m, n)
    u = haar(m, r, rng)
    v = haar(n, r, rng)
    s = np.arange(1, r + 1, dtype=np.float64) ** alpha
    g = (u * s[None, :]) @ v.T
    return round_to(g, dtype)


def spd(d: int, rng: np.random.Generator, log10_lo: float = -8.0, log10_hi: float = 0.0) -> np.ndarray:
    """fp32 SPD matrix Q diag(lam) Q^T, log10(lam) uniform on [log10_lo, log10_hi]."""
    q = haar(d, d, rng)
    lam = 10.0 ** rng.uniform(log10_lo, log10_hi, size=d)
    a = (q * lam[None, :]) @ q.T
    a = 0.5 * (a + a.T)
    return a.astype(np.float32)


def rng_for(config: int, step: int, matrix: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([config, step, matrix]))


# --------------------------------------------------------------------------
# workload definitions
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload.

    kind 'step'     : EMA Gram + root + apply over ``shapes`` for ``steps`` steps
    kind 'inv_root' : root of given SPD matrices of side ``dims`` (no EMA, no G)
    """
    name: str
    index: int
    kind: str
    shapes: Tuple[Tuple[int, int], ...] = ()
    dims: Tuple[int, ...] = ()
    dtype: str = F32
    alpha: float = -1.0
    steps: int = 1
    beta: float = 0.95
    eps: float = 1e-6
    powers: Tuple[float, ...] = (-0.25,)
    redraw: bool = True

    @property
    def count(self) -> int:
        return len(self.shapes) if self.kind == "step" else len(self.dims)


def transformer_stack(layers: int = 24, d: int = 1024, ffn: int = 4096) -> Tuple[Tuple[int, int], ...]:
    per_layer = [(d, d)] * 4 + [(d, ffn), (ffn, d)]
    return tuple(per_layer * layers)


def workloads() -> List[Workload]:
    wide = tuple([(6144, 6144)] * 16 + [(6144, 3072)] * 16)
    return [
        Workload("single-256x128", 0, "step", shapes=((256, 128),), dtype=F32, alpha=-1.0,
                 steps=1, powers=(-0.25,), redraw=False),
        Workload("stack24-d1024-quarter", 1, "step", shapes=transformer_stack(), dtype=BF16,
                 alpha=-0.7, steps=10, powers=(-0.25,)),
        Workload("stack24-d1024-half", 2, "step", shapes=transformer_stack(), dtype=BF16,
                 alpha=-0.7, steps=10, powers=(-0.5,)),
        Workload("spd64-2048", 3, "inv_root", dims=tuple([2048] * 64), dtype=F32,
                 eps=1e-6, powers=(-0.25, -0.5)),
        Workload("wide-6144", 4, "step", shapes=wide, dtype=F32, alpha=-0.5, steps=4,
                 powers=(-0.25,)),
    ]


def workload(index_or_name) -> Workload:
    for w in workloads():
        if w.index == index_or_name or w.name == index_or_name:
            return w
    raise KeyError(index_or_name)


def gradients_for_step(w: Workload, step: int, matrices: Sequence[int] | None = None) -> List[np.ndarray]:
    """Host (numpy) gradients of one step; ``matrices`` selects a subset by index."""
    idx = range(w.count) if matrices is None else matrices
    out = []
    for i in idx:
        m, n = w.shapes[i]
        if w.index == 0:
            rng = np.random.default_rng(0)
        else:
            rng = rng_for(w.index, step if w.redraw else 0, i)
        out.append(gradient(m, n, w.alpha, rng, w.dtype))
    return out


def spd_inputs(w: Workload, matrices: Sequence[int] | None = None) -> List[np.ndarray]:
    idx = range(w.count) if matrices is None else matrices
    return [spd(w.dims[i], rng_for(w.index, 0, i)) for i in idx]


def scaled(w: Workload, shape_div: int) -> Workload:
    """Same recipe with every side divided by ``shape_div`` (small parity cases)."""
    if w.kind == "step":
        shapes = tuple((max(1, m // shape_div), max(1, n // shape_div)) for m, n in w.shapes)
        return dataclasses.replace(w, shapes=shapes)
    return dataclasses.replace(w, dims=tuple(max(1, d // shape_div) for d in w.dims))


# --------------------------------------------------------------------------
# torch backend (device draws, fp32 QR) for the large stacks
# --------------------------------------------------------------------------
def _torch_seed(config: int, step: int, matrix: int) -> int:
    ss = np.random.SeedSequence([config, step, matrix])
    return int(ss.generate_state(1, dtype=np.uint64)[0] & ((1 << 63) - 1))


def torch_haar(n: int, k: int, gen, device):
    import torch
    z = torch.randn((n, k), generator=gen, device=device, dtype=torch.float32)
    q, r = torch.linalg.qr(z)
    sgn = torch.sign(torch.diagonal(r))
    sgn[sgn == 0] = 1.0
    return q * sgn[None, :]


def torch_gradient(m: int, n: int, alpha: float, seed: int, dtype: str, device):
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    r = min(m, n)
    u = torch_haar(m, r, gen, device)
    v = torch_haar(n, r, gen, device)
    s = torch.arange(1, r + 1, device=device, dtype=torch.float32) ** alpha
    g = (u * s[None, :]) @ v.T
    return g.to(torch.bfloat16) if dtype == BF16 else g.contiguous()


def torch_gradients_for_step(w: Workload, step: int, device, matrices: Sequence[int] | None = None):
    idx = range(w.count) if matrices is None else matrices
    out = []
    for i in idx:
        m, n = w.shapes[i]
        out.append(torch_gradient(m, n, w.alpha, _torch_seed(w.index, step if w.redraw else 0, i),
                                  w.dtype, device))
    return out


def torch_spd(d: int, seed: int, device, log10_lo: float = -8.0, log10_hi: float = 0.0):
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q = torch_haar(d, d, gen, device)
    u = torch.rand((d,), generator=gen, device=device, dtype=torch.float64)
    lam = (10.0 ** (log10_lo + (log10_hi - log10_lo) * u)).to(torch.float32)
    a = (q * lam[None, :]) @ q.T
    return (0.5 * (a + a.T)).contiguous()


def torch_spd_inputs(w: Workload, device, matrices: Sequence[int] | None = None):
    idx = range(w.count) if matrices is None else matrices
    return [torch_spd(w.dims[i], _torch_seed(w.index, 0, i), device) for i in idx]
