"""EMA state kept in host memory and streamed through the device around each step.

"Online KL Shampoo" (Tilde Research), the zero-delay CPU offload section
(before Appendix G): a step's products grow as d^3 while the state it reads and
writes grows as d^2, so above some d the state can live in host memory and move
over the host link while other matrices compute, at no cost in step time.  The
pages derive the break-even d >= 1546 for an H100 (989 TFLOP/s fp16, 60 GEMMs
per step, 3 d^2 fp32 state elements, 64 GB/s PCIe); ``break_even_dim`` is that
model.  On GB300 the host link is NVLink-C2C, an order of magnitude faster than
PCIe, so the break-even d of this library's step is small.

``OffloadedState`` holds the EMA states L and R of a list of matrices in host
memory (pinned for CUDA; full d x d or packed upper triangles, d(d+1)/2 floats,
matching the library's ``PRECOND_OPT_PACKED_STATE``) and runs a step over
groups of matrices g = 0 .. G-1 with two device buffers:

    copy stream:     up(0)  up(1)  [wait step(0)] down(0)  up(2)  [wait step(1)] down(1) ...
    compute stream:  [wait up(0)] step(0)  [wait up(1)] step(1)  ...

Group g + 1 goes into the buffer of group g - 1, whose download precedes that
upload on the copy stream, so no buffer is overwritten while it is in use; the
next call's uploads follow this call's downloads on the same stream.  Without
CUDA (CPU tensors) the same schedule runs as plain copies in that order, which
the CPU tests use.

``library_step`` gives the ``compute`` callable that runs the library's step on
one group; ``OffloadedState.compute`` adapts a state to the ``compute`` callable
of ``OwnerSharding.step``, so that owners keep their matrices' state offloaded.
"""
from __future__ import annotations

import contextlib
from typing import Callable, List, Optional, Sequence, Tuple

import torch

StepFn = Callable[[List[int], List[torch.Tensor], List[torch.Tensor], List[torch.Tensor]], Sequence[torch.Tensor]]


def break_even_dim(rate_flops: float, gemms: float, state_elems_per_d2: float, bytes_per_elem: float,
                   link_bytes_per_s: float) -> float:
    """d above which loading a d x d matrix's state (state_elems_per_d2 d^2 elements) over the link
    takes less time than the step's GEMMs (gemms products of 2 d^3 FLOPs at rate_flops)."""
    return state_elems_per_d2 * bytes_per_elem * rate_flops / (2.0 * gemms * link_bytes_per_s)


def state_numel(d: int, packed: bool) -> int:
    return d * (d + 1) // 2 if packed else d * d


def default_groups(shapes: Sequence[Tuple[int, int]], packed: bool, group_bytes: int) -> List[List[int]]:
    """Consecutive matrices, each group's state (L and R, fp32) at most group_bytes unless a single
    matrix exceeds it."""
    groups: List[List[int]] = []
    cur: List[int] = []
    size = 0
    for i, (m, n) in enumerate(shapes):
        b = 4 * (state_numel(m, packed) + state_numel(n, packed))
        if cur and size + b > group_bytes:
            groups.append(cur)
            cur, size = [], 0
        cur.append(i)
        size += b
    if cur:
        groups.append(cur)
    return groups


class OffloadedState:
    """Host-resident EMA state of a list of matrices, streamed through two device buffers."""

    def __init__(self, shapes: Sequence[Tuple[int, int]], device, packed: bool = False,
                 groups: Optional[Sequence[Sequence[int]]] = None, group_bytes: int = 1 << 30):
        self.shapes = [(int(m), int(n)) for m, n in shapes]
        self.device = torch.device(device)
        self.packed = packed
        self.groups = [list(g) for g in (groups if groups is not None
                                          else default_groups(self.shapes, packed, group_bytes))]
        seen = sorted(i for g in self.groups for i in g)
        if seen != list(range(len(self.shapes))) or any(not g for g in self.groups):
            raise ValueError("groups must be non-empty and cover every matrix exactly once")
        cuda = self.device.type == "cuda"
        pin = cuda and torch.cuda.is_available()

        def host(d: int) -> torch.Tensor:
            t = torch.zeros(state_numel(d, packed), dtype=torch.float32, pin_memory=pin)
            return t if packed else t.view(d, d)

        self.L = [host(m) for m, _ in self.shapes]
        self.R = [host(n) for _, n in self.shapes]
        cap = max(sum(state_numel(self.shapes[i][0], packed) + state_numel(self.shapes[i][1], packed)
                      for i in g) for g in self.groups)
        self._buf = [torch.empty(cap, dtype=torch.float32, device=self.device) for _ in range(2)]
        self._copy = torch.cuda.Stream(device=self.device) if cuda else None

    def _views(self, b: int, g: List[int]) -> Tuple[List[torch.Tensor], List[torch.Tensor]]:
        """Device views of group g's states in buffer b (L then R of each matrix)."""
        Ls, Rs = [], []
        off = 0
        for i in g:
            m, n = self.shapes[i]
            for d, out in ((m, Ls), (n, Rs)):
                k = state_numel(d, self.packed)
                v = self._buf[b][off:off + k]
                out.append(v if self.packed else v.view(d, d))
                off += k
        return Ls, Rs

    def step(self, grads: Sequence[torch.Tensor], step: StepFn) -> List[torch.Tensor]:
        """One step of every matrix: ``step(indices, grads, L, R) -> updates`` runs on each group with
        the group's state on the device (updated in place), while the neighbouring groups' states move.
        Returns the updates in matrix order.  The host state is current once the copy stream has
        drained (``synchronize``)."""
        if len(grads) != len(self.shapes):
            raise ValueError("one gradient per matrix")
        out: List[Optional[torch.Tensor]] = [None] * len(self.shapes)
        cuda = self._copy is not None
        compute = torch.cuda.current_stream(self.device) if cuda else None
        views = [self._views(k % 2, g) for k, g in enumerate(self.groups)]

        def upload(k: int):
            Ls, Rs = views[k]
            for j, i in enumerate(self.groups[k]):
                Ls[j].copy_(self.L[i], non_blocking=cuda)
                Rs[j].copy_(self.R[i], non_blocking=cuda)

        def download(k: int):
            Ls, Rs = views[k]
            for j, i in enumerate(self.groups[k]):
                self.L[i].copy_(Ls[j], non_blocking=cuda)
                self.R[i].copy_(Rs[j], non_blocking=cuda)

        # the same schedule on both: on CUDA the copies run on the copy stream, ordered against the
        # steps by events; on the CPU the calls run in this order, which is the order the events enforce
        up_done = [torch.cuda.Event() if cuda else None for _ in self.groups]
        step_done = [torch.cuda.Event() if cuda else None for _ in self.groups]

        def on_copy():
            return torch.cuda.stream(self._copy) if cuda else contextlib.nullcontext()

        # the uploads need nothing from the compute stream: the previous call's downloads, which
        # waited for its steps, precede them on the copy stream
        with on_copy():
            for k in range(min(2, len(self.groups))):
                upload(k)
                if cuda:
                    up_done[k].record(self._copy)
        for k, g in enumerate(self.groups):
            if cuda:
                compute.wait_event(up_done[k])
            u = list(step(g, [grads[i] for i in g], *views[k]))
            if cuda:
                step_done[k].record(compute)
            for i, x in zip(g, u):
                out[i] = x
            with on_copy():
                if cuda:
                    self._copy.wait_event(step_done[k])
                download(k)
                if k + 2 < len(self.groups):
                    upload(k + 2)               # into group k's buffer, after its download
                    if cuda:
                        up_done[k + 2].record(self._copy)
        return out  # type: ignore[return-value]

    def synchronize(self):
        """Wait until every download has landed in host memory."""
        if self._copy is not None:
            self._copy.synchronize()

    def compute(self, step: StepFn) -> Callable[[List[int], List[torch.Tensor]], List[torch.Tensor]]:
        """A ``compute(indices, grads)`` callable for ``OwnerSharding.step`` over all of this state's
        matrices (the owner's, in the order of ``OwnerSharding.mine``)."""

        def run(idx: List[int], grads: List[torch.Tensor]) -> List[torch.Tensor]:
            if len(idx) != len(self.shapes):
                raise ValueError("the state holds one entry per owned matrix")
            return self.step(grads, step)

        return run


def library_step(handle, beta: float, eps: float, power: float) -> StepFn:
    """``step(indices, grads, L, R)`` through the library's ``precond_step`` on the current stream
    (a handle with ``PRECOND_OPT_PACKED_STATE`` set when the state is packed)."""
    from . import precond_step

    def run(idx: List[int], grads: List[torch.Tensor], L: List[torch.Tensor],
            R: List[torch.Tensor]) -> List[torch.Tensor]:
        g = [x.contiguous() for x in grads]
        out = [torch.empty(x.shape, dtype=torch.float32, device=x.device) for x in g]
        precond_step(handle, g, L, R, beta, eps, power, out=out)
        return out

    return run
