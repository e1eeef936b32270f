"""Owner-sharded preconditioner steps across data-parallel ranks.

Every weight matrix gets one owner rank.  The owner alone keeps the matrix's
EMA state (L, R) and computes its update; the other ranks hold neither, so the
optimizer state is split across ranks instead of replicated.  One step:

1. Gradients to owners.  Each rank holds its local gradient of every matrix.
   The owner of a bucket (its matrices' gradients, flattened, fp32) receives
   their sum over ranks divided by the world size: one ``reduce`` per owner,
   which together form a reduce-scatter with buckets of unequal size.
2. Owners compute.  Each rank runs the preconditioner step on the matrices it
   owns, through a callable (on a GPU, the library's ``precond_step`` with the
   owner's state tensors; see ``library_compute``).
3. Updates to everyone.  Each owner's updates (fp32, flattened) go to every
   rank: one ``broadcast`` per owner, which together form an all-gather.

This is the matrix-sharded layout of "Sharding EMA-Gram eigensolves" (Marin
research note: each device owns whole eigensolves rather than slices of one)
and the owner GPU of "Online KL Shampoo", Appendix G.

Owners are chosen by LPT (longest processing time first; Graham 1969): the
matrices in decreasing order of cost, each to the rank with the least load so
far (ties: the lower index, the lower rank).  Its makespan is at most
(4/3 - 1/(3 W)) times the optimum for W ranks.  The cost of a matrix
G (m x n) is its step's multiply-add count up to a common factor:
``iters x (m^3 + n^3)`` for the two roots' iterations, plus ``m n (m + n)``
for the two Gram products and the two-sided apply.

Only ``reduce`` and ``broadcast`` are used, so the same code runs on the gloo
(CPU) and NCCL backends.  For two ranks the sum of step 1 is exactly the sum
a single process forms, so the result matches a single-rank step bit for bit;
for more ranks the reduction order is the backend's.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import torch
import torch.distributed as dist


def matrix_cost(m: int, n: int, iters: int = 7) -> float:
    """Relative cost of one matrix's step: both roots' iterations plus the Gram and apply products."""
    return float(iters) * (float(m) ** 3 + float(n) ** 3) + float(m) * n * (m + n)


def lpt_owners(costs: Sequence[float], world: int) -> List[int]:
    """Owner rank of every item by LPT; deterministic for equal costs."""
    if world < 1:
        raise ValueError("world must be at least 1")
    load = [0.0] * world
    owners = [0] * len(costs)
    for i in sorted(range(len(costs)), key=lambda j: (-costs[j], j)):
        r = min(range(world), key=lambda k: (load[k], k))
        owners[i] = r
        load[r] += costs[i]
    return owners


def makespan(costs: Sequence[float], owners: Sequence[int], world: int) -> float:
    load = [0.0] * world
    for c, r in zip(costs, owners):
        load[r] += c
    return max(load)


class OwnerSharding:
    """The owner plan for a list of gradient shapes on one process group."""

    def __init__(self, shapes: Sequence[Tuple[int, int]], rank: int, world: int, iters: int = 7,
                 group: Optional[object] = None):
        self.shapes = [(int(m), int(n)) for m, n in shapes]
        self.rank, self.world, self.group = rank, world, group
        self.owners = lpt_owners([matrix_cost(m, n, iters) for m, n in self.shapes], world)
        self.owned = [[i for i, r in enumerate(self.owners) if r == k] for k in range(world)]

    @property
    def mine(self) -> List[int]:
        return self.owned[self.rank]

    def _numel(self, k: int) -> int:
        return sum(self.shapes[i][0] * self.shapes[i][1] for i in self.owned[k])

    def reduce_gradients(self, grads: Sequence[torch.Tensor]) -> List[torch.Tensor]:
        """The world-average of this rank's owned gradients (fp32, in index order of ``mine``)."""
        if len(grads) != len(self.shapes):
            raise ValueError("one gradient per matrix")
        mine = None
        for k in range(self.world):
            if not self.owned[k]:
                continue
            bucket = torch.cat([grads[i].reshape(-1).to(torch.float32) for i in self.owned[k]])
            dist.reduce(bucket, dst=k, op=dist.ReduceOp.SUM, group=self.group)
            if k == self.rank:
                mine = bucket
        out = []
        if mine is not None:
            mine.div_(self.world)
            off = 0
            for i in self.mine:
                m, n = self.shapes[i]
                out.append(mine[off:off + m * n].view(m, n))
                off += m * n
        return out

    def gather_updates(self, mine: Sequence[torch.Tensor], device=None) -> List[torch.Tensor]:
        """Every matrix's update (fp32) on every rank, from each owner's ``mine`` (index order of ``mine``)."""
        if len(mine) != len(self.mine):
            raise ValueError("one update per owned matrix")
        dev = device if device is not None else (mine[0].device if mine else torch.device("cpu"))
        out: List[Optional[torch.Tensor]] = [None] * len(self.shapes)
        for k in range(self.world):
            if not self.owned[k]:
                continue
            if k == self.rank:
                bucket = torch.cat([u.reshape(-1).to(torch.float32) for u in mine]).to(dev)
            else:
                bucket = torch.empty(self._numel(k), dtype=torch.float32, device=dev)
            dist.broadcast(bucket, src=k, group=self.group)
            off = 0
            for i in self.owned[k]:
                m, n = self.shapes[i]
                out[i] = bucket[off:off + m * n].view(m, n)
                off += m * n
        return out  # type: ignore[return-value]

    def step(self, grads: Sequence[torch.Tensor],
             compute: Callable[[List[int], List[torch.Tensor]], Sequence[torch.Tensor]]) -> List[torch.Tensor]:
        """Reduce to owners, ``compute(owned indices, averaged grads) -> updates``, gather to all ranks."""
        g = self.reduce_gradients(grads)
        u = list(compute(self.mine, g)) if self.mine else []
        return self.gather_updates(u, device=grads[0].device)


def library_compute(handle, L: Sequence[torch.Tensor], R: Sequence[torch.Tensor], beta: float, eps: float,
                    power: float, stream=None):
    """A ``compute`` callable for ``OwnerSharding.step`` that runs the library's step on this rank's
    owned matrices.  ``L[j]``, ``R[j]`` are the EMA states of the j-th owned matrix (fp32 CUDA tensors,
    kept by the owner across steps)."""
    from . import precond_step

    def compute(idx: List[int], grads: List[torch.Tensor]) -> List[torch.Tensor]:
        if len(idx) != len(L) or len(idx) != len(R):
            raise ValueError("one L and one R per owned matrix")
        g = [x.contiguous() for x in grads]
        out = [torch.empty_like(x, dtype=torch.float32) for x in g]
        precond_step(handle, g, list(L), list(R), beta, eps, power, out=out, stream=stream)
        return out

    return compute
