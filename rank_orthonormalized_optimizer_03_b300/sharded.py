"""Row-sharded Dion / Orth-Dion step: every rank holds some rows of each matrix.

The Dion abstract (searcharxiv 2504.05295) presents the method as integrating
with weight sharding, and the Orth-Dion abstract (thelatestinai.com
2605.16341) keeps Dion's per-step communication.  Sharding the rows of X, G
and R (V replicated) leaves two quantities that need every row: the Gram
P^T P of each CholeskyQR pass of orth(P), and W = M^T U.  So a step is the
library's five stages (dion_shard_stage) with an all-reduce of a workspace
region after stages 0, 1, 2 (the r x r Grams) and 3 (the n x r W's); see
include/dion.h.  Per matrix and step that is 3 r^2 + n r floats summed over
the ranks.

``sharded_step`` is the orchestration and takes the per-rank work from a
backend object (``stage(k)``, ``exchange(name)``) and the collective from a
callable, so that the same sequence runs with the CUDA kernels on GPU ranks
(``ShardPlan`` + ``torch.distributed.all_reduce``), with R ranks emulated on one
GPU (``EmulatedRanks``), or with any other backend and process group.
"""
from __future__ import annotations

import math
from typing import Callable, Sequence

from . import dion

# after stage k, the region to all-reduce
EXCHANGE_AFTER = {0: "gram", 1: "gram", 2: "gram", 3: "w"}
STAGES = 5
_REGION = {"gram": 0, "w": 1}   # DION_EXCHANGE_GRAM, DION_EXCHANGE_W


def sharded_step(backend, allreduce: Callable) -> None:
    """One optimizer step of a row shard: stage 0..4 of ``backend`` with
    ``allreduce(backend.exchange(name))`` (an in-place sum over all ranks)
    between the stages that need it."""
    for k in range(STAGES):
        backend.stage(k)
        if k in EXCHANGE_AFTER:
            allreduce(backend.exchange(EXCHANGE_AFTER[k]))


def row_bounds(m: int, ranks: int) -> list:
    """Rows [a, b) of each of ``ranks`` shards of an m-row matrix, as even as possible."""
    base, extra = divmod(m, ranks)
    out, a = [], 0
    for k in range(ranks):
        b = a + base + (1 if k < extra else 0)
        out.append((a, b))
        a = b
    return out


class ShardPlan(dion.Plan):
    """A plan over one rank's rows of every matrix (CUDA backend of sharded_step).

    ``mats`` as for :class:`dion.Plan`, with X, G, R holding this rank's rows and V
    the replicated warm start; ``m_total[i]`` is matrix i's full row count, which
    fixes the default scale s = sqrt(m_total / n) (a descriptor's own positive
    ``scale`` wins).  Every shard needs at least r rows.
    """

    def __init__(self, mats: Sequence[dict], m_total: Sequence[int], workspace=None):
        fixed = []
        for d, mt in zip(mats, m_total):
            n = d["X"].shape[1]
            sc = d.get("scale", 0.0)
            fixed.append(dict(d, scale=sc if sc and sc > 0 else math.sqrt(mt / n)))
        super().__init__(fixed, workspace=workspace)

    def stage(self, k: int, stream=None):
        dion.check(dion.lib().dion_shard_stage(self._plan, self.workspace.data_ptr(), self.ws_bytes, k,
                                               dion._stream_ptr(stream)), "dion_shard_stage")

    def exchange(self, name: str):
        """float32 view of exchange region ``name`` ("gram" | "w") in the workspace."""
        import ctypes
        import torch
        off, nbytes = ctypes.c_size_t(), ctypes.c_size_t()
        dion.check(dion.lib().dion_plan_exchange(self._plan, _REGION[name], ctypes.byref(off), ctypes.byref(nbytes)),
                   "dion_plan_exchange")
        return self.workspace[off.value: off.value + nbytes.value].view(torch.float32)


def dist_allreduce(group=None) -> Callable:
    """The collective of a torch.distributed process group (NCCL on GPU ranks)."""
    import torch.distributed as dist
    return lambda t: dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)


class EmulatedRanks:
    """R row shards of the same matrices stepped on one GPU as R ranks.

    Each shard has its own :class:`ShardPlan`; between stages the exchange
    regions of the R plans are summed on the device in rank order and the sum
    is written back to every plan (what an all-reduce over R GPUs would leave
    in each rank's buffer).  No kernel of one rank waits on another: the
    stages of all ranks run one after the other on the current stream.
    """

    def __init__(self, shard_plans: Sequence[ShardPlan]):
        self.plans = list(shard_plans)

    def step(self):
        for k in range(STAGES):
            for p in self.plans:
                p.stage(k)
            if k in EXCHANGE_AFTER:
                views = [p.exchange(EXCHANGE_AFTER[k]) for p in self.plans]
                total = views[0].clone()
                for v in views[1:]:
                    total += v
                for v in views:
                    v.copy_(total)

    def status(self):
        return [p.status() for p in self.plans]
