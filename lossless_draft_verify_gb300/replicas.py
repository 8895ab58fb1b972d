"""Host-side aggregation of the replica runs (one process per GPU, each with
its own sequences; the draft-and-verify step has no exchange between them).

The benchmark's whole-job number is the units every rank processed divided by
the slowest rank's time; these helpers compute it over any
torch.distributed process group (NCCL on GPUs, gloo on CPUs), or locally when
there is none.  They carry no arithmetic of the method itself.
"""
from __future__ import annotations

import torch


def _reduce(x: float, pg, op, device) -> float:
    if pg is None:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=op, group=pg if not isinstance(pg, type(dist)) else None)
    return float(t.item())


def max_over_ranks(x: float, pg=None, device="cpu") -> float:
    import torch.distributed as dist
    return _reduce(x, pg, dist.ReduceOp.MAX if pg is not None else None, device)


def sum_over_ranks(x: float, pg=None, device="cpu") -> float:
    import torch.distributed as dist
    return _reduce(x, pg, dist.ReduceOp.SUM if pg is not None else None, device)


def whole_job_rate(units_local: float, ms_local: float, pg=None, device="cpu") -> tuple[float, float]:
    """(units of all ranks per second over the slowest rank's time, that time in ms)."""
    ms_max = max_over_ranks(ms_local, pg, device)
    units = sum_over_ranks(units_local, pg, device)
    return units / (ms_max / 1e3), ms_max
