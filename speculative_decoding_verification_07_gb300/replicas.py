"""Runs over several GPUs: one independent replica per GPU.

Requests are independent (each has its own rows, Philox stream and cache
blocks), so every rank verifies its own batch against its own block pool and no
data crosses ranks.  The only cross-rank steps are bookkeeping: distinct
request ids per rank, so that no two replicas draw the same random numbers, and
the whole-job rate, which divides the units of all ranks by the slowest rank's
time.  Host-side only; tested with the gloo backend on CPU.
"""

from __future__ import annotations

import torch
import torch.distributed as dist

RANK_ID_STRIDE = 1000003  # request ids of rank r start at r * RANK_ID_STRIDE


def rank_request_ids(request_id: torch.Tensor, rank: int) -> torch.Tensor:
    """The request ids rank `rank` uses (keys of its Philox streams)."""
    return request_id + rank * RANK_ID_STRIDE


def whole_job_rate(ms_local: float, units_local: float, device="cpu"):
    """(units of all ranks / max over ranks of the time, max time in ms).

    A no-op reduction when torch.distributed is not initialised (one rank)."""
    ms = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
    units = torch.tensor([float(units_local)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(ms, op=dist.ReduceOp.MAX)
        dist.all_reduce(units, op=dist.ReduceOp.SUM)
    ms_max = float(ms.item())
    return float(units.item()) / (ms_max / 1e3), ms_max
