"""Host-side logic of multi-GPU runs.

Attention heads are independent in the forward and the backward, so a run on
N GPUs is N independent replicas (one process per GPU, each with its own
seeded inputs) with no data-path collective. The only cross-rank step is on
the host side of the measurement: a barrier around the timed region and the
maximum of the per-rank step times, so that the reported throughput is all
ranks' work divided by the slowest rank's time.
"""

from __future__ import annotations


def replica_seed(base_seed: int, rank: int) -> int:
    """Seed of the inputs of one replica: distinct per rank."""
    return base_seed + rank


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a per-rank scalar over the default process group (the
    value itself when torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(flops_per_step_per_rank: float, world: int, ms_per_step_max: float):
    """Whole-job throughput in TFLOP/s: every rank's FLOPs over the slowest
    rank's step time."""
    if ms_per_step_max <= 0:
        raise ValueError("step time must be positive")
    return world * flops_per_step_per_rank / (ms_per_step_max * 1e-3) / 1e12
