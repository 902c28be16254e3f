"""Host-side multi-process plumbing for running the attention path on several GPUs.

Attention is independent across (batch, head), so the path shards with no data-path
exchange: each process owns whole heads and its kernels never wait on another rank. Two
ways to use several GPUs are provided:

* weak scaling (what the benchmark reports): every rank runs the full per-GPU workload on its
  own inputs (seed offset by rank); the job's throughput is the sum over ranks, timed by the
  slowest rank;
* head sharding of one fixed batch (strong scaling): rank r takes a contiguous slice of the
  B*H heads.

The only collectives are a barrier and a max-reduction of the measured times, which work
with the ``gloo`` backend on CPU and ``nccl`` on GPUs.
"""
from __future__ import annotations

import os


def env_rank_world():
    """(rank, world_size, local_rank) from the torchrun environment (defaults 0, 1, 0)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(base_seed: int, rank: int) -> int:
    """Seed of a rank's inputs under weak scaling: distinct per rank, rank 0 keeps the base."""
    return int(base_seed) + 1000 * int(rank)


def partition_heads(bh: int, rank: int, world: int) -> tuple[int, int]:
    """Half-open range [lo, hi) of the B*H heads owned by ``rank``: contiguous, sizes differ
    by at most one, every head owned exactly once."""
    if world < 1 or not (0 <= rank < world) or bh < 0:
        raise ValueError("bad partition arguments")
    base, extra = divmod(bh, world)
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return lo, hi


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of ``value`` over all ranks of the default process group (identity when
    torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier() -> None:
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def weak_scaling_value(flops_per_step_per_rank: float, steps: int, world: int,
                       max_time_s: float) -> float:
    """Whole-job TFLOP/s under weak scaling: all ranks' work over the slowest rank's time."""
    if max_time_s <= 0:
        raise ValueError("time must be positive")
    return world * steps * flops_per_step_per_rank / max_time_s / 1e12
