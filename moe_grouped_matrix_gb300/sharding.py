"""Host-side helpers for running the grouped matmul on several GPUs.

Expert parallelism (page "tpu-inference 0.12.0.dev20251213 -> 0.13.2.dev20251230",
gmm.py: group_offset selects the slice of experts a shard holds, and rows of the
other experts come out zero, _zero_uninitialized_memory): rank p holds a
contiguous run of experts and calls gmm with group_offset set to the first of
them, so that the full result is the sum of the ranks' outputs.  No collective
is needed on the data path; the combine is the MoE layer's business.

The benchmark runs one independent replica of the workload per rank (weak
scaling) and reports the slowest rank's time.
"""

from __future__ import annotations


def expert_shard(num_groups: int, rank: int, world: int) -> tuple[int, int]:
    """(group_offset, num_local_groups) of `rank`: contiguous, sizes differing by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    if num_groups < world:
        raise ValueError("fewer experts than ranks")
    base, extra = divmod(num_groups, world)
    first = rank * base + min(rank, extra)
    return first, base + (1 if rank < extra else 0)


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks of the default process group (the value itself when
    torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
