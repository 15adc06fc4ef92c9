"""Host-side helpers for running RVQ on several GPUs, one process per GPU.

Frames are independent, so encode and decode shard by frame range with no
data-path collective (replicas of the prepared tables on every GPU).  These
helpers cover the host logic around that: the balanced contiguous split of a
frame range, the max-over-ranks of a timing, and an all-gather of
variable-length row blocks for callers that want every rank's results.
They work with any torch.distributed backend (gloo on CPU, nccl on GPUs).
"""

from __future__ import annotations

from typing import Optional, Tuple

import torch
import torch.distributed as dist


def frame_range(n_frames: int, rank: int, world: int) -> Tuple[int, int]:
    """[start, stop) of rank's contiguous share; shares differ by at most one frame."""
    if world < 1 or not 0 <= rank < world or n_frames < 0:
        raise ValueError("bad frame_range arguments")
    base, extra = divmod(n_frames, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def reduce_max(value: float, device: Optional[torch.device] = None) -> float:
    """Maximum of `value` over all ranks (identity without a process group)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def gather_rows(local: torch.Tensor, n_total: int) -> torch.Tensor:
    """Concatenate every rank's row block (in rank order) on every rank.

    local holds this rank's rows of frame_range(n_total, rank, world); blocks
    may differ in length by one row, so they are padded to a common length
    for the collective and trimmed afterwards.
    """
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return local
    world, rank = dist.get_world_size(), dist.get_rank()
    start, stop = frame_range(n_total, rank, world)
    if local.shape[0] != stop - start:
        raise ValueError("local block does not match this rank's frame range")
    longest = max(b - a for a, b in (frame_range(n_total, r, world) for r in range(world)))
    padded = torch.zeros((longest,) + tuple(local.shape[1:]), dtype=local.dtype, device=local.device)
    padded[: local.shape[0]] = local
    parts = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(parts, padded)
    blocks = []
    for r in range(world):
        a, b = frame_range(n_total, r, world)
        blocks.append(parts[r][: b - a])
    return torch.cat(blocks, dim=0)
