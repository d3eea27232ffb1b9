"""Data-parallel sharding of the vision front end over ranks (host bookkeeping).

"vLLM 多模态推理｜ViT 性能优化" §3.1 (ViT Encoder DP Mode) runs the vision encoder
data-parallel:
- the images of a batch are assigned to ranks by their patch counts (not their number), so
  that every rank gets about the same work;
- each rank embeds only its own images;
- one all-gather collects every rank's rows;
- the rows are put back in the original image order.

Its worked example: patch counts [1000, 100, 200, 50] on 2 ranks give rank 0 image 0
(1000 patches) and rank 1 images 1, 2, 3 (350 patches).

This module holds the two host steps around the per-rank embed call:
- `assign_by_patches`: the balance, greedy with the largest item first onto the least-loaded
  rank (which reproduces the example);
- `gather_in_input_order`: the all-gather and the restore of the input order.

Both are independent of the device, so the gather runs on any torch.distributed backend
(gloo on the CPU in the tests, NCCL between GPUs).
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import torch


def assign_by_patches(patches: Sequence[int], world: int) -> List[List[int]]:
    """Items per rank, balanced by patch count.

    Items go in decreasing patch count (ties: lower index first), each onto the rank with the
    fewest patches so far (ties: lower rank).  Each rank's list is returned in input order,
    which is the order its rows are packed in.
    """
    if world < 1:
        raise ValueError("world must be >= 1")
    if any(int(p) < 0 for p in patches):
        raise ValueError("patch counts must be >= 0")
    load = [0] * world
    out: List[List[int]] = [[] for _ in range(world)]
    for i in sorted(range(len(patches)), key=lambda i: (-int(patches[i]), i)):
        r = min(range(world), key=lambda q: (load[q], q))
        out[r].append(i)
        load[r] += int(patches[i])
    for lst in out:
        lst.sort()
    return out


def rank_rows(patches: Sequence[int], assignment: Sequence[Sequence[int]]) -> List[int]:
    """Rows (patches) each rank produces under ``assignment``."""
    return [sum(int(patches[i]) for i in a) for a in assignment]


def gather_in_input_order(local: torch.Tensor, patches: Sequence[int], assignment: Sequence[Sequence[int]],
                          group: Optional["torch.distributed.ProcessGroup"] = None) -> torch.Tensor:
    """All-gather every rank's rows and return them in the original item order.

    ``local`` holds this rank's rows, [rank_rows[rank], ...], packed in the order of
    ``assignment[rank]``.  Every rank passes the same ``patches`` and ``assignment``.  The
    rows travel as bytes (any dtype), padded to the largest rank's row count, because
    all_gather wants equal sizes.
    """
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    if len(assignment) != world:
        raise ValueError("one item list per rank")
    rows = rank_rows(patches, assignment)
    if local.shape[0] != rows[rank]:
        raise ValueError(f"rank {rank} holds {local.shape[0]} rows, its items have {rows[rank]}")
    tail = tuple(local.shape[1:])
    row_bytes = local[:1].contiguous().view(torch.uint8).numel() if local.shape[0] else \
        torch.empty((1,) + tail, dtype=local.dtype).view(torch.uint8).numel()
    maxr = max(rows) if rows else 0
    send = torch.zeros((maxr, row_bytes), dtype=torch.uint8, device=local.device)
    if rows[rank]:
        send[: rows[rank]] = local.contiguous().view(torch.uint8).reshape(rows[rank], row_bytes)
    recv = [torch.empty_like(send) for _ in range(world)]
    dist.all_gather(recv, send, group=group)
    starts = [0]
    for p in patches:
        starts.append(starts[-1] + int(p))
    out = torch.empty((starts[-1], row_bytes), dtype=torch.uint8, device=local.device)
    for r, items in enumerate(assignment):
        off = 0
        for i in items:
            n = int(patches[i])
            out[starts[i]: starts[i] + n] = recv[r][off: off + n]
            off += n
    return out.view(local.dtype).reshape((starts[-1],) + tail)
