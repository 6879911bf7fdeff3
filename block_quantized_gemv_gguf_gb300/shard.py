"""Row sharding of the projection matmul over G GPUs.

Output rows are independent (Y[n, m] reads only row m of W), so a weight
matrix splits by whole rows: rank g of G owns rows [r0, r1) and computes
Y[:, r0:r1] from the replicated X with the same single-GPU call; the LM head
splits by vocabulary slice the same way.  No collective is needed when the
consumer is row-sharded too; otherwise one all-gather of the Y slices
(N * M * 4 bytes) assembles Y.  Splitting K instead would need a reduction
and is not used.

This module holds only the host-side arithmetic of the split (which rows a
rank owns) and the gather of row slices through torch.distributed; every
matmul still runs in the CUDA library.
"""
from __future__ import annotations


def row_partition(M: int, world: int, rank: int, align: int = 16) -> tuple[int, int]:
    """Rows [r0, r1) of an M-row matrix owned by `rank` of `world`.

    Slices are contiguous, in rank order, cover every row exactly once, and
    start at multiples of `align` rows (the GEMV's 16-row tile) except that
    the last slice ends at M; their sizes differ by at most `align` rows.  A
    rank may own zero rows when M < world * align.
    """
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    if M < 0 or align < 1:
        raise ValueError(f"M={M}, align={align}")
    units = -(-M // align)                     # align-row units, the last one may be short
    u0 = units * rank // world
    u1 = units * (rank + 1) // world
    return min(M, u0 * align), min(M, u1 * align)


def gather_rows(y_local, M: int, world: int, group=None):
    """All-gather row slices y_local [N, r1 - r0] (as split by row_partition)
    into Y [N, M] on every rank.  Uses torch.distributed (NCCL on GPUs, gloo
    on CPU); slices of unequal size are padded to the largest one."""
    import torch
    import torch.distributed as dist
    N = y_local.shape[0]
    bounds = [row_partition(M, world, g) for g in range(world)]
    width = max(r1 - r0 for r0, r1 in bounds)
    pad = torch.zeros(N, width, dtype=y_local.dtype, device=y_local.device)
    pad[:, :y_local.shape[1]] = y_local
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad, group=group)
    return torch.cat([p[:, :r1 - r0] for p, (r0, r1) in zip(parts, bounds)], dim=1)
