"""Row (output-channel) partition of a BitLinear across ranks.

The ternary product of one output row depends only on that row's packed
codes, the matrix scale and the activations (BitNet 深度拆解 §3.1: y[m, n] is
a sum over k of the row's ternary weights times x_q[m, k]), so a matrix
splits by output rows with no exchange at all: every rank holds the packed
bytes of its rows (row n is bytes [n K/4, (n+1) K/4) of the packed matrix,
so a range of rows is one contiguous byte range), the activations are
replicated, and each rank computes its slice of y.  The slices are left
where they are, or gathered into [M, N] when a caller needs the whole row.

This module is host logic only: the partition bounds and the reassembly of
the slices.  The per-rank work is an ordinary BitLinear call on the slice.
"""
from __future__ import annotations


def row_bounds(N: int, world: int, rank: int, align: int = 128):
    """Rows [r0, r1) of `rank` among `world` ranks.

    The N rows are split into contiguous ranges that cover [0, N) once, in
    rank order.  Boundaries fall on multiples of `align` rows (whole 128-row
    tensor-core tiles by default) whenever N has at least `world` such
    blocks; ranges then differ by at most one block.  Otherwise rows are
    split one by one (ranges differ by at most one row; a rank may get none
    when N < world).
    """
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if N < 0:
        raise ValueError("N must be >= 0")
    unit = align if align > 0 and N >= align * world else 1
    units = -(-N // unit)
    r0 = min(N, units * rank // world * unit)
    r1 = min(N, units * (rank + 1) // world * unit)
    return r0, r1


def packed_rows(packed, K: int, r0: int, r1: int):
    """The packed codes of rows [r0, r1): a view of `packed` ([N, K/4] or
    flat), no copy."""
    kb = K // 4
    if packed.dim() == 2:
        return packed[r0:r1]
    return packed[r0 * kb:r1 * kb]


def gather_rows(y_local, N: int, world: int, rank: int, group=None, align: int = 128):
    """All ranks' row slices y_local [M, r1 - r0] assembled into [M, N] on
    every rank (torch.distributed all_gather; slices are padded to the
    largest range for the exchange)."""
    import torch
    import torch.distributed as dist

    M = y_local.shape[0]
    bounds = [row_bounds(N, world, r, align) for r in range(world)]
    width = max(b - a for a, b in bounds)
    send = torch.zeros((M, width), dtype=y_local.dtype, device=y_local.device)
    send[:, : y_local.shape[1]] = y_local
    parts = [torch.empty_like(send) for _ in range(world)]
    dist.all_gather(parts, send.contiguous(), group=group)
    return torch.cat([p[:, : b - a] for p, (a, b) in zip(parts, bounds)], dim=1)
