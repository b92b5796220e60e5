"""Column-parallel split of one K-quant product over ranks.

The output rows of y = W x are independent, so rank r can compute rows
[n0, n1) of y from the same Q8_K activations and an all-gather assembles y.
The slabs are made of whole 16-row groups (the row groups of the packed
image), so every rank repacks only its own disk rows and no packed row group
straddles two ranks.  Host logic only: the product on each rank is the
library's ordinary call on its slab.
"""
from __future__ import annotations

GROUP_ROWS = 16


def column_slabs(N: int, world: int, align: int = GROUP_ROWS) -> list[tuple[int, int]]:
    """Row ranges [n0, n1) of the `world` ranks: consecutive, together [0, N),
    each starting on a multiple of `align`; the row groups are dealt out as
    evenly as possible (the first ranks take one more when they do not
    divide).  A rank may get an empty range when N has fewer groups than
    there are ranks."""
    if N < 0 or world < 1 or align < 1:
        raise ValueError("need N >= 0, world >= 1, align >= 1")
    groups = -(-N // align)
    base, extra = divmod(groups, world)
    out, g = [], 0
    for r in range(world):
        take = base + (1 if r < extra else 0)
        n0, n1 = min(N, g * align), min(N, (g + take) * align)
        out.append((n0, n1))
        g += take
    return out


def all_gather_rows(torch, y_slab, slabs, rank: int, group=None):
    """Assemble y [M, N] from every rank's y_slab [M, n1 - n0] (this rank's
    slab is slabs[rank]).  Slabs are padded to the widest one for the
    collective and trimmed after it."""
    import torch.distributed as dist
    M = y_slab.shape[0]
    width = max(n1 - n0 for n0, n1 in slabs)
    n0, n1 = slabs[rank]
    if y_slab.shape[1] != n1 - n0:
        raise ValueError("y_slab does not match this rank's slab")
    pad = torch.zeros((M, width), dtype=y_slab.dtype, device=y_slab.device)
    pad[:, :n1 - n0] = y_slab
    parts = [torch.empty_like(pad) for _ in slabs]
    dist.all_gather(parts, pad, group=group)
    return torch.cat([p[:, :b - a] for p, (a, b) in zip(parts, slabs)], dim=1)
