"""Assignment of a bucket's matrices to the ranks of a data-parallel job.

The matrices of a bucket are independent problems (Dion3 §7 assigns whole
matrices to devices), so a job of W ranks splits each bucket into W
contiguous chunks: rank r orthogonalizes matrices [start, start + count) of
the bucket, as one batched call (a megabatch), and no matrix is split. The
chunks differ in size by at most one matrix; the first G mod W ranks take
the larger ones. Results do not depend on the split: a matrix gives the same
bits alone or inside any bucket.
"""
from __future__ import annotations


def partition(G: int, world: int, rank: int) -> tuple[int, int]:
    """(start, count) of rank `rank`'s contiguous chunk of a bucket of G
    matrices over `world` ranks."""
    if world < 1 or not 0 <= rank < world or G < 0:
        raise ValueError("need world >= 1, 0 <= rank < world and G >= 0")
    base, extra = divmod(G, world)
    start = rank * base + min(rank, extra)
    return start, base + (1 if rank < extra else 0)
