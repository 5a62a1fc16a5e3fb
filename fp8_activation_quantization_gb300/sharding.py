"""Row sharding of a batch across GPUs.

Every row of the per-token casts is independent, and every 128-row block of the
transposed cast is independent, so a batch splits across ranks by contiguous row
ranges with no exchange: rank r quantizes rows [begin, end) and writes
out[begin:end], sf[begin:end] and, for the transposed cast, the token columns
[begin, end) of out_t and [begin/128, end/128) of sf_t.
"""
from __future__ import annotations


def shard_rows(T: int, world_size: int, rank: int, align: int = 1) -> tuple[int, int]:
    """Contiguous, balanced row range of `rank`; boundaries are multiples of
    `align` (use 128 for the transposed cast).  T must be a multiple of align."""
    if world_size <= 0 or not 0 <= rank < world_size:
        raise ValueError("bad world_size / rank")
    if align <= 0 or T < 0 or T % align:
        raise ValueError("T must be a non-negative multiple of align")
    units = T // align
    base, extra = divmod(units, world_size)
    begin = rank * base + min(rank, extra)
    end = begin + base + (1 if rank < extra else 0)
    return begin * align, end * align
