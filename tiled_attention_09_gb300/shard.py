"""Head-parallel sharding across GPUs: no data-path collective.

Every (b, h) head of attention is independent in the forward and the backward
(the score matrix, the softmax and all five gradient products stay inside one
head), so a job over B*H heads splits into contiguous head ranges, one per
rank. A contiguous range of the flattened [B*H, N, d] view is a contiguous
slice of memory, so each rank calls the C ABI on its slice as a problem with
B' = 1, H' = count and nothing is copied. Gathering the per-rank outputs, if
the caller wants them in one place, is the caller's business.
"""
from __future__ import annotations


def head_ranges(total_heads: int, world: int):
    """Contiguous, disjoint, balanced (start, count) ranges covering [0, total_heads).

    The first ``total_heads % world`` ranks get one extra head. Ranks beyond the
    head count get empty ranges.
    """
    if total_heads < 0 or world < 1:
        raise ValueError("total_heads >= 0 and world >= 1 required")
    base, extra = divmod(total_heads, world)
    out, start = [], 0
    for r in range(world):
        n = base + (1 if r < extra else 0)
        out.append((start, n))
        start += n
    return out


def head_slice(t, start: int, count: int):
    """View of heads [start, start+count) of a contiguous [B, H, N, ...] tensor as [1, count, N, ...]."""
    B, H = t.shape[0], t.shape[1]
    flat = t.reshape(B * H, *t.shape[2:])
    return flat[start:start + count].unsqueeze(0)


def local_range(t, rank: int, world: int):
    """(start, count) of this rank's heads for tensor ``t`` of shape [B, H, ...]."""
    return head_ranges(t.shape[0] * t.shape[1], world)[rank]
