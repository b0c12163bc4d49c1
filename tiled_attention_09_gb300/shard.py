"""Head-parallel sharding across GPUs: no data-path collective.

Every (b, h) head of attention is independent in the forward and the backward
(the score matrix, the softmax and all five gradient products stay inside one
head), so a job over B*H heads splits into contiguous head ranges, one per
rank. A contiguous range of the flattened [B*H, N, d] view is a contiguous
slice of memory, so each rank calls the C ABI on its slice and nothing is
copied. Gathering the per-rank outputs, if the caller wants them in one place,
is the caller's business.

Ranges are cut in whole units of heads that must stay together:
* grouped-query / multi-query attention: the G = H / H_kv query heads that
  read one K/V head form a unit, so that a rank holds whole K/V heads (its K,
  V, dK, dV are a contiguous slice of the [B*H_kv, N, d] view, and dK, dV of a
  K/V head are summed over its whole group inside one rank, with no exchange);
* a key-padding mask (one key count per batch): a unit is a whole batch (all H
  query heads of it), so that a rank's slice is [B', H, N, d] with its own
  B' key counts.
"""
from __future__ import annotations


def head_ranges(total_heads: int, world: int, unit: int = 1):
    """Contiguous, disjoint, balanced (start, count) ranges covering [0, total_heads) in whole units.

    ``unit`` heads form one indivisible unit (it must divide ``total_heads``). The first
    ``(total_heads / unit) % world`` ranks get one extra unit; ranks beyond the unit count get
    empty ranges.
    """
    if total_heads < 0 or world < 1 or unit < 1:
        raise ValueError("total_heads >= 0, world >= 1 and unit >= 1 required")
    if total_heads % unit:
        raise ValueError(f"unit {unit} does not divide {total_heads} heads")
    base, extra = divmod(total_heads // unit, world)
    out, start = [], 0
    for r in range(world):
        n = (base + (1 if r < extra else 0)) * unit
        out.append((start, n))
        start += n
    return out


def head_slice(t, start: int, count: int):
    """View of heads [start, start+count) of a contiguous [B, H, N, ...] tensor as [1, count, N, ...]."""
    B, H = t.shape[0], t.shape[1]
    flat = t.reshape(B * H, *t.shape[2:])
    return flat[start:start + count].unsqueeze(0)


def local_range(t, rank: int, world: int, unit: int = 1):
    """(start, count) of this rank's heads for tensor ``t`` of shape [B, H, ...]."""
    return head_ranges(t.shape[0] * t.shape[1], world, unit)[rank]


def shard_views(q, k, v, rank: int, world: int, kv_len=None, extra=()):
    """This rank's share of one attention job, as views (nothing is copied).

    q: [B, H, N, d]; k, v: [B, H_kv, N, d] with H_kv dividing H; kv_len: None or [B] key counts.
    ``extra`` are further [B, H, ...] tensors sliced like q (dO, O, LSE, ...). Returns a dict with
    q, k, v, kv_len (None or this rank's [B'] counts), extra (a tuple), ``heads`` = (start, count)
    of the rank's query heads in the flattened [B*H] order and ``kv_heads`` likewise for K/V.
    """
    B, H = q.shape[0], q.shape[1]
    Hkv = k.shape[1]
    if H % Hkv:
        raise ValueError(f"{Hkv} K/V heads do not divide {H} query heads")
    G = H // Hkv
    if kv_len is None:
        s, n = head_ranges(B * H, world, G)[rank]
        ks, kn = s // G, n // G
        sl_q = lambda t: head_slice(t, s, n)
        return {"q": sl_q(q), "k": head_slice(k, ks, kn), "v": head_slice(v, ks, kn), "kv_len": None,
                "extra": tuple(sl_q(t) for t in extra), "heads": (s, n), "kv_heads": (ks, kn)}
    s, n = head_ranges(B * H, world, H)[rank]  # whole batches
    b0, nb = s // H, n // H
    sl_b = lambda t: t[b0:b0 + nb]
    return {"q": sl_b(q), "k": sl_b(k), "v": sl_b(v), "kv_len": kv_len[b0:b0 + nb],
            "extra": tuple(sl_b(t) for t in extra), "heads": (s, n), "kv_heads": (b0 * Hkv, nb * Hkv)}
