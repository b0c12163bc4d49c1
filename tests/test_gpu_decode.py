"""Paged decode attention (GPU): fa_decode against the fp64 oracle's paged_attention_fwd.

Cases cover grouped-query and multi-query heads (up to 128 query rows per K/V head), one and several
queries per sequence with the causal end alignment, page sizes 16 to 256, sequence lengths that end
inside a page, a sequence shorter than its query count and an empty one, and explicit split counts
(including a single split with long key streams, and more splits than tiles). Rows past each sequence's end inside its
pages hold NaN, as a stale cache may: they must never reach the result.
"""
import numpy as np
import pytest
import torch

import oracle
import tiled_attention_09_gb300 as fa
from tiled_attention_09_gb300.inputs import DecodeWorkload, make_paged_inputs
from helpers import check_lse, check_o, ideal_decode_o, to64

pytestmark = pytest.mark.gpu

CASES = [
    (DecodeWorkload(2, 8, 2, 1, 128, 64, 20, (1000, 77)), 0),
    (DecodeWorkload(2, 8, 2, 1, 128, 64, 20, (1000, 77), dtype="fp16"), 3),
    (DecodeWorkload(3, 4, 4, 4, 64, 16, 40, (640, 5, 0), causal=True), 0),
    (DecodeWorkload(1, 32, 8, 1, 128, 256, 10, (2500,)), 0),
    (DecodeWorkload(1, 32, 8, 1, 128, 256, 10, (2500,)), 1),
    (DecodeWorkload(2, 16, 1, 8, 128, 32, 30, (960, 961), causal=True), 0),
    (DecodeWorkload(2, 2, 2, 2, 64, 128, 3, (1, 384), causal=True), 0),
    (DecodeWorkload(2, 4, 1, 3, 64, 32, 9, (200, 129), dtype="fp16", causal=True), 50),
    (DecodeWorkload(4, 8, 8, 1, 64, 16, 64, (1024, 1, 513, 1023)), 0),
    # long key streams in one split (tens of tiles per stream, each ring reused many times)
    (DecodeWorkload(2, 8, 2, 1, 128, 64, 128, (8192, 8000)), 1),
    (DecodeWorkload(2, 16, 2, 2, 64, 128, 64, (8192, 7777), causal=True), 1),
    # d = 256: 64-key tiles
    (DecodeWorkload(2, 8, 2, 1, 256, 64, 20, (1000, 77)), 0),
    (DecodeWorkload(3, 4, 1, 4, 256, 16, 40, (640, 3, 0), dtype="fp16", causal=True), 0),
    (DecodeWorkload(1, 16, 4, 2, 256, 256, 12, (3000,)), 1),
    (DecodeWorkload(1, 16, 4, 2, 256, 256, 12, (3000,), causal=True), 40),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name()}_split{c[1]}")
def test_decode_matches_oracle(case):
    w, n_split = case
    q, kp, vp, table, ctx = make_paged_inputs(w)
    o, lse = fa.decode(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), ctx.cuda(), causal=w.causal, n_split=n_split)
    torch.cuda.synchronize()
    code, info = fa.device_status()
    assert code == "FA_OK", info
    q64, kp64, vp64 = to64(q), to64(kp), to64(vp)
    o_ref, lse_ref = oracle.paged_attention_fwd(q64, kp64, vp64, table.numpy(), ctx.numpy(), w.scale, w.causal)
    pv_abs, _ = oracle.paged_attention_fwd(q64, kp64, np.abs(vp64), table.numpy(), ctx.numpy(), w.scale, w.causal)
    check_o(to64(o), o_ref, pv_abs, w.dtype, f"O decode {w.name()} split{n_split}",
            ideal=ideal_decode_o(q64, kp64, vp64, table.numpy(), ctx.numpy(), w.scale, w.dtype, w.causal))
    l_gpu, empty = to64(lse), np.isneginf(lse_ref)
    assert np.isneginf(l_gpu[empty]).all() and (to64(o)[empty] == 0).all()
    if (~empty).any():
        check_lse(l_gpu[~empty], lse_ref[~empty])


def test_decode_never_reads_page_table_entries_past_the_sequence():
    """Page-table entries for pages wholly past ctx_len are never read: garbage there changes nothing."""
    w = DecodeWorkload(3, 8, 2, 2, 128, 32, 16, (100, 33, 512), causal=True)
    q, kp, vp, table, ctx = make_paged_inputs(w)
    bad = table.clone()
    for b in range(w.B):
        used = (int(ctx[b]) + w.page_size - 1) // w.page_size
        bad[b, used:] = torch.tensor([-7, 1 << 30, -1] * w.max_pages, dtype=torch.int32)[: w.max_pages - used]
    args = [t.cuda() for t in (q, kp, vp)]
    o1, l1 = fa.decode(*args, table.cuda(), ctx.cuda(), causal=True)
    o2, l2 = fa.decode(*args, bad.cuda(), ctx.cuda(), causal=True)
    torch.cuda.synchronize()
    assert fa.device_status()[0] == "FA_OK"
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_split_count_does_not_change_the_result_much():
    """Any split count gives the same answer up to fp32 summation order."""
    w = DecodeWorkload(2, 8, 2, 2, 128, 64, 16, (1024, 700), causal=True)
    q, kp, vp, table, ctx = (t.cuda() for t in make_paged_inputs(w))
    outs = [fa.decode(q, kp, vp, table, ctx, causal=True, n_split=s) for s in (1, 2, 5, 8)]
    torch.cuda.synchronize()
    for o, lse in outs[1:]:
        assert (o.float() - outs[0][0].float()).abs().max().item() <= 2e-2
        assert (lse - outs[0][1]).abs().max().item() <= 1e-4
