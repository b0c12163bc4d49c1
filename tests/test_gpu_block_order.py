"""The backward main kernels' work order (fa_selftest_block_order runs the device function they call) (GPU).

Checked: every (K/V head, key block) is worked on by exactly one CTA; each head's key blocks launch in
ascending order (block 0, the longest under causal masking, first); the heads come in contiguous groups
of one size (the last may be smaller), each group's blocks all launched before the next group's; there
are never more groups than max(1, heads * nkb / 304) (the tail bound); and a group's shared rows stay
within 64 MB unless a single head's rows exceed it or one head fewer per group would break that bound.
"""
import ctypes

import numpy as np
import pytest
import torch

from tiled_attention_09_gb300 import _lib

pytestmark = pytest.mark.gpu

MB = 1 << 20


def _order(heads, nkb, head_bytes):
    L = _lib.load()
    out = torch.full((heads * nkb,), -1, dtype=torch.int32, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.fa_selftest_block_order(heads, nkb, head_bytes, out.data_ptr(), st) == 0
    torch.cuda.synchronize()
    o = out.cpu().numpy().astype(np.int64)
    return o // nkb, o % nkb


CASES = [(24, 32, 4 * MB), (24, 64, 16 * MB), (24, 128, 33 * MB), (8, 256, 33 * MB), (24, 16, 4 * MB),
         (1, 1, 1), (1, 300, 1 * MB), (7, 3, 100 * MB), (8200, 8, 2 * MB), (5, 1000, 1), (13, 77, 9 * MB)]


@pytest.mark.parametrize("heads,nkb,head_bytes", CASES)
def test_block_order(heads, nkb, head_bytes):
    bh, kb = _order(heads, nkb, head_bytes)
    assert np.array_equal(np.sort(bh * nkb + kb), np.arange(heads * nkb))
    for h in range(min(heads, 64)):
        assert np.all(np.diff(kb[bh == h]) > 0)
    # group size: the heads whose block 0 launches before the first block 1
    hs = heads if nkb == 1 else int(np.argmax(kb == 1))
    assert 1 <= hs <= heads
    n_groups = -(-heads // hs)
    for g in range(n_groups):
        lo, hi = g * hs * nkb, min((g + 1) * hs, heads) * nkb
        assert set(bh[lo:hi].tolist()) == set(range(g * hs, min((g + 1) * hs, heads)))
    tail_bound = max(1, min(heads, heads * nkb // 304))
    assert n_groups <= tail_bound
    if hs * head_bytes > 64 * MB and hs > 1:
        # larger groups only where smaller ones would make more groups than the tail bound allows
        assert -(-heads // (hs - 1)) > tail_bound
