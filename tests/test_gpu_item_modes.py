"""The forward's two work-item modes give the same bits (GPU).

The library runs the d = 64 / 128 forward with two 128-row query tiles per work item, or with one where
short rows and few heads would otherwise leave SMs idle (fa_fwd_tiles_per_item). Each query tile's
computation is the same in both: the same key tiles in the same order, the same products and the same
softmax steps. So a batched call in one mode and the same heads called one at a time in the other must
agree bit for bit in O, its rounding residual and LSE; the one-tile results are also checked against the
fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import tiled_attention_09_gb300 as fa
from tiled_attention_09_gb300 import _lib
from tiled_attention_09_gb300.inputs import Workload, make_inputs
from helpers import check_lse, check_o, ideal_kernel_o, to64

pytestmark = pytest.mark.gpu

CASES = [Workload(2, 12, 1024, 128, "bf16", False), Workload(2, 12, 2048, 128, "bf16", True),
         Workload(2, 12, 1024, 64, "fp16", False), Workload(2, 12, 1900, 128, "bf16", True)]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name())
def test_one_and_two_tile_items_agree(w):
    L = _lib.load()
    batched = L.fa_fwd_tiles_per_item(w.B, w.H, w.N, w.d, int(w.causal))
    single = L.fa_fwd_tiles_per_item(1, 1, w.N, w.d, int(w.causal))
    assert (batched, single) == (2, 1), "the shapes must run the two modes"
    q, k, v, do = make_inputs(w)
    qc, kc, vc = (t.cuda() for t in (q, k, v))
    o, lse, o_lo = fa.fwd(qc, kc, vc, causal=w.causal, residual=True)
    torch.cuda.synchronize()
    for b in range(w.B):
        for h in (0, w.H // 2, w.H - 1):
            qh, kh, vh = (t[b:b + 1, h:h + 1].contiguous() for t in (qc, kc, vc))
            o1, lse1, lo1 = fa.fwd(qh, kh, vh, causal=w.causal, residual=True)
            torch.cuda.synchronize()
            assert torch.equal(o1[0, 0], o[b, h]) and torch.equal(lo1[0, 0], o_lo[b, h]), (b, h)
            assert torch.equal(lse1[0, 0], lse[b, h]), (b, h)
            if b == 0 and h == 0:
                q64, k64, v64 = to64(qh.cpu()), to64(kh.cpu()), to64(vh.cpu())
                o_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, w.scale, w.causal)
                pv_abs, _ = oracle.attention_fwd(q64, k64, np.abs(v64), w.scale, w.causal)
                check_o(to64(o1), o_ref, pv_abs, w.dtype, f"O one-tile items {w.name()}",
                        ideal=ideal_kernel_o(q64, k64, v64, w.scale, w.dtype, w.causal))
                check_lse(to64(lse1), lse_ref, f"LSE one-tile items {w.name()}")
    code, info = fa.device_status()
    assert code == "FA_OK", info
