"""The sweep workload: B=2, H=12, d in {64, 128, 256}, N in {512, ..., 16384}, bf16 and fp16, causal and
non-causal; the forward (with the O residual) and the backward at every point through the C ABI (GPU).

Points with N <= 2048 are compared with the full oracle: every element of O, LSE, dQ, dK and dV of all
24 heads. Longer points are checked against the oracle on sampled query rows of two heads (O, LSE, dQ),
on sampled key columns of one head (dK, dV) and, on all 24 heads, against the gradient-sum invariants
sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i. The four (dtype, mask) variants of a (d, N) point share
one seeded fp32 draw, cast to each dtype.
"""
import numpy as np
import pytest
import torch

import oracle
import tiled_attention_09_gb300 as fa
from tiled_attention_09_gb300.inputs import Workload, cast_inputs, make_inputs_fp32, sample_cols, sample_rows
from helpers import check_grad, check_lse, check_o, ideal_kernel_o, to64

pytestmark = pytest.mark.gpu

ROW_HEADS = [(0, 0), (1, 11)]
COL_HEAD = (1, 5)
FULL_ORACLE_MAX_N = 2048


def _check_point(w, fp32):
    q, k, v, do = cast_inputs(w, fp32)
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse, o_lo = fa.fwd(qc, kc, vc, causal=w.causal, residual=True)
    dq, dk, dv = fa.bwd(qc, kc, vc, o, lse, doc, causal=w.causal, o_lo=o_lo)
    torch.cuda.synchronize()
    code, info = fa.device_status()
    assert code == "FA_OK", info
    if w.N <= FULL_ORACLE_MAX_N:
        q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
        o_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, w.scale, w.causal)
        pv_abs, _ = oracle.attention_fwd(q64, k64, np.abs(v64), w.scale, w.causal)
        check_o(to64(o), o_ref, pv_abs, w.dtype, f"O sweep {w.name()}",
                ideal=ideal_kernel_o(q64, k64, v64, w.scale, w.dtype, w.causal))
        check_lse(to64(lse), lse_ref, f"LSE sweep {w.name()}")
        for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv),
                              oracle.attention_bwd(q64, k64, v64, do64, w.scale, w.causal)):
            check_grad(to64(g), r, f"{name} sweep {w.name()}")
        return
    rows = sample_rows(w.N)
    for b, h in ROW_HEADS:
        q64, k64, v64, do64 = (to64(t[b:b + 1, h:h + 1]) for t in (q, k, v, do))
        o_ref, lse_ref, dq_ref = oracle.attention_rows(q64, k64, v64, do64, w.scale, w.causal, rows)
        pv_abs, _, _ = oracle.attention_rows(q64, k64, np.abs(v64), np.zeros_like(q64), w.scale, w.causal, rows)
        check_o(to64(o[b:b + 1, h:h + 1, rows]), o_ref, pv_abs, w.dtype, f"O sweep {w.name()} head {(b, h)} rows",
                ideal=ideal_kernel_o(q64, k64, v64, w.scale, w.dtype, w.causal, rows=rows))
        check_lse(to64(lse[b:b + 1, h:h + 1, rows]), lse_ref, f"LSE {w.name()} head {(b, h)}")
        check_grad(to64(dq[b:b + 1, h:h + 1, rows]), dq_ref, f"dQ rows {w.name()} head {(b, h)}")
    b, h = COL_HEAD
    cols = sample_cols(w.N)
    q64, k64, v64, do64 = (to64(t[b:b + 1, h:h + 1]) for t in (q, k, v, do))
    dk_ref, dv_ref = oracle.attention_cols(q64, k64, v64, do64, w.scale, w.causal, cols, [(0, 0)], row_block=2048)
    check_grad(to64(dk[b, h, cols])[None], dk_ref, f"dK cols {w.name()}")
    check_grad(to64(dv[b, h, cols])[None], dv_ref, f"dV cols {w.name()}")
    dk_sum = dk.double().sum(dim=2).cpu().numpy()
    dv_sum = dv.double().sum(dim=2).cpu().numpy()
    do_sum = do.double().sum(dim=2).numpy()
    dk_scale = dk.double().abs().amax().item()
    assert np.abs(dk_sum).max() <= 1e-2 * dk_scale * np.sqrt(w.N), (w.name(), np.abs(dk_sum).max())
    assert np.abs(dv_sum - do_sum).max() <= 1e-2 * np.abs(do_sum).max() + 1e-2 * np.sqrt(w.N), w.name()


@pytest.mark.parametrize("N", [512, 1024, 2048, 4096, 8192, 16384])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_sweep_point(d, N):
    fp32 = make_inputs_fp32(Workload(2, 12, N, d, "bf16", True))
    for dtype in ("bf16", "fp16"):
        for causal in (True, False):
            _check_point(Workload(2, 12, N, d, dtype, causal), fp32)
