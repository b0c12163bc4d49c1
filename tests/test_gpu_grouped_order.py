"""Grouped-query heads on shapes where the kernels' L2-grouped launch order takes effect (GPU).

B1 H32 with 8 K/V heads, N = 4096, d = 256: the forward's items run in groups of 16 query heads (4 of the 8
K/V heads), so a group boundary falls inside the grid. Checked against the oracle on sampled query rows
of the first and last query heads (O, LSE, dQ) and on sampled key columns of the last K/V head (dK, dV
summed over its four query heads).
"""
import numpy as np
import pytest
import torch

import oracle
import tiled_attention_09_gb300 as fa
from tiled_attention_09_gb300.inputs import Workload, make_inputs, sample_cols, sample_rows
from helpers import check_grad, check_lse, check_o, ideal_kernel_o, to64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [True, False])
def test_grouped_heads_with_grouped_launch_order(causal):
    w = Workload(1, 32, 4096, 256, "bf16", causal)
    Hkv, G = 8, 4
    q, k, v, do = make_inputs(w)
    k, v = k[:, :Hkv].contiguous(), v[:, :Hkv].contiguous()
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse, o_lo = fa.fwd(qc, kc, vc, causal=causal, residual=True)
    dq, dk, dv = fa.bwd(qc, kc, vc, o, lse, doc, causal=causal, o_lo=o_lo)
    torch.cuda.synchronize()
    code, info = fa.device_status()
    assert code == "FA_OK", info
    rows = sample_rows(w.N)
    for h in (0, 31):
        hk = h // G
        q64, do64 = to64(q[:, h:h + 1]), to64(do[:, h:h + 1])
        k64, v64 = to64(k[:, hk:hk + 1]), to64(v[:, hk:hk + 1])
        o_ref, lse_ref, dq_ref = oracle.attention_rows(q64, k64, v64, do64, w.scale, causal, rows)
        pv_abs, _, _ = oracle.attention_rows(q64, k64, np.abs(v64), np.zeros_like(q64), w.scale, causal, rows)
        check_o(to64(o[:, h:h + 1, rows]), o_ref, pv_abs, w.dtype, f"O grouped order head {h}",
                ideal=ideal_kernel_o(q64, k64, v64, w.scale, w.dtype, causal, rows=rows))
        check_lse(to64(lse[:, h:h + 1, rows]), lse_ref, f"LSE grouped order head {h}")
        check_grad(to64(dq[:, h:h + 1, rows]), dq_ref, f"dQ grouped order head {h}")
    cols = sample_cols(w.N)
    hk = Hkv - 1
    k64, v64 = to64(k[:, hk:hk + 1]), to64(v[:, hk:hk + 1])
    dk_ref = np.zeros((1, len(cols), w.d))
    dv_ref = np.zeros((1, len(cols), w.d))
    for h in range(hk * G, (hk + 1) * G):
        a, b = oracle.attention_cols(to64(q[:, h:h + 1]), k64, v64, to64(do[:, h:h + 1]), w.scale, causal, cols,
                                     [(0, 0)], row_block=2048)
        dk_ref += a
        dv_ref += b
    check_grad(to64(dk[0, hk, cols])[None], dk_ref, "dK grouped order")
    check_grad(to64(dv[0, hk, cols])[None], dv_ref, "dV grouped order")
