"""Sequence lengths that are not a multiple of the 128-row tile (GPU): forward and backward through the C ABI
against the fp64 oracle, on several heads at once so that a tile running past the end of one sequence
would show up as an error in the next head.

Covered: N = 1 (a single key), lengths inside the first tile, just past a tile edge (129), and ragged
tails of longer sequences; d in {64, 128, 256}; causal and non-causal; both dtypes on a subset. The
forward's TMA loads zero-fill the rows past N, the softmax masks keys past N and only rows < N are
stored; the backward masks queries past N and stores only dK / dV rows < N.
"""
import numpy as np
import pytest
import torch

import oracle
import tiled_attention_09_gb300 as fa
from tiled_attention_09_gb300.inputs import Workload, make_inputs
from helpers import cancel_tol, check_grad, check_lse, check_o, ideal_kernel_o, to64

pytestmark = pytest.mark.gpu

CASES = [Workload(2, 2, N, d, "bf16", causal) for d in (64, 128, 256) for N in (1, 7, 100, 129, 383, 1000)
         for causal in (True, False)]
CASES += [Workload(1, 3, 200, 64, "fp16", True), Workload(1, 3, 517, 128, "fp16", False),
          Workload(1, 2, 300, 128, "bf16", True, stress=8.0), Workload(1, 2, 70, 256, "fp16", True)]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name())
def test_ragged_fwd_bwd(w):
    q, k, v, do = make_inputs(w)
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse, o_lo = fa.fwd(qc, kc, vc, causal=w.causal, residual=True)
    dq, dk, dv = fa.bwd(qc, kc, vc, o, lse, doc, causal=w.causal, o_lo=o_lo)
    torch.cuda.synchronize()
    code, info = fa.device_status()
    assert code == "FA_OK", info
    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    o_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, w.scale, w.causal)
    pv_abs, _ = oracle.attention_fwd(q64, k64, np.abs(v64), w.scale, w.causal)
    check_o(to64(o), o_ref, pv_abs, w.dtype, f"O fwd {w.name()}",
            ideal=ideal_kernel_o(q64, k64, v64, w.scale, w.dtype, w.causal))
    check_lse(to64(lse), lse_ref)
    ref = oracle.attention_bwd(q64, k64, v64, do64, w.scale, w.causal)
    floor = cancel_tol(q64, k64, v64, do64, w.scale)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        check_grad(to64(g), r, name, floor[name])
