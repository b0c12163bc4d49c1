"""The separate dQ pass (dq_mode "separate"): parity against the fp64 oracle and against the accumulating path (GPU).

The pass recomputes S and dP query-major and keeps dQ in tensor memory, while the key-major main
kernel then computes dK and dV only. Checked here: dQ, dK, dV against the oracle on the full tensors
(both masks, d = 64 and 128, both dtypes, ragged lengths, the x8 stress input, grouped K/V heads and
key padding), dQ on sampled rows at the benchmark size, dQ bitwise identical from one call to the
next (no reductions in scheduling order), dK and dV bitwise identical to the accumulating path's, the
staged entry points against the one-call backward, and d = 256 refused.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_09_gb300 as fa
from tiled_attention_09_gb300 import _lib
from tiled_attention_09_gb300.inputs import CAUSAL_4K, SMALL, Workload, make_inputs, sample_rows
from helpers import cancel_tol, check_grad, to64

pytestmark = pytest.mark.gpu


def _run(w, dq_mode, Hkv=None, kv_len=None):
    q, k, v, do = make_inputs(w)
    if Hkv is not None:
        k, v = k[:, :Hkv].contiguous(), v[:, :Hkv].contiguous()
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    klc = kv_len.cuda() if kv_len is not None else None
    o, lse, o_lo = fa.fwd(qc, kc, vc, causal=w.causal, residual=True, kv_len=klc)
    grads = fa.bwd(qc, kc, vc, o, lse, doc, causal=w.causal, o_lo=o_lo, kv_len=klc, dq_mode=dq_mode)
    torch.cuda.synchronize()
    code, info = fa.device_status()
    assert code == "FA_OK", info
    return (q, k, v, do), (qc, kc, vc, doc, o, lse, o_lo, klc), grads


CASES = [
    SMALL,
    Workload(1, 2, 256, 64, "fp16", True),
    Workload(1, 3, 384, 128, "bf16", True),
    Workload(1, 3, 384, 128, "bf16", False),
    Workload(2, 2, 640, 128, "fp16", True),
    Workload(1, 2, 300, 128, "bf16", True),
    Workload(1, 2, 1000, 64, "bf16", False),
    Workload(1, 2, 77, 128, "bf16", True),
    Workload(1, 2, 512, 128, "bf16", True, stress=8.0),
    Workload(2, 12, 1024, 128, "bf16", True),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name())
def test_dq_pass_full_oracle(w):
    (q, k, v, do), _, (dq, dk, dv) = _run(w, "separate")
    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    ref = oracle.attention_bwd(q64, k64, v64, do64, w.scale, w.causal)
    floor = cancel_tol(q64, k64, v64, do64, w.scale)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        check_grad(to64(g), r, f"{name} {w.name()}", floor[name])


@pytest.mark.parametrize("w,Hkv,lens", [
    (Workload(2, 4, 300, 128, "bf16", True), 2, (300, 170)),
    (Workload(2, 6, 256, 64, "fp16", False), 1, (256, 1)),
    (Workload(3, 2, 200, 128, "bf16", True), 2, (0, 129, 200)),
], ids=["gqa_padded", "mqa_padded", "empty_batch"])
def test_dq_pass_grouped_heads_and_key_padding(w, Hkv, lens):
    kv_len = torch.tensor(lens, dtype=torch.int32)
    (q, k, v, do), _, (dq, dk, dv) = _run(w, "separate", Hkv=Hkv, kv_len=kv_len)
    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    ref = oracle.attention_bwd(q64, k64, v64, do64, w.scale, w.causal, kv_len=kv_len.numpy())
    floor = cancel_tol(q64, k64, v64, do64, w.scale)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        if np.abs(r).max() == 0:
            assert (g == 0).all(), f"{name} must be exactly zero"
        else:
            check_grad(to64(g), r, name, floor[name])
    empty = [b for b, n in enumerate(lens) if n == 0]
    for b in empty:  # a batch whose queries see no key: all its gradients are exactly zero
        assert (dq[b] == 0).all() and (dk[b] == 0).all() and (dv[b] == 0).all()


def test_dq_pass_sampled_rows_at_the_benchmark_size():
    w = CAUSAL_4K
    (q, k, v, do), _, (dq, dk, dv) = _run(w, "separate")
    rows = sample_rows(w.N)
    _, _, dq_ref = oracle.attention_rows(to64(q), to64(k), to64(v), to64(do), w.scale, w.causal, rows)
    check_grad(to64(dq[:, :, rows]), dq_ref, "dQ rows")


@pytest.mark.parametrize("w", [Workload(1, 3, 384, 128, "bf16", True), Workload(2, 2, 640, 64, "fp16", False)],
                         ids=lambda w: w.name())
def test_dq_pass_is_deterministic_and_dk_dv_match_the_accumulating_path(w):
    _, (qc, kc, vc, doc, o, lse, o_lo, _), (dq1, dk1, dv1) = _run(w, "separate")
    dq2, dk2, dv2 = fa.bwd(qc, kc, vc, o, lse, doc, causal=w.causal, o_lo=o_lo, dq_mode="separate")
    dqa, dka, dva = fa.bwd(qc, kc, vc, o, lse, doc, causal=w.causal, o_lo=o_lo, dq_mode="accumulate")
    torch.cuda.synchronize()
    assert torch.equal(dq1, dq2) and torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert torch.equal(dk1, dka) and torch.equal(dv1, dva)
    check_grad(to64(dq1), to64(dqa), "dQ separate vs accumulate")


def test_staged_entry_points_match_the_one_call_backward():
    """fa_bwd_preprocess_opt, fa_bwd_main_opt (dq NULL) and fa_bwd_dq_pass, in that order, equal fa_bwd_opt."""
    w = Workload(1, 3, 384, 128, "bf16", True)
    _, (qc, kc, vc, doc, o, lse, o_lo, _), (dq, dk, dv) = _run(w, "separate")
    L = _lib.load()
    B, H, N, d = qc.shape
    ws_bytes = int(L.fa_bwd_workspace_size(B, H, N, d))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    dq2, dk2, dv2 = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
    opt = _lib.FAOptions(0, None, 0, 2)
    V = ctypes.c_void_p
    st = V(torch.cuda.current_stream().cuda_stream)
    assert L.fa_bwd_preprocess_opt(o.data_ptr(), o_lo.data_ptr(), doc.data_ptr(), lse.data_ptr(), ws.data_ptr(),
                                   ws_bytes, B, H, N, d, 1, _lib.FA_BF16, ctypes.byref(opt), st) == 0
    assert L.fa_bwd_main_opt(qc.data_ptr(), kc.data_ptr(), vc.data_ptr(), doc.data_ptr(), dk2.data_ptr(),
                             dv2.data_ptr(), None, ws.data_ptr(), ws_bytes, B, H, N, d, w.scale, 1, _lib.FA_BF16,
                             ctypes.byref(opt), st) == 0
    assert L.fa_bwd_dq_pass(qc.data_ptr(), kc.data_ptr(), vc.data_ptr(), doc.data_ptr(), dq2.data_ptr(),
                            ws.data_ptr(), ws_bytes, B, H, N, d, w.scale, 1, _lib.FA_BF16, ctypes.byref(opt), st) == 0
    torch.cuda.synchronize()
    assert fa.device_status()[0] == "FA_OK"
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)


def test_dq_pass_refuses_d256():
    w = Workload(1, 2, 256, 256, "bf16", True)
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    o, lse = fa.fwd(q, k, v, causal=True)
    with pytest.raises(fa.FAError, match="FA_ERR_UNSUPPORTED"):
        fa.bwd(q, k, v, o, lse, do, causal=True, dq_mode="separate")


@pytest.mark.parametrize("w", [Workload(1, 48, 256, 128, "bf16", True), Workload(2, 16, 384, 64, "fp16", True)],
                         ids=lambda w: w.name())
def test_dq_pass_many_short_items_repeated(w):
    """Items with one or two key tiles back to back (short causal heads): the issuers finish an item long
    before the elementwise warps have stored the previous one's dQ. Repeated calls must all complete
    (no wait running out) and give the same dQ as the first, equal to the accumulating path's within tolerance."""
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    o, lse, o_lo = fa.fwd(q, k, v, causal=True, residual=True)
    dq0, _, _ = fa.bwd(q, k, v, o, lse, do, causal=True, o_lo=o_lo, dq_mode="separate")
    for _ in range(20):
        dq, _, _ = fa.bwd(q, k, v, o, lse, do, causal=True, o_lo=o_lo, dq_mode="separate")
    torch.cuda.synchronize()
    code, info = fa.device_status()
    assert code == "FA_OK", info
    assert torch.equal(dq, dq0)
    dqa, _, _ = fa.bwd(q, k, v, o, lse, do, causal=True, o_lo=o_lo, dq_mode="accumulate")
    torch.cuda.synchronize()
    check_grad(to64(dq0), to64(dqa), "dQ separate vs accumulate")
