"""Split-key forward (fa_fwd_split): each query block's key range over several CTAs, joined by the LSE merge (GPU).

Compared with the fp64 oracle element by element (O with the same per-element cap and literal-bound
count as the plain forward, LSE within 2e-3): both masks, d = 64, 128 and 256, bf16 and fp16, ragged
lengths, split counts from 2 up to more ranges than a block has key tiles (empty ranges weigh 0),
grouped K/V heads with key padding (an empty batch included), the fp32 output and the O residual; the
backward run on the split forward's O and LSE; the library's own split choice.
"""
import numpy as np
import pytest
import torch

import oracle
import tiled_attention_09_gb300 as fa
from tiled_attention_09_gb300.inputs import Workload, make_inputs
from helpers import cancel_tol, check_grad, check_lse, check_o, ideal_kernel_o, to64

pytestmark = pytest.mark.gpu


def _check_fwd(w, o, lse, q64, k64, v64, kv_len=None, what=""):
    o_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, w.scale, w.causal, kv_len=kv_len)
    pv_abs, _ = oracle.attention_fwd(q64, k64, np.abs(v64), w.scale, w.causal, kv_len=kv_len)
    if o.dtype == torch.float32:  # unrounded output: the stated bound plus the P-rounding term
        u = 2.0 ** -8 if w.dtype == "bf16" else 2.0 ** -11
        err = np.abs(to64(o) - o_ref)
        assert np.isfinite(to64(o)).all() and (err <= 2e-3 + u * pv_abs).all(), err.max()
    else:
        check_o(to64(o), o_ref, pv_abs, w.dtype, f"O split {w.name()} {what}",
                ideal=ideal_kernel_o(q64, k64, v64, w.scale, w.dtype, w.causal, kv_len=kv_len))
    l_gpu, empty = to64(lse), np.isneginf(lse_ref)
    assert np.isneginf(l_gpu[empty]).all() and (to64(o)[empty] == 0).all()
    if (~empty).any():
        check_lse(l_gpu[~empty], lse_ref[~empty], f"LSE split {w.name()} {what}")
    return o_ref


CASES = [
    (Workload(1, 2, 256, 64, "fp16", False), 2),
    (Workload(1, 3, 384, 128, "bf16", True), 2),
    (Workload(1, 3, 384, 128, "bf16", False), 3),
    (Workload(2, 2, 1000, 128, "bf16", True), 4),
    (Workload(1, 2, 700, 64, "bf16", True), 16),
    (Workload(1, 2, 300, 256, "bf16", True), 2),
    (Workload(1, 2, 512, 256, "fp16", False), 3),
    (Workload(1, 2, 512, 128, "bf16", True, stress=8.0), 2),
    (Workload(2, 12, 1024, 128, "bf16", True), 4),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name()}_s{c[1]}")
def test_split_forward_matches_oracle(case):
    w, splits = case
    q, k, v, do = make_inputs(w)
    qc, kc, vc = (t.cuda() for t in (q, k, v))
    o, lse, o_lo = fa.fwd(qc, kc, vc, causal=w.causal, residual=True, kv_splits=splits)
    torch.cuda.synchronize()
    code, info = fa.device_status()
    assert code == "FA_OK", info
    o_ref = _check_fwd(w, o, lse, to64(q), to64(k), to64(v))
    # o + o_lo carries the merged O at fp32 accuracy: only the P-rounding term remains
    u = 2.0 ** -8 if w.dtype == "bf16" else 2.0 ** -11
    pv_abs, _ = oracle.attention_fwd(to64(q), to64(k), np.abs(to64(v)), w.scale, w.causal)
    err = np.abs(to64(o) + to64(o_lo) - o_ref)
    assert (err <= 2e-3 + u * pv_abs).all(), err.max()


def test_split_forward_grouped_heads_key_padding_and_fp32_output():
    w = Workload(3, 4, 300, 128, "bf16", True)
    q, k, v, _ = make_inputs(w)
    k, v = k[:, :2].contiguous(), v[:, :2].contiguous()
    kv_len = torch.tensor([300, 0, 131], dtype=torch.int32)
    qc, kc, vc, klc = (t.cuda() for t in (q, k, v, kv_len))
    for out_fp32 in (False, True):
        o, lse = fa.fwd(qc, kc, vc, causal=True, kv_len=klc, out_fp32=out_fp32, kv_splits=3)
        torch.cuda.synchronize()
        assert fa.device_status()[0] == "FA_OK"
        _check_fwd(w, o, lse, to64(q), to64(k), to64(v), kv_len=kv_len.numpy(), what=f"fp32={out_fp32}")


@pytest.mark.parametrize("w", [Workload(1, 3, 384, 128, "bf16", True), Workload(1, 2, 640, 64, "fp16", False)],
                         ids=lambda w: w.name())
def test_backward_from_the_split_forward(w):
    q, k, v, do = make_inputs(w)
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse, o_lo = fa.fwd(qc, kc, vc, causal=w.causal, residual=True, kv_splits=2)
    dq, dk, dv = fa.bwd(qc, kc, vc, o, lse, doc, causal=w.causal, o_lo=o_lo)
    torch.cuda.synchronize()
    assert fa.device_status()[0] == "FA_OK"
    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    floor = cancel_tol(q64, k64, v64, do64, w.scale)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), oracle.attention_bwd(q64, k64, v64, do64, w.scale,
                                                                                 w.causal)):
        check_grad(to64(g), r, name, floor[name])


def test_library_split_choice_runs_and_matches():
    """kv_splits = 0: the library's choice (several ranges for this grid of four CTAs with long rows)."""
    from tiled_attention_09_gb300 import _lib
    w = Workload(1, 1, 2048, 128, "bf16", True)
    assert _lib.load().fa_fwd_kv_splits(1, 1, 2048, 128, 1) > 1
    q, k, v, _ = make_inputs(w)
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, kv_splits=0)
    torch.cuda.synchronize()
    assert fa.device_status()[0] == "FA_OK"
    _check_fwd(w, o, lse, to64(q), to64(k), to64(v), what="auto")


def test_attention_autograd_uses_the_library_split():
    """fa.attention picks the library's split count (8 here: one head, four query blocks of 2048 keys at most)
    and its O and gradients match the oracle; with kv_splits=1 the O differs only by rounding."""
    from tiled_attention_09_gb300 import _lib
    w = Workload(1, 1, 2048, 128, "bf16", True)
    assert _lib.load().fa_fwd_kv_splits(1, 1, 2048, 128, 1) == 8
    q, k, v, do = make_inputs(w)
    qa, ka, va = (t.cuda().requires_grad_(True) for t in (q, k, v))
    o = fa.attention(qa, ka, va, causal=True)
    o.backward(do.cuda())
    torch.cuda.synchronize()
    assert fa.device_status()[0] == "FA_OK"
    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    o_ref, _ = oracle.attention_fwd(q64, k64, v64, w.scale, True)
    pv_abs, _ = oracle.attention_fwd(q64, k64, np.abs(v64), w.scale, True)
    check_o(to64(o.detach()), o_ref, pv_abs, w.dtype, "O attention split",
            ideal=ideal_kernel_o(q64, k64, v64, w.scale, w.dtype, True))
    floor = cancel_tol(q64, k64, v64, do64, w.scale)
    for name, g, r in zip(("dQ", "dK", "dV"), (qa.grad, ka.grad, va.grad),
                          oracle.attention_bwd(q64, k64, v64, do64, w.scale, True)):
        check_grad(to64(g), r, name, floor[name])
    o1 = fa.attention(qa.detach(), ka.detach(), va.detach(), causal=True, kv_splits=1)
    assert (o1.float() - o.detach().float()).abs().max().item() <= 2 ** -7 * o1.float().abs().max().item()
