"""Options of the C ABI (GPU): grouped-query / multi-query K/V heads, the key-padding mask (kv_len) and the
fp32 output, forward and backward through fa_fwd_opt / fa_bwd_opt, against the fp64 oracle.

Inputs: the seeded Q, K, V, dO of the workload; with H_kv < H, K and V are the first H_kv heads of the drawn
K and V. Keys past kv_len[b] must get exactly zero dK and dV (their probabilities are exactly 0), and a
query that sees no key gets O = 0 and LSE = -inf.
"""
import numpy as np
import pytest
import torch

import oracle
import tiled_attention_09_gb300 as fa
from tiled_attention_09_gb300.inputs import Workload, make_inputs
from helpers import cancel_tol, check_grad, check_lse, check_o, ideal_kernel_o, to64

pytestmark = pytest.mark.gpu

# (workload, H_kv, kv_len or None)
CASES = [
    (Workload(2, 8, 300, 128, "bf16", True), 2, None),
    (Workload(1, 4, 256, 64, "fp16", False), 1, None),
    (Workload(1, 6, 517, 128, "bf16", False), 3, None),
    (Workload(2, 4, 200, 256, "bf16", True), 2, None),
    (Workload(1, 8, 1024, 128, "bf16", True), 1, None),
    (Workload(2, 2, 500, 128, "bf16", False), 2, [500, 137]),
    (Workload(2, 2, 500, 128, "bf16", True), 2, [129, 383]),
    (Workload(3, 2, 256, 64, "fp16", True), 2, [0, 64, 1000]),
    (Workload(3, 2, 256, 64, "bf16", False), 2, [0, 1, 255]),
    (Workload(2, 2, 300, 256, "bf16", False), 1, [300, 45]),
    (Workload(2, 2, 300, 256, "fp16", True), 2, [0, 200]),
    (Workload(2, 4, 700, 128, "bf16", True), 2, [650, 128]),
]


def _name(c):
    w, hkv, kl = c
    return f"{w.name()}_Hkv{hkv}" + ("" if kl is None else "_kv" + "-".join(map(str, kl)))


def _inputs(w, Hkv):
    q, k, v, do = make_inputs(w)
    return q, k[:, :Hkv].contiguous(), v[:, :Hkv].contiguous(), do


def _check_lse_masked(lse_gpu, lse_ref):
    empty = np.isneginf(lse_ref)
    assert np.isneginf(lse_gpu[empty]).all(), "a query with no visible key must get LSE = -inf"
    check_lse(lse_gpu[~empty], lse_ref[~empty])


@pytest.mark.parametrize("case", CASES, ids=_name)
def test_options_fwd_bwd(case):
    w, Hkv, kl = case
    q, k, v, do = _inputs(w, Hkv)
    kv_len = None if kl is None else torch.tensor(kl[:w.B], dtype=torch.int32)
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    klc = None if kv_len is None else kv_len.cuda()
    o, lse, o_lo = fa.fwd(qc, kc, vc, causal=w.causal, residual=True, kv_len=klc)
    dq, dk, dv = fa.bwd(qc, kc, vc, o, lse, doc, causal=w.causal, o_lo=o_lo, kv_len=klc)
    torch.cuda.synchronize()
    code, info = fa.device_status()
    assert code == "FA_OK", info
    assert dk.shape == k.shape and dv.shape == v.shape
    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    kl64 = None if kv_len is None else kv_len.numpy()
    o_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, w.scale, w.causal, kv_len=kl64)
    pv_abs, _ = oracle.attention_fwd(q64, k64, np.abs(v64), w.scale, w.causal, kv_len=kl64)
    check_o(to64(o), o_ref, pv_abs, w.dtype, f"O fwd {_name(case)}",
            ideal=ideal_kernel_o(q64, k64, v64, w.scale, w.dtype, w.causal, kv_len=kl64))
    _check_lse_masked(to64(lse), lse_ref)
    ref = oracle.attention_bwd(q64, k64, v64, do64, w.scale, w.causal, kv_len=kl64)
    floor = cancel_tol(q64, k64, v64, do64, w.scale)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        if np.abs(r).max() == 0:
            assert (g == 0).all(), f"{name} must be exactly zero"
            continue
        check_grad(to64(g), r, name, floor[name])
    if kl is not None:
        for b in range(w.B):
            L = max(0, min(kl[b], w.N))
            assert (dk[b, :, L:] == 0).all() and (dv[b, :, L:] == 0).all(), "padded keys must get zero dK, dV"
            if L == 0:
                assert (o[b] == 0).all() and (dq[b] == 0).all()


@pytest.mark.parametrize("w", [Workload(2, 3, 640, 128, "bf16", True), Workload(1, 2, 333, 64, "fp16", False),
                               Workload(1, 2, 256, 256, "bf16", True)], ids=lambda w: w.name())
def test_fp32_output(w):
    """O written unrounded in fp32: within 2e-3 + u * (P|V|) of the oracle (no output-rounding term), and
    the backward reading that fp32 O matches the oracle's gradients."""
    q, k, v, do = make_inputs(w)
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qc, kc, vc, causal=w.causal, out_fp32=True)
    assert o.dtype == torch.float32
    dq, dk, dv = fa.bwd(qc, kc, vc, o, lse, doc, causal=w.causal)
    torch.cuda.synchronize()
    code, info = fa.device_status()
    assert code == "FA_OK", info
    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    o_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, w.scale, w.causal)
    pv_abs, _ = oracle.attention_fwd(q64, k64, np.abs(v64), w.scale, w.causal)
    from helpers import UNIT_ROUNDOFF
    err = np.abs(to64(o) - o_ref)
    tol = 2e-3 + UNIT_ROUNDOFF[w.dtype] * pv_abs
    assert (err <= tol).all(), f"max err {err.max():.3e}"
    # the 16-bit path's rounded O: the fp32 one is at least as close to the oracle
    o16, _ = fa.fwd(qc, kc, vc, causal=w.causal)
    assert err.max() <= np.abs(to64(o16) - o_ref).max() + 1e-6
    check_lse(to64(lse), lse_ref)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), oracle.attention_bwd(q64, k64, v64, do64, w.scale,
                                                                                  w.causal)):
        check_grad(to64(g), r, name)


def test_autograd_with_grouped_heads_and_padding():
    w = Workload(2, 4, 384, 64, "bf16", True)
    q, k, v, do = _inputs(w, 2)
    kl = torch.tensor([384, 200], dtype=torch.int32)
    qc, kc, vc = (t.cuda().requires_grad_() for t in (q, k, v))
    o = fa.attention(qc, kc, vc, causal=True, kv_len=kl.cuda())
    o.backward(do.cuda())
    torch.cuda.synchronize()
    ref = oracle.attention_bwd(to64(q), to64(k), to64(v), to64(do), w.scale, True, kv_len=kl.numpy())
    for name, g, r in zip(("dQ", "dK", "dV"), (qc.grad, kc.grad, vc.grad), ref):
        check_grad(to64(g), r, name)
