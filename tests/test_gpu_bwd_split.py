"""The backward main kernel's key-block split (GPU).

On shapes with few heads and long rows the library runs each 128-key block's query steps as two halves
on two CTAs (fa_bwd_key_block_parts = 2); each half leaves fp32 partial dK and dV, and the half that
finishes second adds the other's and stores the block. Checked against the fp64 oracle element by
element (both masks, d = 64 and 128, bf16 and fp16, a ragged length, grouped K/V heads with key padding),
bitwise repeatable over calls (the two halves' sum does not depend on which finishes first), dK and dV
identical between the accumulating dQ path and the separate dQ pass (both split), and the same results
from a workspace without the split's room (the no-allocation entry point's fixed array is one) up to
the order of the dK / dV sums.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_09_gb300 as fa
from tiled_attention_09_gb300 import _lib
from tiled_attention_09_gb300.inputs import Workload, make_inputs
from helpers import cancel_tol, check_grad, to64

pytestmark = pytest.mark.gpu

# (workload, H_kv, kv_len or None)
CASES = [
    (Workload(1, 1, 2048, 128, "bf16", True), 1, None),
    (Workload(1, 2, 2048, 128, "bf16", False), 2, None),
    (Workload(1, 1, 2048, 64, "fp16", True), 1, None),
    (Workload(1, 2, 1500, 128, "bf16", True), 2, None),
    (Workload(1, 4, 2048, 64, "bf16", False), 2, [1700]),
]


def _name(c):
    w, hkv, kl = c
    return f"{w.name()}_Hkv{hkv}" + ("" if kl is None else "_kv" + "-".join(map(str, kl)))


@pytest.mark.parametrize("case", CASES, ids=_name)
def test_split_backward_matches_oracle(case):
    w, Hkv, kl = case
    L = _lib.load()
    assert L.fa_bwd_key_block_parts(w.B, w.H, w.N, w.d, int(w.causal)) == 2, "the shape must take the split"
    q, k, v, do = make_inputs(w)
    k, v = k[:, :Hkv].contiguous(), v[:, :Hkv].contiguous()
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    klc = None if kl is None else torch.tensor(kl, dtype=torch.int32, device="cuda")
    o, lse, o_lo = fa.fwd(qc, kc, vc, causal=w.causal, residual=True, kv_len=klc)
    dq, dk, dv = fa.bwd(qc, kc, vc, o, lse, doc, causal=w.causal, o_lo=o_lo, kv_len=klc)
    dq2, dk2, dv2 = fa.bwd(qc, kc, vc, o, lse, doc, causal=w.causal, o_lo=o_lo, kv_len=klc)
    dqs, dks, dvs = fa.bwd(qc, kc, vc, o, lse, doc, causal=w.causal, o_lo=o_lo, kv_len=klc, dq_mode="separate")
    torch.cuda.synchronize()
    code, info = fa.device_status()
    assert code == "FA_OK", info
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2), "split dK / dV must repeat bit for bit"
    assert torch.equal(dk, dks) and torch.equal(dv, dvs), "both dQ paths split the same way"
    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    kl64 = None if kl is None else np.array(kl)
    ref = oracle.attention_bwd(q64, k64, v64, do64, w.scale, w.causal, kv_len=kl64)
    floor = cancel_tol(q64, k64, v64, do64, w.scale)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        check_grad(to64(g), r, f"{name} split {_name(case)}", floor[name])
    if kl is not None:
        Lk = min(kl[0], w.N)
        assert (dk[0, :, Lk:] == 0).all() and (dv[0, :, Lk:] == 0).all()


def test_split_and_unsplit_workspaces_agree():
    """The same shape with the split's room (split) and with only the base workspace (unsplit, as the
    no-allocation entry point runs when the room does not fit): dK, dV within the gradient tolerance of
    each other (their sums run in another order), dQ likewise."""
    w = Workload(1, 2, 2048, 128, "bf16", True)
    L = _lib.load()
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    o, lse, o_lo = fa.fwd(q, k, v, causal=True, residual=True)
    B, H, N, d = q.shape
    full = int(L.fa_bwd_workspace_size(B, H, N, d))
    rows = B * H * ((N + 127) // 128 * 128)
    r256 = lambda x: (x + 255) // 256 * 256
    base = 2 * r256(rows * 4) + r256(rows * d * 4)
    assert full > base, "the shape must have the split's room"
    outs = []
    for nbytes in (full, base):
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        P = lambda t: t.data_ptr()
        assert L.fa_bwd(P(q), P(k), P(v), P(o), P(do), P(lse), P(dq), P(dk), P(dv), P(o_lo), P(ws), nbytes, B, H, N,
                        d, w.scale, 1, _lib.FA_BF16, st) == 0
        torch.cuda.synchronize()
        outs.append((dq, dk, dv))
    code, info = fa.device_status()
    assert code == "FA_OK", info
    for name, a, b in zip(("dQ", "dK", "dV"), outs[0], outs[1]):
        check_grad(to64(a), to64(b), f"{name} split vs unsplit")
