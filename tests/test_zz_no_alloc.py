"""fa_bwd_noalloc: the backward for callers that must not allocate device memory (GPU).

Some callers cannot call cudaMalloc on the path where they enqueue work: a
plugin hook of an inference runtime or an extension point of a framework whose
contract forbids allocation there, or a process whose device memory belongs to
another allocator. For them the library offers fa_bwd_noalloc, whose scratch
space (D, LSE*log2e, the fp32 dQ accumulator) is a fixed array inside the
library. These tests call it through the C ABI and compare it with fa_bwd,
the entry point that takes a caller-owned workspace, on two calls in a row and
after a call of a different shape (the shared array keeps the last call's
contents, so nothing may depend on them). This file is collected last on
purpose; it also passes when run alone in a fresh process, where the first
call performs the per-device set-up.
"""
import ctypes

import pytest
import torch

import tiled_attention_09_gb300 as fa
from tiled_attention_09_gb300 import _lib
from tiled_attention_09_gb300.inputs import Workload, make_inputs
from helpers import check_grad, to64

pytestmark = pytest.mark.gpu

V = ctypes.c_void_p


def _noalloc(L, q, k, v, o, do, lse, dq, dk, dv, o_lo, w):
    B, H, N, d = q.shape
    stream = V(torch.cuda.current_stream().cuda_stream)
    return L.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), o_lo.data_ptr() if o_lo is not None else None,
                            B, H, N, d, w.scale, int(w.causal), _lib.FA_BF16 if w.dtype == "bf16" else _lib.FA_F16,
                            stream)


def _case(w, residual):
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    if residual:
        o, lse, o_lo = fa.fwd(q, k, v, causal=w.causal, residual=True)
    else:
        (o, lse), o_lo = fa.fwd(q, k, v, causal=w.causal), None
    ref = fa.bwd(q, k, v, o, lse, do, causal=w.causal, o_lo=o_lo)  # caller-owned workspace
    return (q, k, v, o, do, lse, o_lo), ref


def _check_against_reference(L, w, args, ref):
    q, k, v, o, do, lse, o_lo = args
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    assert _noalloc(L, q, k, v, o, do, lse, dq, dk, dv, o_lo, w) == 0
    torch.cuda.synchronize()
    code, info = fa.device_status()
    assert code == "FA_OK", info
    # dK and dV have a fixed summation order: identical to fa_bwd's
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
    # dQ is summed by bulk reductions in scheduling order: same tolerance as the parity tests
    check_grad(to64(dq), to64(ref[0]), "dQ")


def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row():
    L = _lib.load()
    w = Workload(2, 3, 384, 128, "bf16", True)
    args, ref = _case(w, residual=True)
    for _ in range(2):
        _check_against_reference(L, w, args, ref)


def test_noalloc_after_a_call_of_another_shape():
    L = _lib.load()
    w1 = Workload(1, 2, 640, 64, "fp16", False)
    args1, ref1 = _case(w1, residual=False)
    _check_against_reference(L, w1, args1, ref1)
    w2 = Workload(1, 3, 256, 128, "bf16", True, stress=8.0)
    args2, ref2 = _case(w2, residual=True)
    _check_against_reference(L, w2, args2, ref2)


def test_noalloc_rejects_problems_beyond_the_scratch_limit():
    L = _lib.load()
    P = V(1 << 20)  # never dereferenced: the size check comes first
    # B=1, H=8, N=32768, d=128 needs ~136 MB of workspace > 64 MiB
    assert L.fa_bwd_workspace_size(1, 8, 32768, 128) > (64 << 20)
    code = L.fa_bwd_noalloc(P, P, P, P, P, P, P, P, P, None, 1, 8, 32768, 128, 0.088, 1, _lib.FA_BF16, None)
    assert code == 4  # FA_ERR_WORKSPACE
    assert L.fa_bwd_noalloc(P, P, P, P, P, P, P, P, P, None, 1, 1, 256, 96, 0.1, 0, _lib.FA_BF16, None) == 2
