"""GB300 (sm_103a) fused attention: Python binding over the libfa.so C ABI.

    O = softmax(scale * Q K^T [+ causal mask]) V

``fwd`` / ``bwd`` call ``fa_fwd`` / ``fa_bwd`` on the current PyTorch CUDA
stream; ``attention`` wraps them in an autograd Function (the call shape of
``flash_attn_func(q, k, v)`` in the AMP example of the page
"transformer模型详解（十）：FlashAttention优化技术"). PyTorch supplies device memory
and streams only: every arithmetic step runs in the library's kernels, and
these functions raise if the library is missing or the tensors are not on a
CUDA device.

Tensors are ``[B, H, N, d]``, contiguous, fp16 or bf16; ``lse`` is fp32
``[B, H, N]``. ``scale`` defaults to ``d ** -0.5``.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from . import _lib
from ._lib import FA_BF16, FA_F16, FAError

__all__ = ["fwd", "bwd", "attention", "workspace_size", "device_status", "FAError", "selftest_gemm", "lib_path"]

_DT = {torch.float16: FA_F16, torch.bfloat16: FA_BF16}

# When set, every call synchronises and reads the device status word afterwards.
CHECK_STATUS = os.environ.get("FA_CHECK_STATUS", "0") == "1"


def lib_path() -> str:
    return _lib.lib_path()


def _stream_ptr(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _check_qkv(*ts: torch.Tensor):
    q = ts[0]
    if q.device.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    if q.dtype not in _DT:
        raise ValueError(f"dtype {q.dtype} unsupported (fp16 / bf16 only)")
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    for t in ts:
        if t.shape != q.shape or t.dtype != q.dtype or t.device != q.device:
            raise ValueError("q, k, v (and o, dO) must share shape, dtype and device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def device_status(stream=None):
    """Synchronise and read/clear the kernels' device status word. Returns (code_name, info)."""
    L = _lib.load()
    info = (ctypes.c_uint * 4)()
    s = ctypes.c_void_p(stream if stream is not None else torch.cuda.current_stream().cuda_stream)
    code = L.fa_device_status(s, info)
    return _lib.STATUS_NAMES.get(code, str(code)), list(info)


def _after(name, t):
    if CHECK_STATUS:
        code, info = device_status(torch.cuda.current_stream(t.device).cuda_stream)
        if code != "FA_OK":
            raise RuntimeError(f"{name}: device status {code} {info}")


def workspace_size(B, H, N, d) -> int:
    return int(_lib.load().fa_bwd_workspace_size(B, H, N, d))


def fwd(q, k, v, causal=False, scale=None, out=None, lse=None, residual=False, o_lo=None):
    """Forward: returns (o, lse), or (o, lse, o_lo) with residual=True (fa_fwd_ex).

    o_lo is the rounding residual of o (O_fp32 - o in the same dtype); pass it
    to ``bwd`` so that D = rowsum(dO * O) uses O at fp32 accuracy.
    """
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    scale = (1.0 / math.sqrt(d)) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32) if lse is None else lse
    if residual and o_lo is None:
        o_lo = torch.empty_like(q)
    L = _lib.load()
    code = L.fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                       o_lo.data_ptr() if residual else None, B, H, N, d, scale, int(bool(causal)), _DT[q.dtype],
                       _stream_ptr(q))
    _lib.check("fa_fwd_ex", code)
    _after("fa_fwd_ex", q)
    return (o, lse, o_lo) if residual else (o, lse)


def bwd(q, k, v, o, lse, do, causal=False, scale=None, workspace=None, dq=None, dk=None, dv=None, o_lo=None):
    """Backward: returns (dq, dk, dv). o_lo: the residual from ``fwd(..., residual=True)``, or None."""
    _check_qkv(q, k, v, o, do)
    if o_lo is not None:
        _check_qkv(q, o_lo)
    B, H, N, d = q.shape
    scale = (1.0 / math.sqrt(d)) if scale is None else float(scale)
    L = _lib.load()
    ws_bytes = int(L.fa_bwd_workspace_size(B, H, N, d))
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    code = L.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                    dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), o_lo.data_ptr() if o_lo is not None else None,
                    workspace.data_ptr(), workspace.numel(), B, H, N, d, scale, int(bool(causal)), _DT[q.dtype],
                    _stream_ptr(q))
    _lib.check("fa_bwd", code)
    _after("fa_bwd", q)
    return dq, dk, dv


class _AttentionFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal, scale):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        o, lse, o_lo = fwd(q, k, v, causal, scale, residual=True)
        ctx.save_for_backward(q, k, v, o, lse, o_lo)
        ctx.causal, ctx.scale = causal, scale
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse, o_lo = ctx.saved_tensors
        dq, dk, dv = bwd(q, k, v, o, lse, do.contiguous(), ctx.causal, ctx.scale, o_lo=o_lo)
        return dq, dk, dv, None, None


def attention(q, k, v, causal=False, scale=None):
    """Differentiable exact attention over [B, H, N, d] fp16/bf16 CUDA tensors."""
    return _AttentionFn.apply(q, k, v, causal, scale)


def selftest_gemm(a, b, n, k, a_mode, b_mode):
    """Tensor-core operand self-test (see include/fa_selftest.h). Returns d [128, n] fp32."""
    L = _lib.load()
    d = torch.empty((128, n), device=a.device, dtype=torch.float32)
    code = L.fa_selftest_gemm(a.data_ptr(), b.data_ptr(), d.data_ptr(), n, k, a_mode, b_mode, _DT[a.dtype],
                              _stream_ptr(a))
    _lib.check("fa_selftest_gemm", code)
    return d
