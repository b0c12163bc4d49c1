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
``[B, H, N]``. ``scale`` defaults to ``d ** -0.5``. Options (``fa_fwd_opt`` /
``fa_bwd_opt``): ``k``/``v`` may have fewer heads than ``q`` (grouped-query or
multi-query attention, ``H % H_kv == 0``); ``kv_len`` (int32 ``[B]`` on the
device) masks keys ``j >= kv_len[b]``; ``out_fp32`` makes O fp32.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from . import _lib
from ._lib import FA_BF16, FA_F16, FAError

__all__ = ["fwd", "bwd", "attention", "decode", "decode_splits", "workspace_size", "device_status", "FAError",
           "selftest_gemm", "lib_path"]

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


def _check_kv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor) -> int:
    """k, v: [B, H_kv, N, d] with H % H_kv == 0, q's dtype and device. Returns H_kv."""
    _check_qkv(q)
    _check_qkv(k, v)
    B, H, N, d = q.shape
    if k.dim() != 4 or k.shape[0] != B or k.shape[2:] != q.shape[2:] or k.dtype != q.dtype or k.device != q.device:
        raise ValueError("k, v must be [B, H_kv, N, d] with q's B, N, d, dtype and device")
    if k.shape[1] < 1 or H % k.shape[1] != 0:
        raise ValueError(f"H = {H} is not a multiple of H_kv = {k.shape[1]}")
    return int(k.shape[1])


def _check_buf(t: torch.Tensor, shape, dtype, device, name: str):
    """A caller-supplied output or input buffer: the kernels get only its pointer, so its shape, dtype,
    device and layout are checked here (a wrong one would be read or written past its end)."""
    if (not isinstance(t, torch.Tensor) or tuple(t.shape) != tuple(shape) or t.dtype != dtype
            or t.device != device or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} on {device}")


def _check_workspace(t: torch.Tensor, need: int, device) -> int:
    """A caller-supplied workspace: contiguous, on the device, at least ``need`` bytes. Returns its bytes."""
    if not isinstance(t, torch.Tensor) or t.device != device or not t.is_contiguous():
        raise ValueError(f"workspace must be a contiguous tensor on {device}")
    nbytes = t.numel() * t.element_size()
    if nbytes < need:
        raise ValueError(f"workspace holds {nbytes} bytes, {need} needed")
    return nbytes


DQ_MODES = {"default": 0, "accumulate": 1, "separate": 2}


def _options(B, H, Hkv, kv_len, out_fp32, device, dq_mode="default"):
    """fa_options for the call, or None when every option has its default."""
    if dq_mode not in DQ_MODES:
        raise ValueError(f"dq_mode must be one of {sorted(DQ_MODES)}")
    if Hkv == H and kv_len is None and not out_fp32 and dq_mode == "default":
        return None
    if kv_len is not None:
        _check_buf(kv_len, (B,), torch.int32, device, "kv_len")
    return _lib.FAOptions(Hkv, kv_len.data_ptr() if kv_len is not None else None, int(bool(out_fp32)),
                          DQ_MODES[dq_mode])


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


def fwd(q, k, v, causal=False, scale=None, out=None, lse=None, residual=False, o_lo=None, kv_len=None,
        out_fp32=False, kv_splits=1, workspace=None):
    """Forward: returns (o, lse), or (o, lse, o_lo) with residual=True (fa_fwd_ex / fa_fwd_opt).

    o_lo is the rounding residual of o (O_fp32 - o in the same dtype); pass it
    to ``bwd`` so that D = rowsum(dO * O) uses O at fp32 accuracy. k, v may have
    fewer heads than q; kv_len masks keys per batch; out_fp32 writes o as fp32
    (no residual then). kv_splits > 1 splits each query block's key range over
    that many CTAs, joined by a merge launch (fa_fwd_split; 0 = the library's
    choice); workspace: optional caller buffer for the partial outputs.
    """
    Hkv = _check_kv(q, k, v)
    B, H, N, d = q.shape
    if out_fp32 and residual:
        raise ValueError("an fp32 output has no rounding residual")
    scale = (1.0 / math.sqrt(d)) if scale is None else float(scale)
    o_dtype = torch.float32 if out_fp32 else q.dtype
    if out is None:
        o = torch.empty(q.shape, device=q.device, dtype=o_dtype)
    else:
        _check_buf(out, q.shape, o_dtype, q.device, "out")
        o = out
    if lse is None:
        lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    else:
        _check_buf(lse, (B, H, N), torch.float32, q.device, "lse")
    if residual:
        if o_lo is None:
            o_lo = torch.empty_like(q)
        else:
            _check_buf(o_lo, q.shape, q.dtype, q.device, "o_lo")
    L = _lib.load()
    opt = _options(B, H, Hkv, kv_len, out_fp32, q.device)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
            o_lo.data_ptr() if residual else None, B, H, N, d, scale, int(bool(causal)), _DT[q.dtype])
    splits = int(kv_splits) if kv_splits else int(L.fa_fwd_kv_splits(B, H, N, d, int(bool(causal))))
    if splits > 1:
        ws_bytes = int(L.fa_fwd_workspace_size(B, H, N, d, splits))
        if workspace is None:
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
        else:
            ws_bytes = _check_workspace(workspace, ws_bytes, q.device)
        opt = opt if opt is not None else _lib.FAOptions(0, None, 0, 0)
        name, code = "fa_fwd_split", L.fa_fwd_split(*args, ctypes.byref(opt), splits, workspace.data_ptr(), ws_bytes,
                                                     _stream_ptr(q))
    elif opt is None:
        name, code = "fa_fwd_ex", L.fa_fwd_ex(*args, _stream_ptr(q))
    else:
        name, code = "fa_fwd_opt", L.fa_fwd_opt(*args, ctypes.byref(opt), _stream_ptr(q))
    _lib.check(name, code)
    _after(name, q)
    return (o, lse, o_lo) if residual else (o, lse)


def bwd(q, k, v, o, lse, do, causal=False, scale=None, workspace=None, dq=None, dk=None, dv=None, o_lo=None,
        kv_len=None, dq_mode="default"):
    """Backward: returns (dq, dk, dv). o_lo: the residual from ``fwd(..., residual=True)``, or None.

    k, v (and dk, dv) may have fewer heads than q; kv_len as given to ``fwd``; o may be fp32.
    dq_mode: "accumulate" (fp32 partial tiles reduced into the workspace), "separate" (a query-major
    pass that keeps dQ in tensor memory; d = 64 and 128) or "default" (the library's choice).
    """
    Hkv = _check_kv(q, k, v)
    _check_qkv(q, do)
    out_fp32 = o.dtype == torch.float32
    if out_fp32:
        if o.shape != q.shape or o.device != q.device or not o.is_contiguous():
            raise ValueError("o must be contiguous [B, H, N, d] on q's device")
    else:
        _check_qkv(q, o)
    if o_lo is not None:
        _check_qkv(q, o_lo)
    B, H, N, d = q.shape
    _check_buf(lse, (B, H, N), torch.float32, q.device, "lse")
    scale = (1.0 / math.sqrt(d)) if scale is None else float(scale)
    L = _lib.load()
    ws_bytes = int(L.fa_bwd_workspace_size(B, H, N, d))
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    else:
        ws_bytes = _check_workspace(workspace, ws_bytes, q.device)
    for name, t, like in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if t is not None:
            _check_buf(t, like.shape, like.dtype, like.device, name)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), o_lo.data_ptr() if o_lo is not None else None,
            workspace.data_ptr(), ws_bytes, B, H, N, d, scale, int(bool(causal)), _DT[q.dtype])
    opt = _options(B, H, Hkv, kv_len, out_fp32, q.device, dq_mode)
    if opt is None:
        name, code = "fa_bwd", L.fa_bwd(*args, _stream_ptr(q))
    else:
        name, code = "fa_bwd_opt", L.fa_bwd_opt(*args, ctypes.byref(opt), _stream_ptr(q))
    _lib.check(name, code)
    _after(name, q)
    return dq, dk, dv


class _AttentionFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal, scale, kv_len, kv_splits):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        o, lse, o_lo = fwd(q, k, v, causal, scale, residual=True, kv_len=kv_len, kv_splits=kv_splits)
        ctx.save_for_backward(q, k, v, o, lse, o_lo)
        ctx.causal, ctx.scale, ctx.kv_len = causal, scale, kv_len
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse, o_lo = ctx.saved_tensors
        dq, dk, dv = bwd(q, k, v, o, lse, do.contiguous(), ctx.causal, ctx.scale, o_lo=o_lo, kv_len=ctx.kv_len)
        return dq, dk, dv, None, None, None, None


def attention(q, k, v, causal=False, scale=None, kv_len=None, kv_splits=0):
    """Differentiable exact attention over [B, H, N, d] fp16/bf16 CUDA tensors.

    k, v may be [B, H_kv, N, d] (grouped-query / multi-query); kv_len: optional int32 [B] key counts.
    kv_splits: key ranges per query block in the forward (0 = the library's choice, which splits only
    grids with few heads and long rows; 1 = never).
    """
    return _AttentionFn.apply(q, k, v, causal, scale, kv_len, kv_splits)


def decode_splits(B, Hkv, d, page_size, max_pages) -> int:
    """Number of key splits fa_decode picks by itself for this shape."""
    return int(_lib.load().fa_decode_splits(B, Hkv, d, page_size, max_pages))


def decode(q, k_pages, v_pages, page_table, ctx_len, causal=False, scale=None, n_split=0, out=None, lse=None,
           workspace=None):
    """Paged decode attention (fa_decode): returns (o [B, H, Mq, d], lse [B, H, Mq]).

    q [B, H, Mq, d]; k_pages, v_pages [Hkv, n_pages, page_size, d] (q's dtype); page_table int32
    [B, max_pages] and ctx_len int32 [B], all on q's device. n_split <= 0: the library's choice.
    """
    _check_qkv(q)
    _check_qkv(k_pages, v_pages)
    B, H, Mq, d = q.shape
    if k_pages.dim() != 4 or v_pages.shape != k_pages.shape:
        raise ValueError("k_pages, v_pages must both be [Hkv, n_pages, page_size, d]")
    Hkv, n_pages, page_size, dk = k_pages.shape
    if dk != d or k_pages.dtype != q.dtype or k_pages.device != q.device:
        raise ValueError("k_pages, v_pages must be [Hkv, n_pages, page_size, d] with q's d, dtype and device")
    for t in (page_table, ctx_len):
        if t.dtype != torch.int32 or t.device != q.device or not t.is_contiguous():
            raise ValueError("page_table and ctx_len must be contiguous int32 tensors on q's device")
    if page_table.dim() != 2 or page_table.shape[0] != B or ctx_len.shape != (B,):
        raise ValueError("page_table must be [B, max_pages] and ctx_len [B]")
    max_pages = page_table.shape[1]
    scale = (1.0 / math.sqrt(d)) if scale is None else float(scale)
    L = _lib.load()
    ws_bytes = int(L.fa_decode_workspace_size(B, H, Hkv, Mq, d, page_size, max_pages, n_split))
    if ws_bytes == 0:
        raise ValueError("unsupported decode shape")
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    else:
        ws_bytes = _check_workspace(workspace, ws_bytes, q.device)
    if out is None:
        o = torch.empty_like(q)
    else:
        _check_buf(out, q.shape, q.dtype, q.device, "out")
        o = out
    if lse is None:
        lse = torch.empty((B, H, Mq), device=q.device, dtype=torch.float32)
    else:
        _check_buf(lse, (B, H, Mq), torch.float32, q.device, "lse")
    code = L.fa_decode(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), page_table.data_ptr(), ctx_len.data_ptr(),
                       o.data_ptr(), lse.data_ptr(), workspace.data_ptr(), ws_bytes, B, H, Hkv, Mq, d,
                       page_size, n_pages, max_pages, n_split, scale, int(bool(causal)), _DT[q.dtype], _stream_ptr(q))
    _lib.check("fa_decode", code)
    _after("fa_decode", q)
    return o, lse


def selftest_gemm(a, b, n, k, a_mode, b_mode):
    """Tensor-core operand self-test (see include/fa_selftest.h). Returns d [128, n] fp32."""
    for name, t, need in (("a", a, 128 * k), ("b", b, n * k)):
        if t.device.type != "cuda" or t.dtype not in _DT or t.dtype != a.dtype or not t.is_contiguous() \
                or t.numel() < need:
            raise ValueError(f"{name} must be a contiguous fp16/bf16 CUDA tensor of at least {need} elements")
    L = _lib.load()
    d = torch.empty((128, n), device=a.device, dtype=torch.float32)
    code = L.fa_selftest_gemm(a.data_ptr(), b.data_ptr(), d.data_ptr(), n, k, a_mode, b_mode, _DT[a.dtype],
                              _stream_ptr(a))
    _lib.check("fa_selftest_gemm", code)
    return d
