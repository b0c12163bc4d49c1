"""The Python binding's checks on caller-supplied buffers (GPU tensors, no kernel launched for a bad call).

The C ABI receives plain pointers, so an output, workspace or auxiliary tensor of the wrong shape, dtype or
layout would be read or written past its end. The binding checks every such tensor before the call and raises
ValueError; a correct call right after each rejection still succeeds.
"""
import pytest
import torch

import tiled_attention_09_gb300 as fa

pytestmark = pytest.mark.gpu

B, H, N, D = 2, 2, 128, 64


def _qkv(dtype=torch.bfloat16):
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    return tuple(torch.randn(B, H, N, D, device="cuda", dtype=dtype, generator=g) for _ in range(4))


@pytest.mark.parametrize("kw", [
    dict(out=torch.Size([B, H, N - 1, D])),
    dict(out=torch.float16),
    dict(lse=torch.Size([B, H, N + 1])),
    dict(lse=torch.bfloat16),
    dict(o_lo=torch.Size([B, H, N, D // 2])),
    dict(kv_len=torch.Size([B + 1])),
    dict(kv_len=torch.int64),
], ids=lambda kw: "-".join(f"{k}_{v}" for k, v in kw.items()))
def test_fwd_rejects_wrong_buffers(kw):
    q, k, v, _ = _qkv()
    (name, spec), = kw.items()
    shapes = {"out": (q.shape, q.dtype), "lse": ((B, H, N), torch.float32), "o_lo": (q.shape, q.dtype),
              "kv_len": ((B,), torch.int32)}
    shape, dtype = shapes[name]
    if isinstance(spec, torch.Size):
        shape = spec
    else:
        dtype = spec
    bad = torch.zeros(shape, device="cuda", dtype=dtype)
    with pytest.raises(ValueError, match=name):
        fa.fwd(q, k, v, causal=True, residual=True, **{name: bad})
    o, lse, o_lo = fa.fwd(q, k, v, causal=True, residual=True)
    torch.cuda.synchronize()
    assert fa.device_status()[0] == "FA_OK"


def test_bwd_rejects_wrong_buffers():
    q, k, v, do = _qkv()
    o, lse, o_lo = fa.fwd(q, k, v, causal=True, residual=True)
    need = fa.workspace_size(B, H, N, D)
    bad = [
        dict(lse=lse.to(torch.bfloat16)),
        dict(lse=lse[:, :, :-1].contiguous()),
        dict(dq=torch.empty(B, H, N, D // 2, device="cuda", dtype=q.dtype)),
        dict(dk=torch.empty(B, H, N, D, device="cuda", dtype=torch.float32)),
        dict(dv=torch.empty(B, H, N, D, device="cuda", dtype=q.dtype).transpose(2, 3).contiguous().transpose(2, 3)),
        dict(workspace=torch.empty(need - 1, device="cuda", dtype=torch.uint8)),
        dict(kv_len=torch.full((B - 1,), N, device="cuda", dtype=torch.int32)),
    ]
    for kw in bad:
        args = dict(lse=lse)
        args.update(kw)
        with pytest.raises(ValueError):
            fa.bwd(q, k, v, o, args.pop("lse"), do, causal=True, o_lo=o_lo, **args)
    # a workspace of another element type is counted in bytes
    ws = torch.empty((need + 3) // 4, device="cuda", dtype=torch.float32)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=True, o_lo=o_lo, workspace=ws)
    dq2, dk2, dv2 = fa.bwd(q, k, v, o, lse, do, causal=True, o_lo=o_lo)
    torch.cuda.synchronize()
    assert fa.device_status()[0] == "FA_OK"
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    assert (dq.float() - dq2.float()).abs().max().item() <= 1e-2 * dq2.float().abs().max().item()


def test_decode_rejects_wrong_buffers():
    Hkv, ps, max_pages, Mq = 1, 32, 4, 1
    g = torch.Generator(device="cuda")
    g.manual_seed(1)
    q = torch.randn(B, H, Mq, D, device="cuda", dtype=torch.bfloat16, generator=g)
    kp = torch.randn(Hkv, B * max_pages, ps, D, device="cuda", dtype=torch.bfloat16, generator=g)
    vp = torch.randn(Hkv, B * max_pages, ps, D, device="cuda", dtype=torch.bfloat16, generator=g)
    table = torch.arange(B * max_pages, device="cuda", dtype=torch.int32).reshape(B, max_pages)
    ctx = torch.tensor([100, 37], device="cuda", dtype=torch.int32)
    for kw in (dict(out=torch.empty(B, H, Mq + 1, D, device="cuda", dtype=torch.bfloat16)),
               dict(lse=torch.empty(B, H, Mq, device="cuda", dtype=torch.float16)),
               dict(workspace=torch.empty(1, device="cuda", dtype=torch.uint8), n_split=2)):
        with pytest.raises(ValueError):
            fa.decode(q, kp, vp, table, ctx, **kw)
    with pytest.raises(ValueError):
        fa.decode(q, kp, vp[:, :-1].contiguous(), table, ctx)
    o, lse = fa.decode(q, kp, vp, table, ctx)
    torch.cuda.synchronize()
    assert fa.device_status()[0] == "FA_OK"
    assert torch.isfinite(o.float()).all()
