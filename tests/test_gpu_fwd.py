"""Forward parity of the CUDA path (fa_fwd through the C ABI) against the fp64 oracle (GPU).

Full oracle comparison at sizes the oracle finishes in seconds (several tiles,
ragged tails: N % 256 == 128), closed forms computed without the oracle, and
at the full benchmark sizes sampled rows recomputed by the oracle one by one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_09_gb300 as fa
from tiled_attention_09_gb300.inputs import (CAUSAL_4K, CAUSAL_4K_STRESS, LONG_32K, PAGES_SHAPE, SMALL, Workload,
                                             make_inputs, sample_rows)
from helpers import check_lse, check_o, ideal_kernel_o, to64

pytestmark = pytest.mark.gpu


def run_fwd(q, k, v, causal, scale=None):
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    code, info = fa.device_status()
    assert code == "FA_OK", info
    return o, lse


FULL_CASES = [
    SMALL,
    Workload(1, 2, 256, 64, "fp16", True),
    Workload(1, 3, 384, 128, "bf16", False),
    Workload(1, 3, 384, 128, "bf16", True),
    Workload(2, 2, 640, 128, "fp16", True),
    Workload(1, 2, 512, 256, "bf16", False),
    Workload(1, 2, 384, 256, "bf16", True),
    Workload(1, 2, 512, 64, "bf16", True, stress=8.0),
    PAGES_SHAPE,
    Workload(2, 12, 1024, 128, "bf16", True),
]


@pytest.mark.parametrize("w", FULL_CASES, ids=lambda w: w.name())
def test_fwd_full_oracle(w):
    q, k, v, do = make_inputs(w)
    o, lse = run_fwd(q, k, v, w.causal)
    q64, k64, v64 = to64(q), to64(k), to64(v)
    o_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, w.scale, w.causal)
    pv_abs, _ = oracle.attention_fwd(q64, k64, np.abs(v64), w.scale, w.causal)
    check_o(to64(o), o_ref, pv_abs, w.dtype, f"O fwd {w.name()}",
            ideal=ideal_kernel_o(q64, k64, v64, w.scale, w.dtype, w.causal))
    check_lse(to64(lse), lse_ref)


@pytest.mark.parametrize("w", [CAUSAL_4K, CAUSAL_4K_STRESS, LONG_32K], ids=lambda w: w.name())
def test_fwd_sampled_rows(w):
    q, k, v, do = make_inputs(w)
    o, lse = run_fwd(q, k, v, w.causal)
    rows = sample_rows(w.N)
    o_g, lse_g = to64(o[:, :, rows]), to64(lse[:, :, rows])
    q64, k64, v64 = to64(q), to64(k), to64(v)
    o_ref, lse_ref, _ = oracle.attention_rows(q64, k64, v64, np.zeros_like(q64), w.scale, w.causal, rows)
    pv_abs, _, _ = oracle.attention_rows(q64, k64, np.abs(v64), np.zeros_like(q64), w.scale, w.causal, rows)
    check_o(o_g, o_ref, pv_abs, w.dtype, f"O fwd {w.name()} sampled rows",
            ideal=ideal_kernel_o(q64, k64, v64, w.scale, w.dtype, w.causal, rows=rows))
    check_lse(lse_g, lse_ref)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_fwd_closed_form_q_zero(causal, d):
    """Q = 0: uniform attention over the visible keys; LSE = ln(#visible)."""
    B, H, N = 1, 2, 384
    g = torch.Generator().manual_seed(5)
    v = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16)
    q = torch.zeros_like(k)
    o, lse = run_fwd(q, k, v, causal)
    v64 = to64(v)
    if causal:
        want = np.cumsum(v64, axis=2) / np.arange(1, N + 1)[None, None, :, None]
        want_lse = np.broadcast_to(np.log(np.arange(1, N + 1)), (B, H, N))
    else:
        want = np.broadcast_to(v64.mean(axis=2, keepdims=True), v64.shape)
        want_lse = np.full((B, H, N), math.log(N))
    # P is exactly uniform (exp2(0) = 1), so only output rounding and fp32 sums remain
    check_o(to64(o), want, np.zeros_like(want), "bf16", f"O fwd Q=0 d{d} causal{int(causal)}",
            ideal=ideal_kernel_o(to64(q), to64(k), v64, d ** -0.5, "bf16", causal))
    check_lse(to64(lse), want_lse)


def test_fwd_closed_form_constant_v_and_row0():
    B, H, N, d = 1, 2, 512, 128
    g = torch.Generator().manual_seed(6)
    q = (torch.randn(B, H, N, d, generator=g) * 3).to(torch.bfloat16)
    k = (torch.randn(B, H, N, d, generator=g) * 3).to(torch.bfloat16)
    o, _ = run_fwd(q, k, torch.ones_like(q), True)
    # V = 1: O = 1 up to the P-rounding term u*(P|V|) = 2^-8 and output rounding
    ones = np.ones(o.shape)
    check_o(to64(o), ones, ones, "bf16", "O fwd V=1",
            ideal=ideal_kernel_o(to64(q), to64(k), ones, d ** -0.5, "bf16", True))
    v = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16)
    o, lse = run_fwd(q, k, v, True)
    # causal row 0 sees key 0 only: O_0 = V_0 exactly, LSE_0 = scale q0.k0
    assert torch.equal(o[:, :, 0].cpu(), v[:, :, 0])
    want = (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1) / math.sqrt(d)
    assert (lse[:, :, 0].double().cpu() - want).abs().max().item() < 1e-4


@pytest.mark.parametrize("w", [Workload(1, 2, 512, 128, "bf16", True, stress=8.0), PAGES_SHAPE,
                               Workload(1, 2, 384, 256, "bf16", False)], ids=lambda w: w.name())
def test_fwd_residual_restores_fp32_output(w):
    """o + o_lo carries O to fp32 accuracy: only the P-rounding term of the tolerance remains."""
    q, k, v, _ = make_inputs(w)
    o, lse, o_lo = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, residual=True)
    o2, lse2 = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=w.causal)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    q64, k64, v64 = to64(q), to64(k), to64(v)
    o_ref, _ = oracle.attention_fwd(q64, k64, v64, w.scale, w.causal)
    pv_abs, _ = oracle.attention_fwd(q64, k64, np.abs(v64), w.scale, w.causal)
    from helpers import UNIT_ROUNDOFF
    err = np.abs(to64(o) + to64(o_lo) - o_ref)
    assert (err <= 2e-3 + UNIT_ROUNDOFF[w.dtype] * pv_abs).all(), err.max()
    # the residual is at most half an ulp of the stored value
    assert (np.abs(to64(o_lo)) <= np.abs(to64(o)) * 2.0 ** -8 + 1e-30).all()


def test_fwd_is_deterministic_and_leaves_guard_bytes():
    w = Workload(1, 2, 384, 128, "bf16", True)
    q, k, v, _ = make_inputs(w)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    B, H, N, d = q.shape
    guard = 4096
    o_buf = torch.full((B * H * N * d + 2 * guard,), 7.0, device="cuda", dtype=torch.bfloat16)
    l_buf = torch.full((B * H * N + 2 * guard,), 7.0, device="cuda", dtype=torch.float32)
    o = o_buf[guard:guard + B * H * N * d].view(B, H, N, d)
    lse = l_buf[guard:guard + B * H * N].view(B, H, N)
    fa.fwd(qc, kc, vc, causal=True, out=o, lse=lse)
    o1, l1 = o.clone(), lse.clone()
    fa.fwd(qc, kc, vc, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(o, o1) and torch.equal(lse, l1)
    assert (o_buf[:guard] == 7).all() and (o_buf[-guard:] == 7).all()
    assert (l_buf[:guard] == 7).all() and (l_buf[-guard:] == 7).all()
