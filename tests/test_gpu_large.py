"""Tensors of more than 2^31 elements (GPU): every global offset in the forward, the backward and
their auxiliary kernels has to be computed in 64 bits.

Each case holds 2.15e9 elements per Q / K / V / dO tensor (4.3 GB in bf16; about 50 GB on the device
for the whole fwd + bwd). The heads compared with the fp64 oracle sit on both sides of element 2^31
and of byte 2^31 (and of element 2^30 of the fp32 dQ accumulator), plus the first and the last head.
Inputs are drawn on the device (a seeded generator there) and the checked heads are copied back, so
the oracle reads exactly what the kernels read.
"""
import gc

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_09_gb300 as fa
from tiled_attention_09_gb300.inputs import Workload, make_inputs_device
from helpers import check_grad, check_lse, check_o, ideal_kernel_o, to64

pytestmark = pytest.mark.gpu


def _boundary_heads(w: Workload, G: int):
    """K/V heads whose query heads start or end next to element 2^31, byte 2^31 and fp32 byte 2^31."""
    per_head = w.N * w.d
    hkv = w.H // G
    picks = {0, hkv - 1}
    for elem in (1 << 31, 1 << 30, 1 << 29):  # element 2^31; byte 2^31 at 2 B; fp32 byte 2^31 at 4 B
        h = elem // per_head  # first query head at or past the boundary
        for qh in (h - 1, h):
            if 0 <= qh < w.H:
                picks.add(qh // G)
    return sorted(picks)


@pytest.mark.parametrize("w,G", [
    (Workload(1, 16400, 1024, 128, "bf16", True), 1),
    (Workload(1, 16400, 1024, 128, "bf16", True), 8),
    (Workload(1, 8200, 1024, 256, "bf16", True), 1),
], ids=["d128_mha", "d128_gqa8", "d256_mha"])
def test_more_than_2_31_elements(w, G):
    assert w.B * w.H * w.N * w.d > (1 << 31)
    dev = torch.device("cuda", 0)
    q, k, v, do = make_inputs_device(w, dev, n_kv_heads=w.H // G)
    o, lse, o_lo = fa.fwd(q, k, v, causal=w.causal, residual=True)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=w.causal, o_lo=o_lo)
    torch.cuda.synchronize()
    code, info = fa.device_status()
    assert code == "FA_OK", info
    for name, t in (("O", o), ("LSE", lse), ("dQ", dq), ("dK", dk), ("dV", dv)):
        assert bool(torch.isfinite(t).all()), f"{name}: non-finite values"
    kv_heads = _boundary_heads(w, G)
    q_heads = [G * j + t for j in kv_heads for t in range(G)]
    qi, ki = torch.tensor(q_heads, device=dev), torch.tensor(kv_heads, device=dev)
    sel_q = lambda t: to64(t.index_select(1, qi))
    sel_kv = lambda t: to64(t.index_select(1, ki))
    q64, k64, v64, do64 = sel_q(q), sel_kv(k), sel_kv(v), sel_q(do)
    o_g, lse_g, dq_g, dk_g, dv_g = sel_q(o), sel_q(lse), sel_q(dq), sel_kv(dk), sel_kv(dv)
    del q, k, v, do, o, lse, o_lo, dq, dk, dv
    gc.collect()
    torch.cuda.empty_cache()
    o_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, w.scale, w.causal)
    pv_abs, _ = oracle.attention_fwd(q64, k64, np.abs(v64), w.scale, w.causal)
    check_o(o_g, o_ref, pv_abs, w.dtype, f"O fwd {w.name()} G{G} boundary heads",
            ideal=ideal_kernel_o(q64, k64, v64, w.scale, w.dtype, w.causal))
    check_lse(lse_g, lse_ref)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq_g, dk_g, dv_g),
                          oracle.attention_bwd(q64, k64, v64, do64, w.scale, w.causal)):
        check_grad(g, r, name)
