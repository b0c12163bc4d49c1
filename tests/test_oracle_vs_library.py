"""The oracle against an independent library implementation of the same definition (CPU).

``torch.nn.functional.scaled_dot_product_attention`` on the CPU in float64, with gradients from torch's
autograd, computes softmax(scale * Q K^T + mask) V by its own code. The oracle computes the definition
with numpy products and its own softmax. Their agreement to fp64 rounding, at sizes beyond the
finite-difference tests (N <= 16), pins the oracle's forward and backward together:
- both masks, a ragged length and two head dimensions;
- grouped K/V heads, whose gradients are summed by autograd over the repeated heads;
- the key-padding mask;
- paged decode, with the new queries at the end of each sequence.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

RTOL = 1e-11


def _draw(seed, *shapes):
    rng = np.random.Generator(np.random.PCG64(seed))
    return [rng.standard_normal(s) for s in shapes]


def _library(q, k, v, do, scale, mask=None, causal=False):
    """O and (dQ, dK, dV) from torch's attention in float64; k, v repeated to q's heads if grouped."""
    G = q.shape[1] // k.shape[1]
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    kk = tk.repeat_interleave(G, dim=1) if G > 1 else tk
    vv = tv.repeat_interleave(G, dim=1) if G > 1 else tv
    o = F.scaled_dot_product_attention(tq, kk, vv, attn_mask=mask, is_causal=causal and mask is None, scale=scale)
    o.backward(torch.tensor(do, dtype=torch.float64))
    return o.detach().numpy(), (tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy())


def _close(a, b, what):
    err = np.abs(a - b).max()
    assert err <= RTOL * max(1.0, np.abs(b).max()), f"{what}: {err:.3e}"


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(77, 32), (130, 64)])
def test_matches_library_attention(causal, N, d):
    B, H, scale = 2, 3, 0.37
    q, k, v, do = _draw(N + d, *[(B, H, N, d)] * 4)
    o_lib, g_lib = _library(q, k, v, do, scale, causal=causal)
    o, _ = oracle.attention_fwd(q, k, v, scale, causal)
    _close(o, o_lib, "O")
    for name, g, r in zip(("dQ", "dK", "dV"), oracle.attention_bwd(q, k, v, do, scale, causal), g_lib):
        _close(g, r, name)


@pytest.mark.parametrize("Hkv", [1, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_grouped_heads_match_library(Hkv, causal):
    B, H, N, d, scale = 2, 6, 50, 16, 0.25
    q, do = _draw(3, (B, H, N, d), (B, H, N, d))
    k, v = _draw(4, (B, Hkv, N, d), (B, Hkv, N, d))
    o_lib, g_lib = _library(q, k, v, do, scale, causal=causal)
    o, _ = oracle.attention_fwd(q, k, v, scale, causal)
    _close(o, o_lib, "O")
    for name, g, r in zip(("dQ", "dK", "dV"), oracle.attention_bwd(q, k, v, do, scale, causal), g_lib):
        _close(g, r, name)


@pytest.mark.parametrize("causal", [False, True])
def test_key_padding_matches_library(causal):
    B, H, N, d, scale = 3, 2, 40, 16, 0.5
    kv_len = np.array([40, 17, 1])
    q, k, v, do = _draw(5, *[(B, H, N, d)] * 4)
    keys = np.arange(N)
    allowed = keys[None, None, None, :] < kv_len[:, None, None, None]       # [B, 1, 1, N]
    if causal:
        allowed = allowed & (keys[None, None, None, :] <= keys[None, None, :, None])  # [B, 1, N, N]
    o_lib, g_lib = _library(q, k, v, do, scale, mask=torch.tensor(allowed))
    o, _ = oracle.attention_fwd(q, k, v, scale, causal, kv_len=kv_len)
    _close(o, o_lib, "O")
    grads = oracle.attention_bwd(q, k, v, do, scale, causal, kv_len=kv_len)
    for name, g, r in zip(("dQ", "dK", "dV"), grads, g_lib):
        _close(g, r, name)


@pytest.mark.parametrize("causal", [False, True])
def test_paged_decode_matches_library(causal):
    B, H, Hkv, Mq, d, ps, max_pages, scale = 2, 4, 2, 3, 16, 8, 5, 0.3
    ctx = np.array([37, 9])
    n_pages = B * max_pages + 2
    q, = _draw(6, (B, H, Mq, d))
    kp, vp = _draw(7, (Hkv, n_pages, ps, d), (Hkv, n_pages, ps, d))
    table = np.random.Generator(np.random.PCG64(8)).permutation(n_pages)[:B * max_pages].reshape(B, max_pages)
    o, _ = oracle.paged_attention_fwd(q, kp, vp, table, ctx, scale, causal)
    for b in range(B):
        n = int(ctx[b])
        rows = np.arange(n)
        kb = kp[:, table[b, rows // ps], rows % ps]  # [Hkv, n, d]: the sequence's keys gathered in order
        vb = vp[:, table[b, rows // ps], rows % ps]
        mask = None
        if causal:  # query i sits at position n - Mq + i
            mask = torch.tensor(rows[None, :] <= (n - Mq + np.arange(Mq))[:, None])
        G = H // Hkv
        tq = torch.tensor(q[b])
        tk = torch.tensor(kb).repeat_interleave(G, dim=0)
        tv = torch.tensor(vb).repeat_interleave(G, dim=0)
        ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale).numpy()
        _close(o[b], ref, f"O of sequence {b}")
