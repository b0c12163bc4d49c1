"""Pins for the fp64 oracle, each against something other than the oracle itself.

CPU only. The pins: a hand-derived worked example (tests/golden), closed forms
(Q = 0, dominant key, N = 1, causal row 0, V = 1), invariants (gradient sums,
key shift, logit-scale trade, key permutation), agreement of the three
independent forward formulations (full matrix, page-1 query chunks, page-2
online softmax over key blocks), the sampled-row / sampled-column modes, and
central finite differences of the backward.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _ev(expr):
    return float(eval(expr, {"ln3": math.log(3), "ln4": math.log(4), "ln2": math.log(2)}))


# ---------------------------------------------------------------- golden
@pytest.mark.parametrize("causal", [False, True])
def test_golden_two_key_example(causal):
    g = json.load(open(os.path.join(HERE, "golden", "two_key_example.json")))
    inp = {k: np.array([_ev(x) for x in v]).reshape(1, 1, 2, 1) for k, v in g["inputs"].items() if k != "scale"}
    scale = _ev(g["inputs"]["scale"])
    exp = g["expected"]["causal" if causal else "noncausal"]
    o, lse = oracle.attention_fwd(inp["q"], inp["k"], inp["v"], scale, causal)
    dq, dk, dv = oracle.attention_bwd(inp["q"], inp["k"], inp["v"], inp["do"], scale, causal)
    for name, got in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        want = np.array([_ev(x) for x in exp[name]])
        np.testing.assert_allclose(got.reshape(-1), want, rtol=0, atol=1e-14, err_msg=name)


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("causal", [False, True])
def test_q_zero_is_uniform_attention(causal):
    B, H, N, d = 1, 2, 37, 8
    q = np.zeros((B, H, N, d))
    k, v = _rand((B, H, N, d), 1), _rand((B, H, N, d), 2)
    o, lse = oracle.attention_fwd(q, k, v, 0.3, causal)
    if causal:
        want = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
        want_lse = np.log(np.arange(1, N + 1))[None, None, :].repeat(H, 1)
    else:
        want = np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
        want_lse = np.full((B, H, N), math.log(N))
    np.testing.assert_allclose(o, want, atol=1e-13)
    np.testing.assert_allclose(lse, want_lse, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_dominant_key_is_one_hot(causal):
    B, H, N, d = 1, 1, 50, 4
    jstar = 17
    a, b, scale = 8.0, 10.0, 0.5  # scale*a*b = 40
    q = np.zeros((B, H, N, d)); q[..., 0] = a
    k = np.zeros((B, H, N, d)); k[0, 0, jstar, 0] = b
    v = _rand((B, H, N, d), 3)
    o, _ = oracle.attention_fwd(q, k, v, scale, causal)
    for i in range(N):
        if causal and i < jstar:
            want = v[0, 0, : i + 1].mean(axis=0)  # all visible logits are 0
            np.testing.assert_allclose(o[0, 0, i], want, atol=1e-13)
        else:
            np.testing.assert_allclose(o[0, 0, i], v[0, 0, jstar], atol=N * math.exp(-40) * 10)


def test_single_key():
    q, k, v, do = (_rand((2, 3, 1, 5), s) for s in range(4))
    scale = 0.7
    o, lse = oracle.attention_fwd(q, k, v, scale, False)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, scale, False)
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse, scale * np.sum(q * k, axis=-1), atol=1e-14)
    np.testing.assert_allclose(dv, do, atol=1e-15)
    np.testing.assert_allclose(dq, 0, atol=1e-15)
    np.testing.assert_allclose(dk, 0, atol=1e-15)


def test_causal_row_zero_sees_key_zero():
    q, k, v = (_rand((1, 2, 33, 8), s) for s in range(3))
    o, lse = oracle.attention_fwd(q, k, v, 0.35, True)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], atol=1e-15)
    np.testing.assert_allclose(lse[:, :, 0], 0.35 * np.sum(q[:, :, 0] * k[:, :, 0], -1), atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_values_give_constant_output(causal):
    q, k = _rand((1, 2, 40, 8), 5) * 3, _rand((1, 2, 40, 8), 6) * 3
    o, _ = oracle.attention_fwd(q, k, np.ones_like(q), 0.35, causal)
    np.testing.assert_allclose(o, 1.0, atol=1e-14)


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("causal", [False, True])
def test_gradient_sums(causal):
    q, k, v, do = (_rand((2, 2, 45, 8), s) for s in range(4))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, 0.4, causal)
    # softmax is invariant to a shift of all logits of a row -> sum_j dS_ij = 0
    np.testing.assert_allclose(dk.sum(axis=2), 0, atol=1e-12)
    # every row of P sums to 1 -> sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(causal):
    q, k, v = (_rand((1, 2, 30, 8), s) for s in range(3))
    c = _rand((8,), 9)
    o1, lse1 = oracle.attention_fwd(q, k, v, 0.4, causal)
    o2, lse2 = oracle.attention_fwd(q, k + c, v, 0.4, causal)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(lse2 - lse1, 0.4 * (q @ c), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_scale_trade(causal):
    q, k, v = (_rand((1, 2, 30, 8), s) for s in range(3))
    o1, lse1 = oracle.attention_fwd(q, k, v, 0.4, causal)
    o2, lse2 = oracle.attention_fwd(2.5 * q, k, v, 0.4 / 2.5, causal)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(lse1, lse2, atol=1e-12)


def test_key_permutation_invariance():
    q, k, v = (_rand((1, 2, 30, 8), s) for s in range(3))
    perm = np.random.default_rng(4).permutation(30)
    o1, _ = oracle.attention_fwd(q, k, v, 0.4, False)
    o2, _ = oracle.attention_fwd(q, k[:, :, perm], v[:, :, perm], 0.4, False)
    np.testing.assert_allclose(o1, o2, atol=1e-12)


def test_causal_prefix_independence():
    """Causal row i must not depend on keys/values after i."""
    q, k, v = (_rand((1, 1, 30, 8), s) for s in range(3))
    o1, lse1 = oracle.attention_fwd(q, k, v, 0.4, True)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, 20:] = 100.0
    v2[:, :, 20:] = -7.0
    o2, lse2 = oracle.attention_fwd(q, k2, v2, 0.4, True)
    np.testing.assert_allclose(o1[:, :, :20], o2[:, :, :20], atol=1e-14)
    np.testing.assert_allclose(lse1[:, :, :20], lse2[:, :, :20], atol=1e-14)
    assert np.abs(o1[:, :, 25] - o2[:, :, 25]).max() > 1e-3


# ---------------------------------------------------------------- formulations
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [64, 200, 257])
def test_chunked_and_online_match_direct(causal, N):
    q, k, v = (_rand((2, 2, N, 16), s) * 2 for s in range(3))
    o, lse = oracle.attention_fwd(q, k, v, 0.25, causal)
    oc, lsec = oracle.chunked_attention_fwd(q, k, v, 0.25, causal, chunk_size=64)
    oo, lseo = oracle.online_attention_fwd(q, k, v, 0.25, causal, block=48)
    np.testing.assert_allclose(oc, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lsec, lse, rtol=0, atol=1e-13)
    np.testing.assert_allclose(oo, o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lseo, lse, rtol=1e-12, atol=1e-12)


def test_online_softmax_large_logits():
    """Logits of several hundred: the running-max rescale must not overflow."""
    q, k, v = (_rand((1, 1, 300, 8), s) for s in range(3))
    q *= 40.0
    o, lse = oracle.attention_fwd(q, k, v, 0.5, True)
    oo, lseo = oracle.online_attention_fwd(q, k, v, 0.5, True, block=64)
    assert np.isfinite(o).all() and np.abs(lse).max() > 100
    np.testing.assert_allclose(oo, o, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(lseo, lse, rtol=1e-12, atol=1e-10)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_modes_match_full(causal):
    B, H, N, d = 1, 2, 300, 16
    q, k, v, do = (_rand((B, H, N, d), s) for s in range(4))
    o, lse = oracle.attention_fwd(q, k, v, 0.25, causal)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, 0.25, causal)
    rows = [0, 1, 127, 128, 150, 299]
    ro, rl, rdq = oracle.attention_rows(q, k, v, do, 0.25, causal, rows)
    np.testing.assert_allclose(ro, o[:, :, rows], atol=1e-13)
    np.testing.assert_allclose(rl, lse[:, :, rows], atol=1e-13)
    np.testing.assert_allclose(rdq, dq[:, :, rows], atol=1e-13)
    cols = [0, 5, 128, 299]
    ck, cv = oracle.attention_cols(q, k, v, do, 0.25, causal, cols, heads=[(0, 1)], row_block=64)
    np.testing.assert_allclose(ck[0], dk[0, 1, cols], atol=1e-13)
    np.testing.assert_allclose(cv[0], dv[0, 1, cols], atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_row_blocks_partition_the_head(causal):
    B, H, N, d = 1, 2, 200, 8
    q, k, v, do = (_rand((B, H, N, d), 20 + s) for s in range(4))
    o, lse = oracle.attention_fwd(q, k, v, 0.3, causal)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, 0.3, causal)
    dk_sum, dv_sum = np.zeros((N, d)), np.zeros((N, d))
    for r0 in range(0, N, 64):
        r1 = min(N, r0 + 64)
        ob, lb, dqb, dkp, dvp = oracle.attention_row_block(q, k, v, do, 0.3, causal, 0, 1, r0, r1)
        np.testing.assert_allclose(ob, o[0, 1, r0:r1], atol=1e-13)
        np.testing.assert_allclose(lb, lse[0, 1, r0:r1], atol=1e-13)
        np.testing.assert_allclose(dqb, dq[0, 1, r0:r1], atol=1e-13)
        dk_sum += dkp
        dv_sum += dvp
    np.testing.assert_allclose(dk_sum, dk[0, 1], atol=1e-12)
    np.testing.assert_allclose(dv_sum, dv[0, 1], atol=1e-12)


# ---------------------------------------------------------------- finite differences
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(16, 4), (9, 8)])
def test_backward_matches_central_differences(causal, N, d):
    B, H = 1, 2
    q, k, v, do = (_rand((B, H, N, d), 10 + s) for s in range(4))
    scale = 1 / math.sqrt(d)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, scale, causal)

    def loss(qq, kk, vv):
        o, _ = oracle.attention_fwd(qq, kk, vv, scale, causal)
        return float(np.sum(do * o))

    h = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        fd = np.zeros_like(grad)
        args = [q, k, v]
        for idx in np.ndindex(grad.shape):
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[which][idx] += h
            minus[which][idx] -= h
            fd[idx] = (loss(*plus) - loss(*minus)) / (2 * h)
        assert np.abs(fd - grad).max() <= 1e-6 * np.abs(grad).max(), which


# ---------------------------------------------------------------- grouped K/V heads, key padding
def _fd_grads(q, k, v, do, scale, causal, kv_len=None, h=1e-6):
    """Central differences of L = sum(dO * O) w.r.t. q, k, v, straight from the forward definition."""
    def loss(qq, kk, vv):
        o, _ = oracle.attention_fwd(qq, kk, vv, scale, causal, kv_len=kv_len)
        return float(np.sum(do * o))

    out = []
    args = [q, k, v]
    for which in range(3):
        fd = np.zeros_like(args[which])
        for idx in np.ndindex(fd.shape):
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[which][idx] += h
            minus[which][idx] -= h
            fd[idx] = (loss(*plus) - loss(*minus)) / (2 * h)
        out.append(fd)
    return out


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hkv", [1, 2])
def test_grouped_heads_equal_repeated_heads(causal, Hkv):
    """K/V shared by H / H_kv query heads = plain attention on K/V repeated per query head;
    the shared head's gradient is the sum of the repeated heads' gradients."""
    B, H, N, d = 2, 4, 11, 8
    q, do = _rand((B, H, N, d), 40), _rand((B, H, N, d), 41)
    k, v = _rand((B, Hkv, N, d), 42), _rand((B, Hkv, N, d), 43)
    G = H // Hkv
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    o, lse = oracle.attention_fwd(q, k, v, 0.3, causal)
    o_r, lse_r = oracle.attention_fwd(q, kr, vr, 0.3, causal)
    np.testing.assert_allclose(o, o_r, atol=1e-14)
    np.testing.assert_allclose(lse, lse_r, atol=1e-14)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, 0.3, causal)
    dq_r, dk_r, dv_r = oracle.attention_bwd(q, kr, vr, do, 0.3, causal)
    assert dk.shape == k.shape and dv.shape == v.shape
    np.testing.assert_allclose(dq, dq_r, atol=1e-13)
    np.testing.assert_allclose(dk, dk_r.reshape(B, Hkv, G, N, d).sum(axis=2), atol=1e-13)
    np.testing.assert_allclose(dv, dv_r.reshape(B, Hkv, G, N, d).sum(axis=2), atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_grouped_heads_match_central_differences(causal):
    B, H, Hkv, N, d = 1, 3, 1, 6, 3
    q, do = _rand((B, H, N, d), 50), _rand((B, H, N, d), 51)
    k, v = _rand((B, Hkv, N, d), 52), _rand((B, Hkv, N, d), 53)
    grads = oracle.attention_bwd(q, k, v, do, 0.6, causal)
    for g, fd in zip(grads, _fd_grads(q, k, v, do, 0.6, causal)):
        assert np.abs(fd - g).max() <= 1e-6 * np.abs(g).max()


@pytest.mark.parametrize("causal", [False, True])
def test_key_padding_equals_truncated_keys(causal):
    """kv_len[b] = L: the same as attention over the first L keys only; padded keys get zero gradients."""
    B, H, N, d = 3, 2, 10, 4
    q, k, v, do = (_rand((B, H, N, d), 60 + s) for s in range(4))
    kv_len = np.array([10, 4, 7])
    o, lse = oracle.attention_fwd(q, k, v, 0.5, causal, kv_len=kv_len)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, 0.5, causal, kv_len=kv_len)
    for b, L in enumerate(kv_len):
        if causal:
            # a causal row i < L sees keys 0..i in both problems; rows i >= L see keys 0..L-1
            qb = q[b:b + 1]
            ot, lt = oracle.attention_fwd(qb[:, :, :L], k[b:b + 1, :, :L], v[b:b + 1, :, :L], 0.5, True)
            np.testing.assert_allclose(o[b, :, :L], ot[0], atol=1e-14)
            np.testing.assert_allclose(lse[b, :, :L], lt[0], atol=1e-14)
            of, lf = oracle.attention_fwd(qb, k[b:b + 1, :, :L], v[b:b + 1, :, :L], 0.5, False)
            np.testing.assert_allclose(o[b, :, L:], of[0, :, L:], atol=1e-14)
            np.testing.assert_allclose(lse[b, :, L:], lf[0, :, L:], atol=1e-14)
        else:
            ot, lt = oracle.attention_fwd(q[b:b + 1], k[b:b + 1, :, :L], v[b:b + 1, :, :L], 0.5, False)
            np.testing.assert_allclose(o[b], ot[0], atol=1e-14)
            np.testing.assert_allclose(lse[b], lt[0], atol=1e-14)
            gq, gk, gv = oracle.attention_bwd(q[b:b + 1], k[b:b + 1, :, :L], v[b:b + 1, :, :L], do[b:b + 1], 0.5,
                                              False)
            np.testing.assert_allclose(dq[b], gq[0], atol=1e-13)
            np.testing.assert_allclose(dk[b, :, :L], gk[0], atol=1e-13)
            np.testing.assert_allclose(dv[b, :, :L], gv[0], atol=1e-13)
        assert not dk[b, :, L:].any() and not dv[b, :, L:].any()


def test_key_padding_matches_central_differences():
    B, H, N, d = 2, 1, 6, 3
    q, k, v, do = (_rand((B, H, N, d), 70 + s) for s in range(4))
    kv_len = np.array([4, 6])
    for causal in (False, True):
        grads = oracle.attention_bwd(q, k, v, do, 0.7, causal, kv_len=kv_len)
        for g, fd in zip(grads, _fd_grads(q, k, v, do, 0.7, causal, kv_len=kv_len)):
            assert np.abs(fd - g).max() <= 1e-6 * np.abs(g).max()


@pytest.mark.parametrize("causal", [False, True])
def test_no_visible_key_gives_zero_output(causal):
    B, H, N, d = 2, 2, 5, 4
    q, k, v, do = (_rand((B, H, N, d), 80 + s) for s in range(4))
    kv_len = np.array([0, -3])  # clamped to 0
    o, lse = oracle.attention_fwd(q, k, v, 0.5, causal, kv_len=kv_len)
    assert not o.any() and np.isneginf(lse).all()
    for g in oracle.attention_bwd(q, k, v, do, 0.5, causal, kv_len=kv_len):
        assert not g.any()
    # kv_len >= N is no mask at all
    o2, lse2 = oracle.attention_fwd(q, k, v, 0.5, causal, kv_len=np.array([N, N + 7]))
    o3, lse3 = oracle.attention_fwd(q, k, v, 0.5, causal)
    np.testing.assert_array_equal(o2, o3)
    np.testing.assert_array_equal(lse2, lse3)


# ---------------------------------------------------------------- paged decode, split merge
def _paged(B, Hkv, n_pages, ps, max_pages, d, seed):
    rng = np.random.default_rng(seed)
    kp = rng.standard_normal((Hkv, n_pages, ps, d))
    vp = rng.standard_normal((Hkv, n_pages, ps, d))
    if n_pages >= B * max_pages:  # every sequence its own pages
        table = rng.permutation(n_pages)[:B * max_pages].reshape(B, max_pages)
    else:
        table = np.stack([rng.permutation(n_pages)[:max_pages] for _ in range(B)])
    return kp, vp, table


def _gather(pages, table_b, L):
    ps = pages.shape[2]
    j = np.arange(L)
    return pages[:, table_b[j // ps], j % ps]  # [Hkv, L, d]


@pytest.mark.parametrize("Hkv", [1, 2])
def test_paged_decode_with_all_queries_is_causal_attention(Hkv):
    """Mq = ctx_len: the decode queries are the whole sequence, and causal decode equals causal attention
    over the gathered sequence (bottom-right alignment meets the ordinary causal mask)."""
    B, H, ps, d = 2, 4, 4, 8
    kp, vp, table = _paged(B, Hkv, 12, ps, 5, d, 90)
    L = 17
    q = _rand((B, H, L, d), 91)
    o, lse = oracle.paged_attention_fwd(q, kp, vp, table, np.array([L, L]), 0.4, causal=True)
    for b in range(B):
        kb = _gather(kp, table[b], L)[None]
        vb = _gather(vp, table[b], L)[None]
        oc, lc = oracle.attention_fwd(q[b:b + 1], kb, vb, 0.4, causal=True)
        np.testing.assert_allclose(o[b], oc[0], atol=1e-14)
        np.testing.assert_allclose(lse[b], lc[0], atol=1e-14)


def test_paged_decode_page_permutation_invariance():
    """Moving pages within the pool (and the page table with them) changes nothing; values in pages or rows
    past ctx_len never matter."""
    B, H, Hkv, ps, d, n_pages, max_pages = 3, 4, 2, 8, 8, 20, 6
    kp, vp, table = _paged(B, Hkv, n_pages, ps, max_pages, d, 92)
    q = _rand((B, H, 3, d), 93)
    ctx = np.array([41, 8, 0])
    o, lse = oracle.paged_attention_fwd(q, kp, vp, table, ctx, 0.3, causal=True)
    perm = np.random.default_rng(94).permutation(n_pages)
    inv = np.argsort(perm)
    kp2, vp2 = kp[:, perm], vp[:, perm]  # new page i holds old page perm[i]
    o2, lse2 = oracle.paged_attention_fwd(q, kp2, vp2, inv[table], ctx, 0.3, causal=True)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    kp3, vp3 = kp.copy(), vp.copy()
    kp3[:, table[0, 5], 1:] = np.nan  # rows 41.. of sequence 0 (page 5, rows 1..7)
    vp3[:, table[0, 5], 1:] = np.inf
    kp3[:, table[1, 1:]] = np.nan     # sequence 1 uses page 0 only
    o3, lse3 = oracle.paged_attention_fwd(q, kp3, vp3, table, ctx, 0.3, causal=True)
    np.testing.assert_array_equal(o[:2], o3[:2])
    assert not o[2].any() and np.isneginf(lse[2]).all()


@pytest.mark.parametrize("causal", [False, True])
def test_split_merge_recovers_full_attention(causal):
    """Attention over disjoint key ranges, merged by log-sum-exp weights, equals attention over all keys."""
    B, H, N, d = 1, 2, 40, 8
    q, k, v = (_rand((B, H, N, d), 95 + s) for s in range(3))
    o, lse = oracle.attention_fwd(q, k, v, 0.35, causal)
    cuts = [0, 7, 8, 30, 40]  # includes a one-key range
    parts_o, parts_l = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        s = 0.35 * np.einsum("bhid,bhjd->bhij", q, k[:, :, a:b])
        if causal:
            s = np.where(np.arange(a, b)[None, None, None, :] > np.arange(N)[None, None, :, None], -np.inf, s)
        m = s.max(axis=-1, keepdims=True)
        empty = np.isneginf(m)
        e = np.where(empty, 0.0, np.exp(s - np.where(empty, 0.0, m)))
        l = e.sum(axis=-1, keepdims=True)
        with np.errstate(divide="ignore", invalid="ignore"):
            parts_o.append(np.where(empty, 0.0, (e @ v[:, :, a:b]) / l))
            parts_l.append(np.where(empty[..., 0], -np.inf, (m + np.log(l))[..., 0]))
    om, lm = oracle.split_merge(np.stack(parts_o), np.stack(parts_l))
    np.testing.assert_allclose(om, o, atol=1e-13)
    np.testing.assert_allclose(lm, lse, atol=1e-13)
    oe, le = oracle.split_merge(np.zeros((3, 2, d)), np.full((3, 2), -np.inf))
    assert not oe.any() and np.isneginf(le).all()


def test_paged_decode_grouped_heads_equal_repeated_heads():
    B, H, Hkv, ps, d = 2, 6, 2, 16, 8
    kp, vp, table = _paged(B, Hkv, 10, ps, 4, d, 97)
    q = _rand((B, H, 2, d), 98)
    ctx = np.array([50, 33])
    o, lse = oracle.paged_attention_fwd(q, kp, vp, table, ctx, 0.3, causal=False)
    o2, lse2 = oracle.paged_attention_fwd(q, np.repeat(kp, 3, axis=0), np.repeat(vp, 3, axis=0), table, ctx, 0.3)
    np.testing.assert_allclose(o, o2, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, atol=1e-14)
