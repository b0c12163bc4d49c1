"""fp64 CPU oracle for exact scaled-dot-product attention, forward and backward.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import or call this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it. It shares no code with the
CUDA path and imports nothing from the ``tiled_attention_09_gb300`` package.

Every array is ``numpy.float64`` with layout ``[B, H, N, d]`` (LSE and D are
``[B, H, N]``). Inputs are the fp16/bf16 test inputs upcast exactly to fp64.
Library matrix products (``numpy.matmul``) serve as the only building block;
there is no blocking, fusion or reordering beyond what each function's
docstring states.

Sources (web pages, cited by title and section):

* Page 2, "transformer模型详解（十）：FlashAttention优化技术" (Transformer explained,
  part 10: FlashAttention). Section "Kernel Fusion：消灭中间落盘" gives the
  unfused three-step definition (scores = QK^T, softmax over the last axis,
  output = scores-softmax times V). Section "Tiling 分块策略：匹配硬件极限" gives
  the online softmax (per-tile local max and exponential sum, update of the
  global max with rescaling of the normaliser, one final normalisation).
  Section "Re-computation 而非缓存" gives the recompute-based backward: outer
  loop over K/V column blocks, inner loop over Q row blocks, scores recomputed
  as q_block @ k_block^T / sqrt(d).
* Page 1, "在TPU上移植Flash Attention的工程实践与挑战" (porting Flash Attention to
  TPU). Example 2 ("TPU分块计算处理超长序列", chunked attention over query
  chunks) computes, per chunk of query rows, the full softmax over all keys.

Readings where the pages are silent (each also listed in the design notes):

* scale: an explicit argument, default d^-1/2 (both pages divide the scores by
  sqrt(head_dim)); applied to the logits before max and exp.
* causal mask: query i attends to keys j <= i (the pages name masking only as
  ``attn_bias``); masked logits are -inf, masked probabilities exactly 0.
* LSE: natural log of the sum of exp of the scaled logits, per query row.
* grouped K/V heads (``attention_fwd`` / ``attention_bwd`` only): K and V may
  have H_kv heads with H a multiple of H_kv; query head h reads K/V head
  h // (H / H_kv) (page 3, "高级特性：探索PyTorch/XLA的Pallas内核和Flash
  Attention实现", section "Pallas内核：自定义高效计算的关键", names a multi-query
  attention kernel: H_kv = 1). The gradient of a shared K/V head is the sum of
  its query heads' contributions (chain rule for a shared input).
* key-padding mask (``kv_len``, same two functions): in batch b only keys
  j < kv_len[b] exist for every query (clamped to [0, N]); the masking use of
  an attention bias on page 2, section "精度与稳定性的平衡". A row that sees no
  key has no softmax; read as O = 0, LSE = -inf (the empty sum) and zero
  gradients.
* backward: the page-2 sketch calls a block-local ``softmax(s_ij)``; read as
  P_ij = exp(S_ij - LSE_i) with the saved LSE, which is what makes the
  recomputed block equal to the true probabilities. The gradient formulas
  (D = rowsum(dO*O), dS = P*(dP - D), dQ = scale*dS@K, dK = scale*dS^T@Q,
  dV = P^T@dO) are the chain rule of the forward definition; they are pinned
  by central finite differences in the tests.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "attention_fwd",
    "attention_bwd",
    "chunked_attention_fwd",
    "online_attention_fwd",
    "attention_rows",
    "attention_cols",
    "attention_row_block",
    "head_scores",
    "paged_attention_fwd",
    "split_merge",
]


def _as64(x):
    return np.asarray(x, dtype=np.float64)


def head_scores(q, k, scale, causal, row0=0, kv_len=None):
    """Scaled logits of one (b, h) head: S = scale * q @ k^T, masked to -inf.

    ``q`` holds query rows ``row0 .. row0+len(q)-1`` of the head, ``k`` all keys.
    Page 2, section "Kernel Fusion": scores = q @ k^T (divided by sqrt(d)).
    Masked: keys after the query (causal) and keys j >= kv_len (key padding).
    """
    s = scale * (q @ k.T)
    cols = np.arange(k.shape[0])[None, :]
    if causal:
        rows = np.arange(row0, row0 + q.shape[0])[:, None]
        s = np.where(cols > rows, -np.inf, s)
    if kv_len is not None:
        s = np.where(cols >= kv_len, -np.inf, s)
    return s


def _softmax_rows(s):
    """Row softmax with its log-sum-exp: P = exp(S - LSE), LSE = m + ln(sum exp(S - m)).

    A row whose logits are all -inf (no visible key) gets P = 0 and LSE = -inf.
    """
    m = np.max(s, axis=-1, keepdims=True)
    empty = np.isneginf(m)
    m = np.where(empty, 0.0, m)
    e = np.exp(s - m)
    l = np.sum(e, axis=-1, keepdims=True)
    with np.errstate(divide="ignore"):
        lse = m + np.log(l)
    p = np.where(empty, 0.0, np.exp(s - np.where(empty, 0.0, lse)))
    return p, lse[..., 0]


def _kv_head(h, H, Hkv):
    """K/V head that query head h reads: h // (H / H_kv)."""
    return h // (H // Hkv)


def _key_count(kv_len, b, N):
    """Keys that exist in batch b: kv_len[b] clamped to [0, N] (all N without a mask)."""
    if kv_len is None:
        return None
    return int(min(max(int(kv_len[b]), 0), N))


def attention_fwd(q, k, v, scale, causal=False, kv_len=None):
    """O = softmax(scale * Q K^T [+ causal mask] [+ key-padding mask]) V and LSE, per (b, h) head.

    The definition written out: the full N x N score matrix of each head,
    row softmax, then P @ V (page 2, section "Kernel Fusion", the unfused path).
    k, v may have H_kv heads (H a multiple of H_kv); kv_len: optional [B] key counts.
    Returns (O [B,H,N,d], LSE [B,H,N]).
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    o = np.empty_like(q)
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            hk = _kv_head(h, H, Hkv)
            s = head_scores(q[b, h], k[b, hk], scale, causal, kv_len=_key_count(kv_len, b, N))
            p, l = _softmax_rows(s)
            o[b, h] = p @ v[b, hk]
            lse[b, h] = l
    return o, lse


def attention_bwd(q, k, v, do, scale, causal=False, kv_len=None):
    """Gradients of the forward w.r.t. Q, K, V for upstream dO.

    Per head, with P the forward probabilities and O the oracle's own fp64
    output:  dV = P^T dO;  dP = dO V^T;  D = rowsum(dO * O);  dS = P * (dP - D);
    dQ = scale * dS K;  dK = scale * dS^T Q.
    Page 2, section "Re-computation": the backward rebuilds the scores
    q @ k^T / sqrt(d) and the probabilities instead of storing them; here the
    whole head is rebuilt at once (no blocking). With H_kv < H K/V heads, a K/V
    head's dK and dV are the sums over the query heads that read it.
    Returns (dQ, dK, dV).
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            hk = _kv_head(h, H, Hkv)
            s = head_scores(q[b, h], k[b, hk], scale, causal, kv_len=_key_count(kv_len, b, N))
            p, _ = _softmax_rows(s)
            o = p @ v[b, hk]
            dv[b, hk] += p.T @ do[b, h]
            dp = do[b, h] @ v[b, hk].T
            D = np.sum(do[b, h] * o, axis=-1, keepdims=True)
            ds = p * (dp - D)
            dq[b, h] = scale * (ds @ k[b, hk])
            dk[b, hk] += scale * (ds.T @ q[b, h])
    return dq, dk, dv


def chunked_attention_fwd(q, k, v, scale, causal=False, chunk_size=64):
    """Page-1 Example 2 style: loop over chunks of query rows.

    Each chunk gets the full softmax over all keys and its output rows are
    written into place (page 1, Example 2, "TPU分块计算处理超长序列"). Same
    per-row arithmetic as ``attention_fwd``. Returns (O, LSE).
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, H, N, d = q.shape
    o = np.zeros_like(q)
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            for i in range(0, N, chunk_size):
                qc = q[b, h, i:i + chunk_size]
                s = head_scores(qc, k[b, h], scale, causal, row0=i)
                p, l = _softmax_rows(s)
                o[b, h, i:i + chunk_size] = p @ v[b, h]
                lse[b, h, i:i + chunk_size] = l
    return o, lse


def online_attention_fwd(q, k, v, scale, causal=False, block=128):
    """Page-2 online softmax over key blocks, in fp64.

    Page 2, section "Tiling 分块策略", the three numbered steps: for each key
    block, (1) take the block's local row max and exponential sum; (2) update
    the running max m' = max(m, local max) and rescale the running normaliser
    and accumulator by exp(m - m'); (3) normalise once at the end (O = acc / l).
    LSE = m + ln l. Returns (O, LSE).
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, H, N, d = q.shape
    o = np.empty_like(q)
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            m = np.full((N, 1), -np.inf)
            l = np.zeros((N, 1))
            acc = np.zeros((N, d))
            for j in range(0, N, block):
                kb = k[b, h, j:j + block]
                vb = v[b, h, j:j + block]
                s = scale * (q[b, h] @ kb.T)
                if causal:
                    rows = np.arange(N)[:, None]
                    cols = np.arange(j, j + kb.shape[0])[None, :]
                    s = np.where(cols > rows, -np.inf, s)
                local_max = np.max(s, axis=1, keepdims=True)
                m_new = np.maximum(m, local_max)
                # rows whose keys so far are all masked keep m = -inf; guard the rescale
                finite = np.isfinite(m_new)
                alpha = np.where(finite, np.exp(np.where(finite, m - m_new, 0.0)), 1.0)
                e = np.where(finite, np.exp(s - np.where(finite, m_new, 0.0)), 0.0)
                l = l * alpha + np.sum(e, axis=1, keepdims=True)
                acc = acc * alpha + e @ vb
                m = m_new
            o[b, h] = acc / l
            lse[b, h] = (m + np.log(l))[:, 0]
    return o, lse


def attention_rows(q, k, v, do, scale, causal, rows):
    """Sampled-row mode: O, LSE and dQ for the given query rows of every head.

    All three are row-local (they need only row i of S, P and dP), so each row
    is the definition applied to one query: s = scale * K q_i (masked), LSE_i,
    p = exp(s - LSE_i), O_i = p V, D_i = dO_i . O_i, dp = V dO_i,
    ds = p * (dp - D_i), dQ_i = scale * ds K.
    Returns (O [B,H,R,d], LSE [B,H,R], dQ [B,H,R,d]) for R = len(rows).
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    B, H, N, d = q.shape
    rows = np.asarray(rows)
    R = len(rows)
    o = np.empty((B, H, R, d))
    lse = np.empty((B, H, R))
    dq = np.empty((B, H, R, d))
    for b in range(B):
        for h in range(H):
            s = scale * (q[b, h, rows] @ k[b, h].T)
            if causal:
                s = np.where(np.arange(N)[None, :] > rows[:, None], -np.inf, s)
            p, l = _softmax_rows(s)
            o[b, h] = p @ v[b, h]
            lse[b, h] = l
            D = np.sum(do[b, h, rows] * o[b, h], axis=-1, keepdims=True)
            dp = do[b, h, rows] @ v[b, h].T
            ds = p * (dp - D)
            dq[b, h] = scale * (ds @ k[b, h])
    return o, lse, dq


def attention_cols(q, k, v, do, scale, causal, cols, heads, row_block=1024):
    """Sampled-column mode: dK and dV for the given key columns of some heads.

    dK_j and dV_j sum over every query row, so this needs LSE_i and D_i of all
    rows: the forward of each listed head is run in row blocks of
    ``row_block`` (the definition, one block of rows at a time), then for the
    sampled keys j: P_ij = exp(S_ij - LSE_i), dP_ij = dO_i . V_j,
    dS_ij = P_ij (dP_ij - D_i), dV_j = sum_i P_ij dO_i, dK_j = scale sum_i dS_ij Q_i.
    ``heads`` is a list of (b, h). Returns (dK, dV), each [len(heads), C, d].
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    B, H, N, d = q.shape
    cols = np.asarray(cols)
    C = len(cols)
    dk = np.zeros((len(heads), C, d))
    dv = np.zeros((len(heads), C, d))
    for t, (b, h) in enumerate(heads):
        kc, vc = k[b, h, cols], v[b, h, cols]
        for i in range(0, N, row_block):
            qb = q[b, h, i:i + row_block]
            dob = do[b, h, i:i + row_block]
            s = head_scores(qb, k[b, h], scale, causal, row0=i)
            p, l = _softmax_rows(s)
            ob = p @ v[b, h]
            D = np.sum(dob * ob, axis=-1, keepdims=True)
            pc = p[:, cols]
            dpc = dob @ vc.T
            dsc = pc * (dpc - D)
            dv[t] += pc.T @ dob
            dk[t] += scale * (dsc.T @ qb)
    return dk, dv


def attention_row_block(q, k, v, do, scale, causal, b, h, row0, row1):
    """Forward and backward of one (b, h) head restricted to query rows [row0, row1).

    Every quantity is the definition applied to those rows only: S = scale * Q_blk K^T
    (masked), P = exp(S - LSE), O_blk = P V, D = rowsum(dO_blk * O_blk),
    dS = P * (dO_blk V^T - D), dQ_blk = scale * dS K, and the block's shares of
    the key gradients dK_part = scale * dS^T Q_blk, dV_part = P^T dO_blk. Summing
    the shares over a partition of the rows gives the head's dK and dV.
    Returns (O_blk, LSE_blk, dQ_blk, dK_part, dV_part).
    """
    qb = _as64(q[b, h, row0:row1])
    kh, vh = _as64(k[b, h]), _as64(v[b, h])
    dob = _as64(do[b, h, row0:row1])
    s = head_scores(qb, kh, scale, causal, row0=row0)
    p, lse = _softmax_rows(s)
    o = p @ vh
    D = np.sum(dob * o, axis=-1, keepdims=True)
    ds = p * (dob @ vh.T - D)
    return o, lse, scale * (ds @ kh), scale * (ds.T @ qb), p.T @ dob


def paged_attention_fwd(q, k_pages, v_pages, page_table, ctx_len, scale, causal=False):
    """Decode attention over a paged K/V cache: O [B,H,Mq,d] and LSE [B,H,Mq].

    Page 3, section "Pallas内核：自定义高效计算的关键": a paged multi-query
    attention kernel. Key j of sequence b is row j % page_size of page
    page_table[b][j // page_size] of k_pages / v_pages ([H_kv, n_pages,
    page_size, d]); the sequence has ctx_len[b] keys (clamped to [0, max_pages
    * page_size]). The Mq queries of q[b, h] sit at positions ctx_len[b] - Mq
    + i; causal: query i sees keys j <= ctx_len[b] - Mq + i. The keys are
    gathered into a contiguous sequence and the definition applied to it
    (scores, row softmax, P @ V); a query with no visible key gets O = 0,
    LSE = -inf.
    """
    q, k_pages, v_pages = _as64(q), _as64(k_pages), _as64(v_pages)
    B, H, Mq, d = q.shape
    Hkv, n_pages, ps, _ = k_pages.shape
    max_pages = page_table.shape[1]
    o = np.zeros_like(q)
    lse = np.full((B, H, Mq), -np.inf)
    for b in range(B):
        L = int(min(max(int(ctx_len[b]), 0), max_pages * ps))
        if L == 0:
            continue
        keys = np.arange(L)
        pages = np.asarray(page_table[b])[keys // ps]
        rows = keys % ps
        for h in range(H):
            hk = _kv_head(h, H, Hkv)
            kb = k_pages[hk, pages, rows]
            vb = v_pages[hk, pages, rows]
            s = scale * (q[b, h] @ kb.T)
            if causal:
                pos = (L - Mq + np.arange(Mq))[:, None]
                s = np.where(keys[None, :] > pos, -np.inf, s)
            p, l = _softmax_rows(s)
            o[b, h] = p @ vb
            lse[b, h] = l
    return o, lse


def split_merge(o_parts, lse_parts):
    """Merge attention results computed over disjoint key ranges.

    Each part s holds, per query row, O_s (normalised over its own keys) and
    LSE_s. The page-2 online softmax (section "Tiling 分块策略") combines blocks
    by taking the larger max and rescaling each block's sum and output by
    exp(m_s - m); in log-sum-exp form that is LSE = ln sum_s exp(LSE_s) and
    O = sum_s exp(LSE_s - LSE) O_s. Parts with LSE_s = -inf (no key) weigh 0;
    all of them empty gives O = 0, LSE = -inf. Arrays: o_parts [S, ..., d],
    lse_parts [S, ...].
    """
    o_parts, lse_parts = _as64(o_parts), _as64(lse_parts)
    m = np.max(lse_parts, axis=0)
    empty = np.isneginf(m)
    m0 = np.where(empty, 0.0, m)
    w = np.exp(lse_parts - m0[None])
    total = np.sum(w, axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(empty, -np.inf, m0 + np.log(total))
        o = np.where(empty[..., None], 0.0, np.sum(w[..., None] * o_parts, axis=0) / total[..., None])
    return o, lse
