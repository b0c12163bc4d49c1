"""Parity over seeded random configurations (GPU): forward and backward against the fp64 oracle, every
element, with the options mixed the way a caller may mix them.

Each configuration draws (numpy generator, fixed seed) batch 1-3, 1-8 query heads with a K/V head count
that divides them, a sequence length 1-700 (most not a multiple of any tile), d in {64, 128, 256}, bf16
or fp16, causal or full, a key-padding mask or none (counts anywhere in [0, N], zero included), a split
count for the forward (1, 2 or 4), the input seed, and for d <= 128 how dQ is formed. The checks are the
ones of the fixed-shape tests: O per element within 2e-3 + half an ulp + u * (P|V|) and the literal
bound by count (`check_o`), LSE within 2e-3 (-inf exactly where a query sees no key), dQ, dK and dV
within the gradient tolerance relative to their largest magnitude (or, where the exact gradient is 0 by
cancellation, within the fp32 cancellation bound), padded keys with exactly zero dK and dV and a batch
with no key at all with exactly zero gradients.
"""
import numpy as np
import pytest
import torch

import oracle
import tiled_attention_09_gb300 as fa
from tiled_attention_09_gb300.inputs import Workload, make_inputs
from helpers import cancel_tol, check_grad, check_lse, check_o, ideal_kernel_o, to64

pytestmark = pytest.mark.gpu

N_CONFIGS = 40


def _configs():
    rng = np.random.default_rng(20261203)
    out = []
    for i in range(N_CONFIGS):
        B = int(rng.integers(1, 4))
        H = int(rng.integers(1, 9))
        divisors = [g for g in range(1, H + 1) if H % g == 0]
        Hkv = int(rng.choice(divisors))
        N = int(rng.integers(1, 701)) if i % 4 else int(rng.choice([1, 2, 63, 64, 65, 127, 128, 129, 255, 256]))
        d = int(rng.choice([64, 128, 256]))
        dtype = str(rng.choice(["bf16", "fp16"]))
        causal = bool(rng.integers(0, 2))
        kv_len = None
        if rng.random() < 0.4:
            kv_len = [int(rng.integers(0, N + 1)) for _ in range(B)]
        splits = int(rng.choice([1, 1, 2, 4]))
        dq_mode = str(rng.choice(["default", "separate"])) if d <= 128 else "default"
        w = Workload(B, H, N, d, dtype, causal, seed=int(rng.integers(0, 1 << 16)))
        out.append((w, Hkv, kv_len, splits, dq_mode))
    return out


CONFIGS = _configs()


def _name(c):
    w, Hkv, kl, s, mode = c
    return (f"{w.name()}_Hkv{Hkv}" + ("" if kl is None else "_kv" + "-".join(map(str, kl))) +
            f"_s{s}_{mode}_seed{w.seed}")


@pytest.mark.parametrize("cfg", CONFIGS, ids=_name)
def test_random_config_matches_oracle(cfg):
    w, Hkv, kl, splits, mode = cfg
    q, k, v, do = make_inputs(w)
    k, v = k[:, :Hkv].contiguous(), v[:, :Hkv].contiguous()
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    klc = None if kl is None else torch.tensor(kl, dtype=torch.int32, device="cuda")
    o, lse, o_lo = fa.fwd(qc, kc, vc, causal=w.causal, residual=True, kv_len=klc, kv_splits=splits)
    dq, dk, dv = fa.bwd(qc, kc, vc, o, lse, doc, causal=w.causal, o_lo=o_lo, kv_len=klc, dq_mode=mode)
    torch.cuda.synchronize()
    code, info = fa.device_status()
    assert code == "FA_OK", info

    q64, k64, v64, do64 = to64(q), to64(k), to64(v), to64(do)
    kl64 = None if kl is None else np.array(kl)
    o_ref, lse_ref = oracle.attention_fwd(q64, k64, v64, w.scale, w.causal, kv_len=kl64)
    pv_abs, _ = oracle.attention_fwd(q64, k64, np.abs(v64), w.scale, w.causal, kv_len=kl64)
    check_o(to64(o), o_ref, pv_abs, w.dtype, f"O random {_name(cfg)}",
            ideal=ideal_kernel_o(q64, k64, v64, w.scale, w.dtype, w.causal, kv_len=kl64))
    l_gpu, empty = to64(lse), np.isneginf(lse_ref)
    assert np.isneginf(l_gpu[empty]).all(), "a query with no visible key must get LSE = -inf"
    assert (to64(o)[empty] == 0).all(), "a query with no visible key must get O = 0"
    if (~empty).any():
        check_lse(l_gpu[~empty], lse_ref[~empty], f"LSE random {_name(cfg)}")

    ref = oracle.attention_bwd(q64, k64, v64, do64, w.scale, w.causal, kv_len=kl64)
    # where the exact gradient vanishes by cancellation (a causal row with one key: P = 1, dP = D) the
    # relative rule has no scale and the bound is the fp32 rounding of dP - D (cancel_tol); a batch
    # whose keys are all padded away has P = 0 exactly and must give exact zeros
    floor = cancel_tol(q64, k64, v64, do64, w.scale)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert g.shape == r.shape
        if kl is not None:
            for b in range(w.B):
                if min(kl[b], w.N) <= 0:
                    assert (g[b] == 0).all(), f"{name}: batch {b} sees no key and must get exact zeros"
        check_grad(to64(g), r, name, floor[name])
    if kl is not None:
        for b in range(w.B):
            L = max(0, min(kl[b], w.N))
            assert (dk[b, :, L:] == 0).all() and (dv[b, :, L:] == 0).all(), "padded keys must get zero dK, dV"
