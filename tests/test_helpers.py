"""The ideal-kernel model that scales the O parity tests' count bound (tests/helpers.py), checked on the
CPU against the oracle: its errors stay inside the per-element cap, its masks agree with the oracle's
(causal, key padding, decode alignment), and Q = 0 gives the rounded mean of V."""
import numpy as np
import pytest

import oracle
from tiled_attention_09_gb300.inputs import DecodeWorkload, Workload, make_inputs, make_paged_inputs
from helpers import check_o, ideal_decode_o, ideal_kernel_o, o_tolerance, round16, to64


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
def test_ideal_kernel_within_the_per_element_cap(dtype, causal):
    w = Workload(1, 2, 300, 64, dtype, causal, stress=8.0 if causal else 1.0)
    q, k, v, _ = (to64(t) for t in make_inputs(w))
    o_ref, _ = oracle.attention_fwd(q, k, v, w.scale, causal)
    pv_abs, _ = oracle.attention_fwd(q, k, np.abs(v), w.scale, causal)
    ideal = ideal_kernel_o(q, k, v, w.scale, dtype, causal)
    assert (np.abs(ideal - o_ref) <= o_tolerance(o_ref, pv_abs, dtype)).all()
    assert np.array_equal(ideal, round16(ideal, dtype))  # already rounded to the dtype
    stats = check_o(ideal, o_ref, pv_abs, dtype, "ideal vs oracle", ideal=ideal)
    assert stats["outside"] == stats["ideal_outside"]


def test_ideal_kernel_masks_match_the_oracle():
    w = Workload(3, 4, 130, 32, "bf16", True)
    q, k, v, _ = (to64(t) for t in make_inputs(w))
    k, v = k[:, :2], v[:, :2]
    kv_len = np.array([130, 17, 0])
    o_ref, _ = oracle.attention_fwd(q, k, v, w.scale, True, kv_len=kv_len)
    pv_abs, _ = oracle.attention_fwd(q, k, np.abs(v), w.scale, True, kv_len=kv_len)
    ideal = ideal_kernel_o(q, k, v, w.scale, "bf16", True, kv_len=kv_len)
    assert (ideal[2] == 0).all()  # no visible key: O = 0
    assert (np.abs(ideal - o_ref) <= o_tolerance(o_ref, pv_abs, "bf16")).all()
    rows = np.array([0, 5, 129])
    assert np.array_equal(ideal_kernel_o(q, k, v, w.scale, "bf16", True, kv_len=kv_len, rows=rows),
                          ideal[:, :, rows])


def test_ideal_decode_matches_the_paged_oracle():
    dw = DecodeWorkload(2, 8, 2, 3, 64, 16, 12, (150, 2), causal=True)
    q, kp, vp, table, ctx = make_paged_inputs(dw)
    q64, kp64, vp64 = to64(q), to64(kp), to64(vp)
    o_ref, _ = oracle.paged_attention_fwd(q64, kp64, vp64, table.numpy(), ctx.numpy(), dw.scale, True)
    pv_abs, _ = oracle.paged_attention_fwd(q64, kp64, np.abs(vp64), table.numpy(), ctx.numpy(), dw.scale, True)
    ideal = ideal_decode_o(q64, kp64, vp64, table.numpy(), ctx.numpy(), dw.scale, "bf16", True)
    assert np.isfinite(ideal).all()
    assert (np.abs(ideal - o_ref) <= o_tolerance(o_ref, pv_abs, "bf16")).all()


def test_ideal_kernel_q_zero_is_the_rounded_mean():
    rng = np.random.default_rng(3)
    v = round16(rng.standard_normal((1, 1, 64, 16)), "bf16").astype(np.float64)
    q = np.zeros_like(v)
    ideal = ideal_kernel_o(q, v, v, 0.25, "bf16", False)
    want = round16(np.broadcast_to(v.mean(axis=2, keepdims=True, dtype=np.float32), v.shape), "bf16")
    assert np.abs(ideal - want).max() <= 2.0 ** -7 * np.abs(want).max()
