"""Tolerances and comparison helpers shared by the GPU parity tests.

Tolerance reading (fixed before any kernel ran; derivation in the design notes):

* O, elementwise:  |O_gpu - O_orc| <= 2e-3 + half_ulp_dtype(O_orc) + u_dtype * (P|V|)_i
  where 2e-3 is the stated bound, half_ulp is the unavoidable rounding of the
  output to fp16/bf16, and u_dtype * (P|V|)_i bounds the error of rounding the
  probabilities P to the input dtype before the P.V tensor-core product
  (u_bf16 = 2^-8, u_fp16 = 2^-11; (P|V|)_i is the oracle's attention output
  with |V| in place of V). The literal max-abs error and the share of elements
  inside 2e-3 + half_ulp are reported alongside.
* LSE: |LSE_gpu - LSE_orc| <= 2e-3 (fp32 output).
* dQ, dK, dV: max|g_gpu - g_orc| <= 1e-2 * max|g_orc|, per tensor. Where the exact
  gradient is zero (a single key: the softmax is the constant 1, so dQ = dK = 0
  and dS = P (dP - D) is pure cancellation), that relative rule has no scale;
  there the bound is fp32 rounding of the cancelling terms (cancel_tol).
"""
from __future__ import annotations

import numpy as np
import torch

UNIT_ROUNDOFF = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11}
MANT_BITS = {"bf16": 7, "fp16": 10}


def half_ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1e-30)))
    if dtype == "fp16":
        e = np.maximum(e, -14)  # subnormal spacing
    return np.where(ax > 0, 2.0 ** (e - MANT_BITS[dtype] - 1), 0.0)


def o_tolerance(o_ref: np.ndarray, pv_abs: np.ndarray, dtype: str) -> np.ndarray:
    return 2e-3 + half_ulp(o_ref, dtype) + UNIT_ROUNDOFF[dtype] * pv_abs


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_o(o_gpu: np.ndarray, o_ref: np.ndarray, pv_abs: np.ndarray, dtype: str, what: str = "O"):
    err = np.abs(o_gpu - o_ref)
    tol = o_tolerance(o_ref, pv_abs, dtype)
    bad = err > tol
    literal = float(np.mean(err <= 2e-3 + half_ulp(o_ref, dtype)))
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite values"
    assert not bad.any(), (
        f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; max err {err.max():.3e}; "
        f"worst excess {(err - tol).max():.3e}")
    return {"max_abs": float(err.max()), "within_2e-3+half_ulp": literal}


def check_lse(lse_gpu: np.ndarray, lse_ref: np.ndarray, what: str = "LSE"):
    err = np.abs(lse_gpu - lse_ref)
    assert np.isfinite(lse_gpu).all(), f"{what}: non-finite values"
    assert err.max() <= 2e-3, f"{what}: max err {err.max():.3e}"
    return float(err.max())


def check_grad(g_gpu: np.ndarray, g_ref: np.ndarray, what: str, abs_tol: float = 0.0):
    scale = np.abs(g_ref).max()
    err = np.abs(g_gpu - g_ref).max()
    tol = max(1e-2 * scale, abs_tol)
    assert np.isfinite(g_gpu).all(), f"{what}: non-finite values"
    assert err <= tol, f"{what}: max err {err:.3e} vs tolerance {tol:.3e} (1e-2 * max|g| = {1e-2 * scale:.3e})"
    return float(err / scale) if scale > 0 else 0.0


def cancel_tol(q: np.ndarray, k: np.ndarray, v: np.ndarray, do: np.ndarray, scale: float) -> dict:
    """Absolute error bound for dQ and dK from fp32 cancellation in dS = P (dP - D).

    dP_ij = dO_i . V_j and D_i = dO_i . O_i are d-term fp32 dot products, each within
    d * 2^-24 * sum_k |dO_ik V_jk| of its exact value; their difference is that large even when
    the exact gradient is 0. Doubled for the two products, doubled again for P's rounding, then
    carried through dQ = scale * dS K (dK = scale * dS^T Q) for one key (or query): the bound
    matters only where the exact gradient vanishes.
    """
    d = q.shape[-1]
    G = do.shape[1] // v.shape[1]  # query heads per K/V head
    absdot = np.einsum("bhik,bhjk->bhij", np.abs(do), np.repeat(np.abs(v), G, axis=1)).max()
    base = 4 * d * 2.0 ** -24 * scale * absdot
    return {"dQ": base * np.abs(k).max(), "dK": base * np.abs(q).max(), "dV": 0.0}
