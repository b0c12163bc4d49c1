"""Seeded synthetic inputs shared by the CUDA path's tests, the bench and the oracle's tests.

This module holds no attention arithmetic. It draws Q, K, V and dO the same way
for every consumer, so that the GPU path and the fp64 oracle always see
bit-identical inputs:

* numpy's PCG64 bit generator seeded with ``seed`` and its float32
  ``standard_normal``, drawn in the order Q, K, V, dO, each shaped
  ``[B, H, N, d]`` (the layout of the pages' own examples: the query-chunked JAX
  example on page 1 and the XLA example on page 2 both use
  ``(batch, heads, seq, head_dim)``). ``torch.randn`` is not used: its CPU
  output differs in the last bits between x86 and Arm builds, which moved a few
  values to a neighbouring bf16 and made inputs machine-dependent;
* a cast to fp16 or bf16 (round to nearest even);
* for the stress variant, the cast Q and K are multiplied by 8, which is exact
  in both formats and pushes the scaled logits to a few hundred.

It also holds the sampled-row and sampled-column recipes used where the full
fp64 oracle is too slow (sequence length above 2048).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, dtype, mask and input recipe."""

    B: int
    H: int
    N: int
    d: int
    dtype: str = "bf16"
    causal: bool = False
    stress: float = 1.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    def fwd_flops(self) -> float:
        """4*B*H*N^2*d, halved when causal (the metric's own count)."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        return 2.5 * self.fwd_flops()

    def name(self) -> str:
        s = f"B{self.B}_H{self.H}_N{self.N}_d{self.d}_{self.dtype}_{'causal' if self.causal else 'full'}"
        if self.stress != 1.0:
            s += f"_x{self.stress:g}"
        return s


# The five workloads the build is measured and checked on.
SMALL = Workload(1, 2, 256, 64, "fp16", False)
PAGES_SHAPE = Workload(2, 12, 1024, 64, "fp16", False)
CAUSAL_4K = Workload(2, 12, 4096, 128, "bf16", True)
CAUSAL_4K_STRESS = Workload(2, 12, 4096, 128, "bf16", True, stress=8.0)
LONG_32K = Workload(1, 8, 32768, 128, "bf16", True)


def sweep_workloads():
    out = []
    for d in (64, 128, 256):
        for N in (512, 1024, 2048, 4096, 8192, 16384):
            for dt in ("bf16", "fp16"):
                for causal in (True, False):
                    out.append(Workload(2, 12, N, d, dt, causal))
    return out


def make_inputs_fp32(w: Workload):
    """The fp32 draws behind ``make_inputs`` (before the cast and the stress factor)."""
    rng = np.random.Generator(np.random.PCG64(w.seed))
    shape = (w.B, w.H, w.N, w.d)
    return tuple(torch.from_numpy(rng.standard_normal(shape, dtype=np.float32)) for _ in range(4))  # Q, K, V, dO


def cast_inputs(w: Workload, fp32):
    """``make_inputs`` from already drawn fp32 values: cast to ``w.torch_dtype`` (RNE), then stress Q and K."""
    q, k, v, do = (x.to(w.torch_dtype) for x in fp32)
    if w.stress != 1.0:
        q = q * w.stress
        k = k * w.stress
    return q, k, v, do


def make_inputs(w: Workload):
    """Return q, k, v, do as CPU tensors of ``w.torch_dtype``, shape [B,H,N,d]."""
    return cast_inputs(w, make_inputs_fp32(w))


def make_inputs_device(w: Workload, device, n_kv_heads: int | None = None):
    """q [B,H,N,d] and k, v, do drawn on ``device`` for tensors too large to draw on the host in seconds.

    ``torch.randn`` with a ``torch.Generator`` on the device, seeded with ``w.seed``, in the order Q, K,
    V, dO, directly in ``w.torch_dtype``; k and v have ``n_kv_heads`` heads (default H). The values
    depend on the device and the torch build, so a consumer copies back whatever it checks: the oracle
    then reads exactly the values the CUDA path read.
    """
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    hkv = w.H if n_kv_heads is None else n_kv_heads
    shapes = ((w.B, w.H, w.N, w.d), (w.B, hkv, w.N, w.d), (w.B, hkv, w.N, w.d), (w.B, w.H, w.N, w.d))
    return tuple(torch.randn(s, generator=g, device=device, dtype=w.torch_dtype) for s in shapes)


def sample_rows(N: int, n_random: int = 57, seed: int = 1):
    """Query rows checked when the full oracle is too slow.

    {0, 1, 127, 128, 129, N/2, N-1} plus ``n_random`` distinct random rows drawn
    with a CPU generator seeded by ``seed``. Sorted, unique, all < N.
    """
    fixed = {0, 1, 127, 128, 129, N // 2, N - 1}
    fixed = {r for r in fixed if 0 <= r < N}
    perm = np.random.Generator(np.random.PCG64(seed)).permutation(N).tolist()
    extra = [r for r in perm if r not in fixed][:n_random]
    return sorted(fixed | set(extra))


def sample_cols(N: int, n: int = 64, seed: int = 1):
    """Key columns checked for dK and dV when the full oracle is too slow."""
    fixed = {0, N - 1, N // 2}
    perm = np.random.Generator(np.random.PCG64(seed + 1000)).permutation(N).tolist()
    extra = [c for c in perm if c not in fixed][: max(0, n - len(fixed))]
    return sorted(fixed | set(extra))


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """One paged-decode problem: Mq new queries per sequence over a paged K/V pool.

    ``ctx`` gives each sequence's cached length. The pool holds ``B * max_pages`` pages plus
    ``spare`` pages no sequence uses; each sequence owns ``max_pages`` distinct pages in a random
    order (so neighbouring keys live in scattered pages).
    """

    B: int
    H: int
    Hkv: int
    Mq: int
    d: int
    page_size: int
    max_pages: int
    ctx: tuple
    dtype: str = "bf16"
    causal: bool = False
    spare: int = 3
    seed: int = 0
    poison: bool = True  # rows past a sequence's end (in its own pages) hold NaN, as a stale cache may

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def n_pages(self) -> int:
        return self.B * self.max_pages + self.spare

    def kv_bytes(self) -> int:
        """Bytes of K and V the sequences' keys occupy (what one decode step must read)."""
        keys = sum(min(max(c, 0), self.max_pages * self.page_size) for c in self.ctx)
        return 2 * keys * self.Hkv * self.d * 2

    def flops(self) -> float:
        keys = sum(min(max(c, 0), self.max_pages * self.page_size) for c in self.ctx)
        return 4.0 * keys * self.H * self.Mq * self.d

    def name(self) -> str:
        ctx = str(self.ctx[0]) if len(set(self.ctx)) == 1 else "-".join(map(str, self.ctx))
        return (f"B{self.B}_H{self.H}_Hkv{self.Hkv}_Mq{self.Mq}_d{self.d}_ps{self.page_size}_"
                f"ctx{ctx}_{self.dtype}_{'causal' if self.causal else 'full'}")


def make_paged_inputs(w: DecodeWorkload):
    """q [B,H,Mq,d], k_pages, v_pages [Hkv,n_pages,page_size,d] (w.dtype), page_table int32 [B,max_pages],
    ctx_len int32 [B], all CPU tensors. PCG64(seed): q, k_pages, v_pages as float32 standard normals, then
    the page assignment as one permutation of the pool."""
    rng = np.random.Generator(np.random.PCG64(w.seed))
    q = rng.standard_normal((w.B, w.H, w.Mq, w.d), dtype=np.float32)
    kp = rng.standard_normal((w.Hkv, w.n_pages, w.page_size, w.d), dtype=np.float32)
    vp = rng.standard_normal((w.Hkv, w.n_pages, w.page_size, w.d), dtype=np.float32)
    table = rng.permutation(w.n_pages)[: w.B * w.max_pages].reshape(w.B, w.max_pages).astype(np.int32)
    ctx = np.asarray(w.ctx, dtype=np.int32)
    if w.poison:
        for b in range(w.B):
            L = int(min(max(ctx[b], 0), w.max_pages * w.page_size))
            for j in range(L, w.max_pages * w.page_size):
                pg, row = table[b, j // w.page_size], j % w.page_size
                kp[:, pg, row] = np.nan
                vp[:, pg, row] = np.nan
    dt = DTYPES[w.dtype]
    return (torch.from_numpy(q).to(dt), torch.from_numpy(kp).to(dt), torch.from_numpy(vp).to(dt),
            torch.from_numpy(table), torch.from_numpy(ctx))
