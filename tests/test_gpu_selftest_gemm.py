"""Tensor-core operand forms against a CPU matrix product (GPU).

Every operand layout the attention kernels hand to tcgen05.mma (K-major and
MN-major 128-byte-swizzled shared memory filled by TMA; A in tensor memory) is
checked here on its own, so a descriptor mistake shows up as a wrong product.
"""
import itertools

import pytest
import torch

import tiled_attention_09_gb300 as fa

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("n,k", [(64, 64), (128, 128), (64, 128), (256, 128), (128, 64)])
@pytest.mark.parametrize("a_mode,b_mode", list(itertools.product([0, 1, 2], [0, 1])))
def test_selftest_gemm(dtype, n, k, a_mode, b_mode):
    g = torch.Generator().manual_seed(1000 + n + k + 10 * a_mode + b_mode)
    A = torch.randn(128, k, generator=g).to(dtype)
    Bm = torch.randn(n, k, generator=g).to(dtype)
    ref = A.double() @ Bm.double().T
    a_store = A.T.contiguous() if a_mode == 1 else A.contiguous()
    b_store = Bm.T.contiguous() if b_mode == 1 else Bm.contiguous()
    d = fa.selftest_gemm(a_store.cuda(), b_store.cuda(), n, k, a_mode, b_mode)
    torch.cuda.synchronize()
    code, info = fa.device_status()
    assert code == "FA_OK", info
    got = d.double().cpu()
    err = (got - ref).abs().max().item()
    assert err <= 1e-5 * k * ref.abs().max().item() + 1e-4, err
