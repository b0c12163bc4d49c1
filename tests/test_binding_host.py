"""Host-side checks of the Python binding on caller-supplied buffers (CPU; no library call).

The kernels receive only pointers, so ``_check_buf`` and ``_check_workspace`` are what stands between a
wrong-sized output or workspace and a kernel writing past its end. Their GPU counterpart, with CUDA tensors
through the public functions, is ``tests/test_gpu_binding.py``.
"""
import pytest
import torch

import tiled_attention_09_gb300 as fa

CPU = torch.device("cpu")


def test_check_buf_accepts_the_exact_buffer():
    t = torch.empty(2, 3, 5, 8, dtype=torch.bfloat16)
    fa._check_buf(t, (2, 3, 5, 8), torch.bfloat16, CPU, "out")
    fa._check_buf(torch.empty(2, 3, 5), (2, 3, 5), torch.float32, CPU, "lse")


@pytest.mark.parametrize("bad", [
    torch.empty(2, 3, 5, 7, dtype=torch.bfloat16),                                     # shape
    torch.empty(2, 3, 5, 8, dtype=torch.float16),                                      # dtype
    torch.empty(2, 3, 8, 5, dtype=torch.bfloat16).transpose(2, 3),                     # not contiguous
    torch.empty(2 * 3 * 5 * 8, dtype=torch.bfloat16),                                  # flat, same size
    torch.empty(2, 3, 5, 8, dtype=torch.bfloat16, device="meta"),                      # device
    None,
], ids=["shape", "dtype", "strided", "flat", "device", "none"])
def test_check_buf_rejects(bad):
    with pytest.raises(ValueError, match="out"):
        fa._check_buf(bad, (2, 3, 5, 8), torch.bfloat16, CPU, "out")


def test_check_workspace_counts_bytes():
    assert fa._check_workspace(torch.empty(100, dtype=torch.uint8), 100, CPU) == 100
    assert fa._check_workspace(torch.empty(25, dtype=torch.float32), 100, CPU) == 100
    assert fa._check_workspace(torch.empty(26, dtype=torch.float32), 100, CPU) == 104
    with pytest.raises(ValueError, match="holds 96 bytes"):
        fa._check_workspace(torch.empty(24, dtype=torch.float32), 100, CPU)
    with pytest.raises(ValueError):
        fa._check_workspace(torch.empty(200, dtype=torch.uint8)[::2], 50, CPU)  # strided
    with pytest.raises(ValueError):
        fa._check_workspace(torch.empty(200, dtype=torch.uint8, device="meta"), 50, CPU)


def test_public_functions_refuse_host_tensors():
    q = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        fa.fwd(q, q, q)
    with pytest.raises(ValueError, match="CUDA"):
        fa.bwd(q, q, q, q, torch.zeros(1, 1, 16), q)
    pages = torch.zeros(1, 2, 16, 64, dtype=torch.bfloat16)
    i32 = dict(dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        fa.decode(q, pages, pages, torch.zeros(1, 2, **i32), torch.ones(1, **i32))
