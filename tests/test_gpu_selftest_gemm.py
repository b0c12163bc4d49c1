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


@pytest.mark.parametrize("n,a_tmem,n_acc", [(64, 0, 1), (64, 0, 2), (64, 0, 4), (64, 1, 4), (128, 0, 1),
                                            (128, 0, 2), (128, 0, 4), (128, 1, 2), (256, 0, 1), (256, 1, 1),
                                            (256, 0, 2)])
def test_mma_rate_microbenchmark(n, a_tmem, n_acc):
    """Sustained cycles per tcgen05.mma (M=128, N=n, K=16): never faster than the nominal dense rate."""
    import ctypes
    from tiled_attention_09_gb300 import _lib
    L = _lib.load()
    blocks = torch.cuda.get_device_properties(0).multi_processor_count
    reps = 2048
    cyc = torch.zeros(blocks, dtype=torch.int64, device="cuda")
    code = L.fa_selftest_mma_rate(n, a_tmem, n_acc, reps, blocks, ctypes.c_void_p(cyc.data_ptr()),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0
    torch.cuda.synchronize()
    assert fa.device_status()[0] == "FA_OK"
    per_mma = cyc.double().median().item() / (8 * reps)
    flop_per_clk = 2 * 128 * n * 16 / per_mma
    print(f"MMA rate n={n} a_tmem={a_tmem} n_acc={n_acc}: {per_mma:.1f} cycles/instr, {flop_per_clk:.0f} FLOP/clk/SM")
    assert per_mma >= n / 2 * 0.95  # nominal 8192 dense bf16 FLOP/clk/SM


def test_ex2_rate_microbenchmark():
    """Exponentials per second of the whole GPU: finite results, and a rate between 1e12/s and the
    nominal 32 per clock per SM at 2.1 GHz."""
    import ctypes
    from tiled_attention_09_gb300 import _lib
    L = _lib.load()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sink = torch.zeros(2 * sms, dtype=torch.float32, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.fa_selftest_ex2_rate(64, 2 * sms, ctypes.c_void_p(sink.data_ptr()), st) == 0  # warm-up
    reps = 4096
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    assert L.fa_selftest_ex2_rate(reps, 2 * sms, ctypes.c_void_p(sink.data_ptr()), st) == 0
    e1.record()
    torch.cuda.synchronize()
    rate = 2 * sms * 512 * 8 * reps / (e0.elapsed_time(e1) / 1e3)
    print(f"ex2 rate {rate / 1e12:.2f} T/s = {rate / sms / 2.07e9:.1f} per clock per SM at 2.07 GHz")
    assert torch.isfinite(sink).all()
    assert 1e12 < rate < 32 * sms * 2.1e9


PATTERNS = [  # (n, a_tmem, a_mn, b_mn, issuers, mode): the shapes and operand forms of the attention kernels
    (64, 0, 0, 0, 1, 0), (128, 0, 0, 0, 1, 0), (256, 0, 0, 0, 1, 0), (64, 1, 0, 0, 1, 0), (128, 1, 0, 0, 1, 0),
    (256, 1, 0, 0, 1, 0), (128, 1, 0, 1, 1, 0), (64, 0, 1, 1, 1, 0), (128, 0, 1, 1, 1, 0), (128, 0, 0, 1, 1, 0),
    (64, 0, 0, 0, 2, 0), (128, 0, 0, 0, 2, 0), (128, 1, 0, 1, 2, 0),
    (64, 0, 0, 0, 4, 0), (128, 0, 0, 0, 4, 0), (128, 0, 1, 1, 4, 0), (64, 1, 0, 0, 4, 0), (64, 1, 0, 1, 4, 0),
    (128, 1, 0, 0, 1, 1), (64, 1, 0, 1, 2, 1), (64, 1, 0, 0, 1, 1),
    (64, 0, 0, 0, 1, 2), (128, 0, 0, 0, 1, 2), (128, 0, 0, 0, 2, 2),
]


@pytest.mark.parametrize("n,a_tmem,a_mn,b_mn,issuers,mode", PATTERNS)
def test_mma_pattern_microbenchmark(n, a_tmem, a_mn, b_mn, issuers, mode):
    """Cycles per tcgen05.mma with distinct random operand tiles: never faster than the nominal
    dense rate; prints the shared-memory operand bytes the tensor core read per cycle."""
    import ctypes
    from tiled_attention_09_gb300 import _lib
    L = _lib.load()
    blocks = torch.cuda.get_device_properties(0).multi_processor_count
    reps = 1024
    cyc = torch.zeros(4 * blocks, dtype=torch.int64, device="cuda")
    code = L.fa_selftest_mma_pattern(n, a_tmem, a_mn, b_mn, issuers, mode, reps, blocks,
                                     ctypes.c_void_p(cyc.data_ptr()),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0
    torch.cuda.synchronize()
    assert fa.device_status()[0] == "FA_OK"
    span = cyc.view(blocks, 4)[:, :issuers].amax(dim=1).double().median().item()
    n_mma = 8 * reps * issuers * (2 if mode == 2 else 1)
    per_mma = span / n_mma  # cycles of the SM per instruction, all issuers together
    a_bytes = 128 * 16 * 2
    if mode == 1:
        smem_bytes = a_bytes / 2 + n * 16 * 2  # half the instructions read A from shared memory
    else:
        smem_bytes = (0 if a_tmem else a_bytes) + n * 16 * 2
    print(f"MMA pattern n={n} a_tmem={a_tmem} a_mn={a_mn} b_mn={b_mn} issuers={issuers} mode={mode}: "
          f"{per_mma:.1f} cycles/instr, {2 * 128 * n * 16 / per_mma:.0f} FLOP/clk/SM, "
          f"{smem_bytes / per_mma:.0f} operand B/clk")
    assert per_mma >= n / 2 * 0.95


def test_selftest_copy_between_device_and_pinned_host():
    """fa_selftest_copy (the host-link copy-rate microbenchmark) copies exactly, device to device, pinned host to
    device and device to pinned host, and refuses memory CUDA does not report as device or pinned host memory."""
    import ctypes as _ct
    from tiled_attention_09_gb300 import _lib as _l
    L = _l.load()
    n = (1 << 20) + 48
    src_h = torch.randint(0, 255, (n,), dtype=torch.uint8).pin_memory()
    dst_d = torch.zeros(n, dtype=torch.uint8, device="cuda")
    dst_h = torch.zeros(n, dtype=torch.uint8).pin_memory()
    d2 = torch.zeros(n, dtype=torch.uint8, device="cuda")
    st = _ct.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.fa_selftest_copy(src_h.data_ptr(), dst_d.data_ptr(), n, 7, st) == 0
    assert L.fa_selftest_copy(dst_d.data_ptr(), d2.data_ptr(), n, 3, st) == 0
    assert L.fa_selftest_copy(d2.data_ptr(), dst_h.data_ptr(), n, 152, st) == 0
    torch.cuda.synchronize()
    assert torch.equal(dst_h, src_h) and torch.equal(d2.cpu(), src_h)
    pageable = torch.zeros(n, dtype=torch.uint8)
    assert L.fa_selftest_copy(pageable.data_ptr(), dst_d.data_ptr(), n, 4, st) == 1  # FA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert L.fa_selftest_copy(src_h.data_ptr(), dst_d.data_ptr(), n - 8, 4, st) == 3  # not a multiple of 16
