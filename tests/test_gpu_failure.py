"""Failure detection on the GPU without a fault (GPU).

Every wait in the library's kernels is bounded: when it runs out, the kernel records a timeout in a
device status word, stops waiting and returns, and fa_device_status() reports it. Here a self-test
kernel waits on an mbarrier phase that nothing completes (a flag nothing sets); the test checks the
reported status and that the CUDA context still runs attention correctly afterwards.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_09_gb300 as fa
from tiled_attention_09_gb300 import _lib
from tiled_attention_09_gb300.inputs import Workload, make_inputs
from helpers import check_lse, to64

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_the_context_survives():
    L = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert fa.device_status()[0] == "FA_OK"
    t0 = time.perf_counter()
    assert L.fa_selftest_wait_timeout(50_000_000, stream) == 0  # 50 ms
    code, info = fa.device_status()
    elapsed = time.perf_counter() - t0
    assert code == "FA_ERR_TIMEOUT", (code, info)
    assert info[1] == 90 and info[3] >= 1
    assert 0.04 <= elapsed < 5.0
    assert fa.device_status()[0] == "FA_OK"  # read and cleared
    # the context is intact: a forward pass still matches the oracle
    w = Workload(1, 2, 256, 64, "bf16", True)
    q, k, v, _ = make_inputs(w)
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert fa.device_status()[0] == "FA_OK"
    o_ref, lse_ref = oracle.attention_fwd(to64(q), to64(k), to64(v), w.scale, True)
    assert np.abs(to64(o) - o_ref).max() < 3e-2
    check_lse(to64(lse), lse_ref)
