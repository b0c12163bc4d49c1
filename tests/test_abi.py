"""Host-side checks of the C ABI (CPU only: no call here reaches a CUDA API).

The library must load without a GPU, export every function the headers in
include/ declare, and reject bad arguments synchronously: every case below
returns before the library touches the device, so fake pointer values are
never dereferenced.
"""
import ctypes
import os
import re

import pytest

from tiled_attention_09_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from tiled_attention_09_gb300 import build
    build.build()
    return _lib.load()


def _declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(inc, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(?:fa_status|size_t|const char\s*\*|void|int)\s+(fa_\w+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def _declared_arities():
    """{function: parameter count} from the headers' declarations."""
    out = {}
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if not f.endswith(".h"):
            continue
        text = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, f)).read(), flags=re.S)
        for m in re.finditer(r"\b(?:fa_status|size_t|const char\s*\*|void|int)\s+(fa_\w+)\s*\(([^)]*)\)\s*;", text):
            params = m.group(2).strip()
            out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_ctypes_signatures_match_header_arity():
    ar = _declared_arities()
    assert "fa_decode" in ar and ar["fa_decode"] == 22
    for name, _, args in _lib.SIGNATURES:
        assert len(args) == ar[name], f"{name}: {len(args)} ctypes arguments, {ar[name]} declared"


def test_every_declared_symbol_is_exported_and_bound(L):
    names = _declared_functions()
    assert "fa_fwd" in names and "fa_bwd" in names and len(names) >= 10
    bound = {n for n, _, _ in _lib.SIGNATURES}
    for n in names:
        assert hasattr(L, n), n
        assert n in bound, f"{n} has no ctypes signature"


def test_status_strings_and_version(L):
    for code, name in _lib.STATUS_NAMES.items():
        assert L.fa_status_string(code).decode() == name
    assert L.fa_status_string(99).decode() == "FA_ERR_UNKNOWN"
    assert L.fa_version() == 102


def test_workspace_size(L):
    B, H, N, d = 2, 3, 256, 128
    rows = B * H * ((N + 63) // 64 * 64)  # each head's rows padded to a multiple of 64
    r256 = lambda x: (x + 255) // 256 * 256
    assert L.fa_bwd_workspace_size(B, H, N, d) == r256(rows * 4) * 2 + r256(rows * d * 4)
    assert L.fa_bwd_workspace_size(1, 1, 100, 64) == r256(128 * 4) * 2 + r256(128 * 64 * 4)  # any N >= 1
    assert L.fa_bwd_workspace_size(2, 3, 65, 128) == r256(768 * 4) * 2 + r256(768 * 128 * 4)
    assert L.fa_bwd_workspace_size(1, 1, 0, 64) == 0
    assert L.fa_bwd_workspace_size(1, 1, 256, 96) == 0


P = 1 << 20  # a 16-byte aligned fake address; never dereferenced (calls fail before any device work)
V = ctypes.c_void_p


def fwd(L, q=P, k=P, v=P, o=P, lse=P, B=1, H=1, N=256, d=64, scale=0.125, causal=0, dtype=0):
    return L.fa_fwd(V(q), V(k), V(v), V(o), V(lse), B, H, N, d, scale, causal, dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), 1), (dict(lse=0), 1),
    (dict(N=0), 2), (dict(N=-5), 2), (dict(d=96), 2), (dict(d=32), 2), (dict(B=0), 2),
    (dict(H=-1), 2), (dict(B=1 << 16, H=1 << 8, N=1 << 8), 2), (dict(N=65535 * 128 + 1), 2),
    (dict(dtype=7), 1), (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1), (dict(scale=-1.0), 1),
    (dict(scale=0.0), 1),
    (dict(q=P + 8), 3), (dict(o=P + 2), 3), (dict(lse=P + 4), 3),
])
def test_fwd_rejects_bad_arguments(L, kw, code):
    assert fwd(L, **kw) == code


def bwd(L, ws=P, ws_bytes=1 << 40, N=256, d=64, scale=0.125, dq=P, o_lo=None, **kw):
    return L.fa_bwd(V(P), V(P), V(P), V(P), V(P), V(P), V(dq), V(P), V(P), V(o_lo), V(ws), ws_bytes, 1, 1, N, d,
                    scale, 0, 0, None)


def test_bwd_rejects_bad_arguments(L):
    assert bwd(L, ws=0) == 4
    assert bwd(L, ws_bytes=10) == 4
    assert bwd(L, ws=P + 16) == 3   # workspace must be 256-byte aligned
    assert bwd(L, N=0) == 2
    assert bwd(L, N=65535 * 128 + 1) == 2  # more 128-key blocks than a grid's y extent
    assert bwd(L, scale=float("nan")) == 1
    assert bwd(L, dq=0) == 1
    assert bwd(L, dq=P + 4) == 3
    assert bwd(L, o_lo=P + 8) == 3


def test_fwd_ex_rejects_misaligned_residual(L):
    assert L.fa_fwd_ex(V(P), V(P), V(P), V(P), V(P), V(P + 2), 1, 1, 256, 64, 0.125, 0, 0, None) == 3
    assert L.fa_fwd_ex(V(P), V(P), V(P), V(P), V(0), V(P), 1, 1, 256, 64, 0.125, 0, 0, None) == 1


def fwd_opt(L, H=4, n_kv_heads=0, kv_len=None, o_fp32=0, o_lo=None):
    opt = _lib.FAOptions(n_kv_heads, kv_len, o_fp32)
    return L.fa_fwd_opt(V(P), V(P), V(P), V(P), V(P), V(o_lo), 1, H, 256, 64, 0.125, 0, 0, ctypes.byref(opt), None)


def bwd_opt(L, H=4, n_kv_heads=0, kv_len=None, o_fp32=0, o_lo=None):
    opt = _lib.FAOptions(n_kv_heads, kv_len, o_fp32)
    return L.fa_bwd_opt(V(P), V(P), V(P), V(P), V(P), V(P), V(P), V(P), V(P), V(o_lo), V(P), 1 << 40, 1, H, 256, 64,
                        0.125, 0, 0, ctypes.byref(opt), None)


@pytest.mark.parametrize("call", [fwd_opt, bwd_opt])
def test_options_reject_bad_arguments(L, call):
    assert call(L, n_kv_heads=3) == 2           # 4 query heads cannot share 3 K/V heads evenly
    assert call(L, n_kv_heads=-1) == 1
    assert call(L, kv_len=P + 2) == 3           # int32 key counts need 4-byte alignment
    assert call(L, o_fp32=1, o_lo=P) == 1       # an fp32 O has no rounding residual


def test_selftest_rejects_bad_arguments(L):
    f = L.fa_selftest_gemm
    assert f(V(0), V(P), V(P), 128, 64, 0, 0, 0, None) == 1
    assert f(V(P), V(P), V(P), 96, 64, 0, 0, 0, None) == 2
    assert f(V(P), V(P), V(P), 128, 64, 3, 0, 0, None) == 1
    assert f(V(P + 2), V(P), V(P), 128, 64, 0, 0, 0, None) == 3


def test_python_layer_requires_cuda_tensors():
    import torch
    import tiled_attention_09_gb300 as fa
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fwd(q, q, q)


def test_wait_timeout_selftest_rejects_bad_limits(L):
    assert L.fa_selftest_wait_timeout(10, None) == 1           # below 1 us
    assert L.fa_selftest_wait_timeout(2_000_000_000, None) == 1  # above 1 s


def test_decode_split_choice_and_workspace(L):
    # the library's split count for a shape, and the workspace it implies
    s = L.fa_decode_splits(1, 8, 128, 64, 1024)
    assert 1 <= s <= 64
    assert L.fa_decode_splits(1, 8, 256, 64, 1024) <= 32
    assert L.fa_decode_splits(19, 8, 128, 64, 128) == 1  # 152 CTAs fill the GPU once: no split
    assert L.fa_decode_splits(1, 8, 96, 64, 16) == 0      # unsupported head dimension
    # the counts that timed fastest among 1, 2, 3, 4, 6, 8, 12, 16, 24 on a GB300 (the first within 3%
    # of 16, the fastest)
    for args, best in (((1, 8, 128, 64, 1024), 19), ((16, 8, 128, 64, 128), 1), ((64, 1, 128, 16, 256), 2),
                       ((32, 2, 64, 128, 64), 2), ((8, 8, 128, 256, 64), 2), ((8, 8, 256, 64, 128), 2)):
        assert L.fa_decode_splits(*args) == best, args
    r256 = lambda x: (x + 255) // 256 * 256
    rows = 2 * 16 * 1
    for n_split in (1, 3):
        assert L.fa_decode_workspace_size(2, 16, 4, 1, 128, 64, 32, n_split) == \
            r256(n_split * rows * 128 * 4) + r256(n_split * rows * 4)
    assert L.fa_decode_workspace_size(2, 16, 4, 1, 128, 64, 32, 500) == r256(64 * rows * 128 * 4) + r256(64 * rows * 4)
    assert L.fa_decode_workspace_size(2, 16, 3, 1, 128, 64, 32, 1) == 0   # 16 query heads on 3 K/V heads
    assert L.fa_decode_workspace_size(2, 16, 1, 9, 128, 64, 32, 1) == 0   # 16 heads x 9 queries > 128 rows
    assert L.fa_decode_workspace_size(2, 16, 4, 1, 128, 48, 32, 1) == 0   # page size not a power of two


@pytest.mark.parametrize("kw,code", [
    (dict(page_table=0), 1), (dict(ctx_len=0), 1), (dict(d=96), 2), (dict(page_size=8), 2),
    (dict(H=16, Hkv=3), 2), (dict(scale=0.0), 1), (dict(ws=0), 4), (dict(ws=P + 64), 3), (dict(ws_bytes=16), 4),
    (dict(page_table=P + 2), 3), (dict(q=P + 8), 3),
])
def test_decode_rejects_bad_arguments(L, kw, code):
    a = dict(q=P, kp=P, vp=P, page_table=P, ctx_len=P, o=P, lse=P, ws=P, ws_bytes=1 << 40, B=2, H=16, Hkv=4, Mq=1,
             d=128, page_size=64, n_pages=64, max_pages=32, n_split=0, scale=0.125, causal=0, dtype=1)
    a.update(kw)
    assert L.fa_decode(V(a["q"]), V(a["kp"]), V(a["vp"]), V(a["page_table"]), V(a["ctx_len"]), V(a["o"]), V(a["lse"]),
                       V(a["ws"]), a["ws_bytes"], a["B"], a["H"], a["Hkv"], a["Mq"], a["d"], a["page_size"],
                       a["n_pages"], a["max_pages"], a["n_split"], a["scale"], a["causal"], a["dtype"], None) == code


def test_split_forward_workspace_and_choice(L):
    """Host-side sizing of the split-key forward: partial O [S][B*H*N][d] and LSE [S][B*H*N], fp32, each
    256-byte aligned; none for one range. The library's split count: the counts below are the ones that
    timed fastest among 1, 2, 4, 8 on a GB300 (152 SMs, the count assumed without a device)."""
    r256 = lambda x: (x + 255) // 256 * 256
    B, H, N, d, S = 2, 3, 300, 128, 4
    rows = B * H * N * S
    assert L.fa_fwd_workspace_size(B, H, N, d, S) == r256(rows * d * 4) + r256(rows * 4)
    assert L.fa_fwd_workspace_size(B, H, N, d, 1) == 0 and L.fa_fwd_workspace_size(B, H, N, d, 17) == 0
    assert L.fa_fwd_workspace_size(1, 1, 0, 64, 2) == 0
    measured_best = {
        (1, 1, 4096, 128, 1): 8, (1, 1, 16384, 128, 1): 4, (1, 2, 16384, 128, 1): 2, (2, 2, 8192, 128, 1): 2,
        (1, 1, 8192, 128, 0): 4, (1, 4, 4096, 128, 1): 4, (1, 1, 16384, 64, 1): 4, (1, 1, 8192, 256, 1): 4,
        # many heads: the partial outputs cost more than the shorter critical path saves
        (2, 12, 4096, 128, 1): 1, (2, 12, 1024, 128, 1): 1, (2, 12, 512, 64, 1): 1, (2, 12, 2048, 256, 0): 1,
    }
    for args, s in measured_best.items():
        assert L.fa_fwd_kv_splits(*args) == s, args
    assert L.fa_fwd_kv_splits(1, 1, 128, 64, 0) == 1      # one key tile: nothing to split
    for args in ((1, 2, 1024, 128, 1), (1, 4, 8192, 64, 0), (4, 8, 2048, 256, 1)):
        s = L.fa_fwd_kv_splits(*args)
        assert 1 <= s <= 16 and (s & (s - 1)) == 0



def test_forward_tiles_per_item_choice(L):
    """Query tiles per forward work item: the mode that timed faster on a GB300 (152 SMs, the count assumed
    without a device) for each of these shapes; 1 only where two-tile items would leave SMs idle or make
    the longest item the critical path."""
    measured_best = {  # (B, H, N, d, causal): tiles per item
        (2, 12, 512, 128, 1): 1, (2, 12, 512, 128, 0): 1, (2, 12, 1024, 128, 1): 1, (2, 12, 1024, 128, 0): 2,
        (2, 12, 2048, 128, 1): 2, (2, 12, 4096, 128, 0): 2, (2, 12, 1024, 64, 1): 1, (2, 12, 1024, 64, 0): 2,
        (1, 4, 2048, 128, 1): 1, (1, 4, 4096, 128, 0): 1, (4, 32, 512, 128, 1): 2, (4, 32, 1024, 128, 0): 2,
    }
    for args, t in measured_best.items():
        assert L.fa_fwd_tiles_per_item(*args) == t, args
    assert L.fa_fwd_tiles_per_item(1, 2, 4096, 256, 1) == 1   # d = 256: one tile an item always
    assert L.fa_fwd_tiles_per_item(1, 1, 0, 64, 0) == 0       # unsupported shape
