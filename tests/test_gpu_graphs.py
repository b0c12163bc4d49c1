"""The C-ABI calls can be captured in a CUDA graph and replayed (GPU).

Nothing in fa_fwd_ex / fa_bwd / fa_decode synchronises or allocates on the compute path, so a step
(forward + backward, or a decode call) captured once replays with the same buffers; replays must give
the eager results bit for bit (dQ up to the order of its fp32 reductions).
"""
import pytest
import torch

import tiled_attention_09_gb300 as fa
from tiled_attention_09_gb300.inputs import DecodeWorkload, Workload, make_inputs, make_paged_inputs

pytestmark = pytest.mark.gpu


def test_forward_backward_step_replays_from_a_graph():
    w = Workload(2, 4, 640, 128, "bf16", True)
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    ws = torch.empty(fa.workspace_size(w.B, w.H, w.N, w.d), dtype=torch.uint8, device="cuda")
    o, lse, o_lo = (torch.empty_like(q), torch.empty((w.B, w.H, w.N), device="cuda"), torch.empty_like(q))
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def step():
        fa.fwd(q, k, v, causal=True, out=o, lse=lse, residual=True, o_lo=o_lo)
        fa.bwd(q, k, v, o, lse, do, causal=True, workspace=ws, dq=dq, dk=dk, dv=dv, o_lo=o_lo)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # eager, on the capture stream (first calls set kernel attributes)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (o, lse, dq, dk, dv)]
    for t in (o, lse, dq, dk, dv):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert fa.device_status()[0] == "FA_OK"
    for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), (o, lse, dq, dk, dv), ref):
        if name == "dQ":
            assert torch.allclose(a.float(), b.float(), atol=2e-2, rtol=0), name
        else:
            assert torch.equal(a, b), name


def test_decode_replays_from_a_graph():
    w = DecodeWorkload(4, 16, 4, 1, 128, 64, 24, (1500, 700, 64, 1))
    q, kp, vp, table, ctx = (t.cuda() for t in make_paged_inputs(w))
    ref_o, ref_lse = fa.decode(q, kp, vp, table, ctx, n_split=3)
    torch.cuda.synchronize()
    o, lse = torch.zeros_like(ref_o), torch.zeros_like(ref_lse)
    ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fa.decode(q, kp, vp, table, ctx, n_split=3, out=o, lse=lse, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    o.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.decode(q, kp, vp, table, ctx, n_split=3, out=o, lse=lse, workspace=ws)
    g.replay()
    torch.cuda.synchronize()
    assert fa.device_status()[0] == "FA_OK"
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
