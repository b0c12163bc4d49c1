"""Head-parallel sharding: planner properties, a 2-rank gloo run on CPU, and shards run in sequence on one GPU."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from tiled_attention_09_gb300.shard import head_ranges, head_slice, local_range


@pytest.mark.parametrize("heads,world", [(24, 1), (24, 2), (24, 5), (8, 8), (3, 4), (0, 2), (97, 7)])
def test_head_ranges_cover_disjoint_balanced(heads, world):
    rs = head_ranges(heads, world)
    assert len(rs) == world
    pos = 0
    for s, n in rs:
        assert s == pos and n >= 0
        pos += n
    assert pos == heads
    counts = [n for _, n in rs]
    assert max(counts) - min(counts) <= 1


def test_head_slice_is_a_view():
    t = torch.arange(2 * 3 * 4 * 2).reshape(2, 3, 4, 2)
    s = head_slice(t, 2, 3)
    assert s.shape == (1, 3, 4, 2)
    assert s.data_ptr() == t.data_ptr() + 2 * 4 * 2 * t.element_size()
    assert torch.equal(s[0, 0], t[0, 2]) and torch.equal(s[0, 2], t[1, 1])


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, ret):
    import oracle
    from tiled_attention_09_gb300.inputs import Workload, make_inputs
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = Workload(2, 3, 64, 16, "bf16", True)
    q, k, v, do = make_inputs(w)
    start, count = local_range(q, rank, world)
    sl = lambda t: head_slice(t, start, count).double().numpy()
    o, lse = oracle.attention_fwd(sl(q), sl(k), sl(v), w.scale, True)
    dq, dk, dv = oracle.attention_bwd(sl(q), sl(k), sl(v), sl(do), w.scale, True)
    local = torch.from_numpy(np.concatenate([o, dq, dk, dv], axis=-1)[0])  # [count, N, 4d]
    counts = [n for _, n in head_ranges(w.B * w.H, world)]
    pad = torch.zeros(max(counts), *local.shape[1:], dtype=local.dtype)
    pad[:count] = local
    gathered = [torch.zeros_like(pad) for _ in range(world)]
    dist.all_gather(gathered, pad)
    if rank == 0:
        full = torch.cat([g[:n] for g, n in zip(gathered, counts)])
        f = lambda t: t.double().numpy()
        o_ref, _ = oracle.attention_fwd(f(q), f(k), f(v), w.scale, True)
        g_ref = oracle.attention_bwd(f(q), f(k), f(v), f(do), w.scale, True)
        ref = np.concatenate([o_ref] + list(g_ref), axis=-1).reshape(w.B * w.H, w.N, -1)
        ret["max_err"] = float(np.abs(full.numpy() - ref).max())
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_gloo_sharded_oracle_equals_unsharded():
    """Two CPU ranks each take their head range; the gathered result equals the whole-job result."""
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    ret = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, ret)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
        assert p.exitcode == 0
    assert ret["max_err"] == 0.0


@pytest.mark.gpu
def test_shards_in_sequence_on_one_gpu_equal_whole_job():
    import tiled_attention_09_gb300 as fa
    from tiled_attention_09_gb300.inputs import Workload, make_inputs
    w = Workload(2, 3, 384, 128, "bf16", True)
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    o, lse, lo = fa.fwd(q, k, v, causal=True, residual=True)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=True, o_lo=lo)
    world = 4
    for rank in range(world):
        s, n = local_range(q, rank, world)
        sl = lambda t: head_slice(t, s, n)
        o_s, lse_s, lo_s = fa.fwd(sl(q), sl(k), sl(v), causal=True, residual=True)
        dq_s, dk_s, dv_s = fa.bwd(sl(q), sl(k), sl(v), o_s, lse_s, sl(do), causal=True, o_lo=lo_s)
        assert torch.equal(o_s, sl(o)) and torch.equal(lse_s, head_slice(lse, s, n))
        assert torch.equal(dk_s, sl(dk)) and torch.equal(dv_s, sl(dv))
        assert (dq_s.float() - sl(dq).float()).abs().max().item() <= 1e-2 * dq.float().abs().max().item()
