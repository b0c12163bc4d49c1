"""Head-parallel sharding: planner properties, a 2-rank gloo run on CPU, and shards run in sequence on one GPU."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from tiled_attention_09_gb300.shard import head_ranges, head_slice, local_range, shard_views


@pytest.mark.parametrize("heads,world,unit", [(24, 1, 1), (24, 2, 1), (24, 5, 1), (8, 8, 1), (3, 4, 1), (0, 2, 1),
                                             (97, 7, 1), (24, 5, 3), (24, 2, 12), (48, 7, 4), (8, 3, 8)])
def test_head_ranges_cover_disjoint_balanced(heads, world, unit):
    rs = head_ranges(heads, world, unit)
    assert len(rs) == world
    pos = 0
    for s, n in rs:
        assert s == pos and n >= 0 and s % unit == 0 and n % unit == 0
        pos += n
    assert pos == heads
    counts = [n // unit for _, n in rs]
    assert max(counts) - min(counts) <= 1


def test_head_ranges_reject_a_unit_that_does_not_divide():
    with pytest.raises(ValueError):
        head_ranges(24, 2, 5)


@pytest.mark.parametrize("H,Hkv,world", [(12, 12, 5), (12, 4, 5), (12, 1, 2), (8, 2, 3)])
def test_shard_views_hold_whole_kv_groups(H, Hkv, world):
    """Each rank's query heads read exactly its own K/V heads (h // G of the flattened order)."""
    B, N, d = 2, 8, 4
    q = torch.arange(B * H * N * d, dtype=torch.float32).reshape(B, H, N, d)
    k = -torch.arange(B * Hkv * N * d, dtype=torch.float32).reshape(B, Hkv, N, d)
    G = H // Hkv
    covered = []
    for r in range(world):
        sv = shard_views(q, k, k, r, world)
        s, n = sv["heads"]
        ks, kn = sv["kv_heads"]
        assert sv["q"].shape == (1, n, N, d) and sv["k"].shape == (1, kn, N, d) and kn * G == n
        for i in range(n):
            flat = s + i
            b, h = divmod(flat, H)
            assert torch.equal(sv["q"][0, i], q[b, h])
            assert torch.equal(sv["k"][0, i // G], k[b, h // G])  # the K/V head this query head reads
        covered += list(range(s, s + n))
    assert covered == list(range(B * H))


def test_shard_views_with_key_padding_take_whole_batches():
    B, H, Hkv, N, d = 5, 4, 2, 8, 4
    q = torch.randn(B, H, N, d)
    k = torch.randn(B, Hkv, N, d)
    kv_len = torch.tensor([8, 3, 5, 1, 0], dtype=torch.int32)
    seen = []
    for r in range(2):
        sv = shard_views(q, k, k, r, 2, kv_len=kv_len, extra=(q,))
        s, n = sv["heads"]
        b0, nb = s // H, n // H
        assert torch.equal(sv["q"], q[b0:b0 + nb]) and torch.equal(sv["k"], k[b0:b0 + nb])
        assert torch.equal(sv["kv_len"], kv_len[b0:b0 + nb]) and torch.equal(sv["extra"][0], q[b0:b0 + nb])
        seen += list(range(b0, b0 + nb))
    assert seen == list(range(B))


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


CASES = {  # name: (B, H, H_kv, N, d, causal, key counts or None)
    "plain": (2, 3, 3, 64, 16, True, None),
    "grouped": (2, 6, 2, 48, 16, True, None),
    "multi_query_padded": (3, 4, 1, 40, 8, False, (40, 17, 1)),
}


def _worker(rank, world, port, case, ret):
    import oracle
    from tiled_attention_09_gb300.inputs import Workload, make_inputs
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    B, H, Hkv, N, d, causal, lens = CASES[case]
    w = Workload(B, H, N, d, "bf16", causal)
    q, k, v, do = make_inputs(w)
    k, v = k[:, :Hkv].contiguous(), v[:, :Hkv].contiguous()
    kv_len = torch.tensor(lens, dtype=torch.int32) if lens else None
    sv = shard_views(q, k, v, rank, world, kv_len=kv_len, extra=(do,))
    f = lambda t: t.double().numpy()
    kl = sv["kv_len"].numpy() if kv_len is not None else None
    o, lse = oracle.attention_fwd(f(sv["q"]), f(sv["k"]), f(sv["v"]), w.scale, causal, kv_len=kl)
    dq, dk, dv = oracle.attention_bwd(f(sv["q"]), f(sv["k"]), f(sv["v"]), f(sv["extra"][0]), w.scale, causal,
                                      kv_len=kl)
    Dq = d * 2  # o, dq per query head; dk, dv per K/V head
    loc_q = torch.from_numpy(np.concatenate([o, dq], axis=-1).reshape(-1, N, Dq))
    loc_kv = torch.from_numpy(np.concatenate([dk, dv], axis=-1).reshape(-1, N, Dq))
    unit = H if kv_len is not None else H // Hkv
    rq = head_ranges(B * H, world, unit)
    nq = [n for _, n in rq]
    nkv = [n * Hkv // H for n in nq]
    out = {}
    for name, loc, counts in (("q", loc_q, nq), ("kv", loc_kv, nkv)):
        pad = torch.zeros(max(counts), N, Dq, dtype=loc.dtype)
        pad[:loc.shape[0]] = loc
        gathered = [torch.zeros_like(pad) for _ in range(world)]
        dist.all_gather(gathered, pad)
        out[name] = torch.cat([g[:n] for g, n in zip(gathered, counts)])
    if rank == 0:
        kl_all = kv_len.numpy() if kv_len is not None else None
        o_ref, _ = oracle.attention_fwd(f(q), f(k), f(v), w.scale, causal, kv_len=kl_all)
        dq_r, dk_r, dv_r = oracle.attention_bwd(f(q), f(k), f(v), f(do), w.scale, causal, kv_len=kl_all)
        ref_q = np.concatenate([o_ref, dq_r], axis=-1).reshape(B * H, N, Dq)
        ref_kv = np.concatenate([dk_r, dv_r], axis=-1).reshape(B * Hkv, N, Dq)
        ret["max_err"] = max(float(np.abs(out["q"].numpy() - ref_q).max()),
                             float(np.abs(out["kv"].numpy() - ref_kv).max()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("case", sorted(CASES))
def test_two_rank_gloo_sharded_oracle_equals_unsharded(case):
    """Two CPU ranks each take their head range (whole K/V groups; whole batches with key padding);
    the gathered O, dQ (per query head) and dK, dV (per K/V head) equal the whole-job result."""
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    ret = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, case, ret)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
        assert p.exitcode == 0
    assert ret["max_err"] == 0.0


@pytest.mark.gpu
def test_grouped_shards_in_sequence_on_one_gpu_equal_whole_job():
    """Grouped K/V heads (12 query heads on 4): each shard holds whole groups; O, LSE, dK, dV bitwise."""
    import tiled_attention_09_gb300 as fa
    from tiled_attention_09_gb300.inputs import Workload, make_inputs
    w = Workload(2, 12, 384, 128, "bf16", True)
    q, k, v, do = (t.cuda() for t in make_inputs(w))
    k, v = k[:, :4].contiguous(), v[:, :4].contiguous()
    o, lse, lo = fa.fwd(q, k, v, causal=True, residual=True)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=True, o_lo=lo)
    world = 3
    for rank in range(world):
        sv = shard_views(q, k, v, rank, world, extra=(do, o, lse, dq))
        do_s, o_ref, lse_ref, dq_ref = sv["extra"]
        ks, kn = sv["kv_heads"]
        o_s, lse_s, lo_s = fa.fwd(sv["q"], sv["k"], sv["v"], causal=True, residual=True)
        dq_s, dk_s, dv_s = fa.bwd(sv["q"], sv["k"], sv["v"], o_s, lse_s, do_s, causal=True, o_lo=lo_s)
        assert torch.equal(o_s, o_ref) and torch.equal(lse_s, lse_ref)
        assert torch.equal(dk_s, head_slice(dk, ks, kn)) and torch.equal(dv_s, head_slice(dv, ks, kn))
        assert (dq_s.float() - dq_ref.float()).abs().max().item() <= 1e-2 * dq.float().abs().max().item()


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
