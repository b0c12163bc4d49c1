"""Benchmark: attention fwd+bwd TFLOP/s (bf16, causal) on GB300 through the libfa.so C ABI.

One step = the whole hot path over one batch of synthetic input: fa_fwd_ex (the
forward, also writing the rounding residual of O that the backward's D uses),
then fa_bwd's three phases (preprocess, main, dQ convert), on the workload
B=2, H=12, N=4096, d=128, bf16, causal (Q, K, V, dO iid N(0,1), seed 0).
FLOPs follow the metric's own count: forward 4*B*H*N^2*d halved when causal,
backward 2.5x that; value = 3.5*F_fwd / (t_fwd + t_bwd).

Timing: W untimed warm-up steps, then exactly K timed steps bracketed by a
barrier and torch.cuda.synchronize(); the L2 cache is flushed (a 256 MiB write, then a 256 MiB read)
before each step, outside the CUDA-event-timed interval of that step. A step is
timed between two events (fa_fwd_ex, fa_bwd through the C ABI); per-kernel times (kernels_ms and the
roofline's launch duration) come from a second pass of min(K, 50) steps with an
event between every two kernels. The max over ranks is reported; under torchrun
every rank runs the same workload on its own GPU (weak scaling, no data-path
collective), or with --shard heads its contiguous range of the job's B*H heads
(strong scaling: value = the whole job's FLOPs over the slowest rank's time;
heads are independent, so there is still no data-path collective).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--shard replicas|heads]
       python bench.py --decode | --sweep | --shape B,H,N,d | --oracle-timing | --sdpa
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# NVIDIA's published dense (no 2:4 sparsity) bf16 tensor-core peak of one GB300 GPU, TFLOP/s
PUBLISHED_DENSE_BF16_TFLOPS = 2250.0
METRIC = "attention fwd+bwd TFLOP/s (bf16, causal) and % of GB300 dense tensor peak"
_CSRC = "tiled_attention_09_gb300/csrc/"
# sources each timed kernel is built from: a recorded ncu traffic figure is used only while these are unchanged
KERNEL_SOURCES = {
    "fa_bwd_pipe_kernel": [_CSRC + f for f in ("fa_bwd_pipe.cuh", "fa_bwd_order.cuh", "fa_bwd_main.cuh", "ptx.cuh",
                                                "common.cuh")],
    "fa_fwd_kernel": [_CSRC + f for f in ("fa_fwd.cu", "ptx.cuh", "common.cuh")],
    "fa_bwd_dq_kernel": [_CSRC + f for f in ("fa_bwd_dq.cuh", "fa_bwd_main.cuh", "ptx.cuh", "common.cuh")],
}
ROOFLINE_KERNEL = "fa_bwd_pipe_kernel"  # the step's dominant kernel (d = 128 backward)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU work in the oracle's timed sample")
    ap.add_argument("--decode", action="store_true",
                    help="time paged decode attention on the decode points instead (one JSON line each)")
    ap.add_argument("--decode-point", type=int, default=-1, help="with --decode: only this point (0-based)")
    ap.add_argument("--decode-splits", default="0",
                    help="with --decode: comma-separated split counts to time at every point (0 = the library's choice)")
    ap.add_argument("--shape", default="", help="B,H,N,d: time this bf16 causal shape instead (profiling)")
    ap.add_argument("--oracle-timing", action="store_true",
                    help="time the fp64 CPU oracle on the host cores: the small, pages and causal-4k workloads in "
                         "full (forward and backward apart, the small one also single-threaded), the 32k one on "
                         "sampled rows; one JSON line each, no GPU")
    ap.add_argument("--oracle-single", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--sdpa", action="store_true",
                    help="context only: time torch's scaled_dot_product_attention (each backend that runs) "
                         "forward+backward on the headline workload, one JSON line")
    ap.add_argument("--dq-mode", default="default", choices=["default", "accumulate", "separate"],
                    help="how the backward forms dQ: the library's choice, fp32 partial tiles reduced into the "
                         "workspace, or the separate query-major pass (d = 64, 128)")
    ap.add_argument("--shard", default="replicas", choices=["replicas", "heads"],
                    help="under torchrun: every rank runs the whole workload (replicas, weak scaling) or its "
                         "contiguous range of the job's B*H heads (heads, strong scaling, no data-path collective)")
    ap.add_argument("--sweep-bf16", action="store_true", help="with --sweep: bf16 points only")
    ap.add_argument("--split-sweep", action="store_true",
                    help="time the forward on grids with few heads and long rows at 1, 2, 4 and 8 key ranges per "
                         "query block and at the library's choice; one JSON line per shape")
    ap.add_argument("--sweep", action="store_true",
                    help="time every sweep point (B2 H12, d 64/128/256, N 512-16384, both dtypes and masks) "
                         "instead of the headline step; one JSON line per point")
    return ap.parse_args()


def dq_separate(L, mode, d, causal):
    """Whether the backward forms dQ with the separate pass for this mode, head dimension and mask."""
    opt = _lib_options(mode)
    return bool(L.fa_bwd_uses_dq_pass(d, int(causal), ctypes.byref(opt)))


def _lib_options(mode):
    import tiled_attention_09_gb300 as fa
    from tiled_attention_09_gb300 import _lib
    return _lib.FAOptions(0, None, 0, fa.DQ_MODES[mode])


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    for p in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernel source."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            d = json.load(f)
        e = d.get(kernel)
        if e and e.get("source_hash") == kernel_source_hash(kernel):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, flag in zip(names, parts[5:9]):
                if flag.lower() in ("active", "1", "yes"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def _visible(w, r0, r1):
    """Number of (query, key) pairs the metric counts for query rows [r0, r1) of one head."""
    if w.causal:
        return (r1 * (r1 + 1) - r0 * (r0 + 1)) // 2
    return (r1 - r0) * w.N


class OracleSampler:
    """Times the fp64 oracle, as it stands, on row blocks of the workload (fwd + bwd of those rows).

    A row block of one (b, h) head is the definition restricted to query rows
    [r0, r1): O, LSE and dQ of those rows and their shares of dK and dV. Its
    useful FLOPs are 3.5 * 4 * d * (visible (query, key) pairs), the metric's
    own count restricted to the block.
    """

    def __init__(self, w):
        from tiled_attention_09_gb300.inputs import make_inputs
        self.w = w
        self.q, self.k, self.v, self.do = make_inputs(w)
        self.cursor = 0  # (head, row) position, walks the workload in order

    def run(self, rows):
        import oracle
        w = self.w
        head, r0 = divmod(self.cursor, w.N)
        head %= w.B * w.H
        r1 = min(w.N, r0 + rows)
        b, h = divmod(head, w.H)
        sl = lambda t: t[b:b + 1, h:h + 1].double().numpy()
        q, k, v, do = sl(self.q), sl(self.k), sl(self.v), sl(self.do)
        t0 = time.perf_counter()
        oracle.attention_row_block(q, k, v, do, w.scale, w.causal, 0, 0, r0, r1)
        dt = time.perf_counter() - t0
        self.cursor = head * w.N + r1 if r1 < w.N else (head + 1) * w.N
        return 3.5 * 4 * w.d * _visible(w, r0, r1), dt, (b, h, r0, r1)


def oracle_baseline(w, budget_s=12.0, block=512):
    """cpu_baseline: the oracle on consecutive row blocks until about budget_s of CPU work."""
    smp = OracleSampler(w)
    smp.run(64)  # page in, start BLAS threads
    smp.cursor = 0
    flops = secs = 0.0
    blocks = []
    while secs < budget_s:
        f, dt, where = smp.run(block)
        flops += f
        secs += dt
        blocks.append(where)
    first, last = blocks[0], blocks[-1]
    sample = (f"{len(blocks)} row blocks of {block} query rows, (b,h,rows) {first[:2]}:{first[2]} .. "
              f"{last[:2]}:{last[3]} of {w.name()}, fwd+bwd of those rows, {secs:.1f} s")
    return flops / secs / 1e12, sample


def cpu_cores():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args):
    """Reference arm: the fp64 CPU oracle on a bounded sample of the same workload per step."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if int(os.environ.get("RANK", "0")) != 0:
        return
    w = bench_workload(args)
    smp = OracleSampler(w)
    smp.run(64)
    # size the per-step sample so warm-up + timed steps stay within ~2.5 minutes
    f, dt, _ = smp.run(256)
    per_step = min(3.0, 150.0 / (args.steps + args.warmup))
    rows = int(max(64, min(w.N, 256 * per_step / max(dt, 1e-3))) // 64 * 64)
    smp.cursor = 0
    for _ in range(args.warmup):
        smp.run(rows)
    flops = secs = 0.0
    for _ in range(args.steps):
        f, dt, _ = smp.run(rows)
        flops += f
        secs += dt
    value = flops / secs / 1e12
    cores = cpu_cores()
    sample = f"{rows} query rows of one (b,h) head of {w.name()} per step (fwd+bwd of those rows), fp64 numpy oracle"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name(), "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": True,
                   "sample": f"{rows} query rows per step"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


class L2Flush:
    """Evicts the L2 cache between timed steps: a write of a buffer larger than L2, then a read of a second
    one, so that the dirty lines the write leaves behind are written back here, outside the timed interval,
    and the step starts from a cold, clean L2."""

    def __init__(self, torch, dev, mib=256):
        n = mib * 1024 * 1024 // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.ones(n, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)
        self.torch = torch

    def __call__(self):
        self.w.zero_()
        self.torch.sum(self.r, dim=0, out=self.sink)


def bench_workload(args):
    """The timed workload: B2 H12 N4096 d128 bf16 causal, or --shape B,H,N,d (bf16, causal) for profiling
    other sizes with the same step."""
    from tiled_attention_09_gb300.inputs import CAUSAL_4K, Workload
    if not getattr(args, "shape", ""):
        return CAUSAL_4K
    B, H, N, d = (int(x) for x in args.shape.split(","))
    return Workload(B, H, N, d, "bf16", True)


def measure_ex2_rate(torch, L, dev, reps=4096):
    """Exponentials per second of the whole GPU (fa_selftest_ex2_rate on 2 CTAs per SM, median of 5 timed
    launches after one warm-up): the peak of the softmax's secondary roofline."""
    blocks = 2 * torch.cuda.get_device_properties(dev).multi_processor_count
    sink = torch.zeros(blocks, dtype=torch.float32, device=dev)
    sp = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    times = []
    for i in range(6):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        if L.fa_selftest_ex2_rate(reps, blocks, ctypes.c_void_p(sink.data_ptr()), sp) != 0:
            return None
        e1.record()
        torch.cuda.synchronize()
        if i > 0:
            times.append(e0.elapsed_time(e1) / 1e3)
    return blocks * 512 * 8 * reps / statistics.median(times)


def run_native(args):
    import torch
    import tiled_attention_09_gb300 as fa
    from tiled_attention_09_gb300 import _lib
    from tiled_attention_09_gb300.inputs import make_inputs

    world, rank, local, dist = dist_setup(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = bench_workload(args)
    roof_kernel = ROOFLINE_KERNEL if w.d != 256 else "fa_bwd_d256_kernel"
    B, H, N, d = w.B, w.H, w.N, w.d
    sharded = args.shard == "heads" and world > 1
    job_heads = B * H
    if sharded:  # this rank's contiguous range of the job's heads, as a B' = 1, H' = count problem
        from tiled_attention_09_gb300.shard import head_ranges
        h0, nh = head_ranges(job_heads, world)[rank]
        if nh == 0:
            raise SystemExit(f"rank {rank}: no heads left for this rank ({job_heads} heads, {world} ranks)")
    F = w.fwd_flops() * ((nh / job_heads) if sharded else 1.0)  # forward FLOPs of this rank's share
    step_flops = 3.5 * F
    job_step_flops = 3.5 * w.fwd_flops() if sharded else world * step_flops

    # CPU baseline first (rank 0, N=1 only), before the GPU work starts
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        val, sample = oracle_baseline(w, budget_s=args.cpu_seconds)
        cpu = {"value": val, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle", "sample": sample}

    L = _lib.load()
    q, k, v, do = make_inputs(w)
    if sharded:
        from tiled_attention_09_gb300.shard import head_slice
        q, k, v, do = (head_slice(t, h0, nh).contiguous() for t in (q, k, v, do))
        B, H = 1, nh
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws_bytes = int(L.fa_bwd_workspace_size(B, H, N, d))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    scale = w.scale
    DT = _lib.FA_BF16

    opt = _lib.FAOptions(0, None, 0, fa.DQ_MODES[args.dq_mode])
    optp = ctypes.byref(opt)
    sep = dq_separate(L, args.dq_mode, d, True)

    def launch(ptrs, evs=None):
        """One step through the public entry points (fa_fwd_ex, fa_bwd_opt); evs: [start, end] events or None."""
        qp, kp, vp, op, lp, dop, dqp, dkp, dvp, lop = ptrs
        if evs:
            evs[0].record(stream)
        _lib.check("fa_fwd_ex", L.fa_fwd_ex(qp, kp, vp, op, lp, lop, B, H, N, d, scale, 1, DT, sp))
        _lib.check("fa_bwd_opt", L.fa_bwd_opt(qp, kp, vp, op, dop, lp, dqp, dkp, dvp, lop, ws.data_ptr(), ws_bytes, B,
                                              H, N, d, scale, 1, DT, optp, sp))
        if evs:
            evs[1].record(stream)

    def launch_phases(ptrs, evs):
        """The same step as its four kernels with an event between each (per-kernel times; an event between
        two kernels can keep the second from starting early, so this pass is not the step time). The last
        kernel is the dQ conversion, or the separate dQ pass."""
        qp, kp, vp, op, lp, dop, dqp, dkp, dvp, lop = ptrs
        evs[0].record(stream)
        _lib.check("fa_fwd_ex", L.fa_fwd_ex(qp, kp, vp, op, lp, lop, B, H, N, d, scale, 1, DT, sp))
        evs[1].record(stream)
        _lib.check("pre", L.fa_bwd_preprocess_opt(op, lop, dop, lp, ws.data_ptr(), ws_bytes, B, H, N, d, 1, DT, optp,
                                                  sp))
        evs[2].record(stream)
        _lib.check("main", L.fa_bwd_main_opt(qp, kp, vp, dop, dkp, dvp, None, ws.data_ptr(), ws_bytes, B, H, N, d,
                                             scale, 1, DT, optp, sp))
        evs[3].record(stream)
        if sep:
            _lib.check("dq", L.fa_bwd_dq_pass(qp, kp, vp, dop, dqp, ws.data_ptr(), ws_bytes, B, H, N, d, scale, 1, DT,
                                              optp, sp))
        else:
            _lib.check("conv", L.fa_bwd_dq_convert(dqp, ws.data_ptr(), ws_bytes, B, H, N, d, scale, DT, sp))
        evs[4].record(stream)

    o_lo = torch.empty_like(qd)
    dptrs = [t.data_ptr() for t in (qd, kd, vd, o, lse, dod, dq, dk, dv, o_lo)]
    for _ in range(args.warmup):
        flush()
        launch(dptrs)
    torch.cuda.synchronize()
    code, info = fa.device_status(stream.cuda_stream)
    if code != "FA_OK":
        raise RuntimeError(f"device status after warm-up: {code} {info}")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    K2 = max(3, min(args.steps, 50))
    pevs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K2)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.25)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    for s in range(args.steps):
        flush()
        launch(dptrs, evs[s])
    torch.cuda.synchronize()
    for s in range(K2):
        flush()
        launch_phases(dptrs, pevs[s])
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    code, info = fa.device_status(stream.cuda_stream)
    if code != "FA_OK":
        raise RuntimeError(f"device status after timed steps: {code} {info}")
    total = sum(e[0].elapsed_time(e[1]) for e in evs) / 1e3
    # per-kernel averages from the phase pass
    t_fwd = sum(e[0].elapsed_time(e[1]) for e in pevs) / 1e3 / K2
    t_pre = sum(e[1].elapsed_time(e[2]) for e in pevs) / 1e3 / K2
    t_main = sum(e[2].elapsed_time(e[3]) for e in pevs) / 1e3 / K2
    t_conv = sum(e[3].elapsed_time(e[4]) for e in pevs) / 1e3 / K2
    if dist:
        tt = torch.tensor([total], device=dev, dtype=torch.float64)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total = tt.item()
    K = args.steps
    value = job_step_flops * K / total / 1e12

    # ---- end to end through the public API with host buffers (pinned), copies inside the timed region.
    # Every step copies its own Q, K, V, dO in and its O, LSE, dQ, dK, dV out; the copies of neighbouring
    # steps overlap the current step's kernels (an input stream, the compute stream, an output stream, two
    # sets of device buffers), as a serving or training loop would run them.
    hq, hk, hv, hdo = (t.pin_memory() for t in (q, k, v, do))
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    dsets, hsets = [], []
    for b in range(2):
        ins = [torch.empty_like(t) for t in (qd, kd, vd, dod)]
        outs = [torch.empty_like(qd), torch.empty((B, H, N), device=dev, dtype=torch.float32), torch.empty_like(qd),
                torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)]  # o, lse, o_lo, dq, dk, dv
        dsets.append((ins, outs))
        hsets.append([torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (outs[0], outs[1], outs[3], outs[4],
                                                                                outs[5])])
    d2h = sum(t.numel() * t.element_size() for t in hsets[0])
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    started = [False, False]

    def e2e_step(i):
        b = i % 2
        (qi, ki, vi, doi), (o_, lse_, lo_, dq_, dk_, dv_) = dsets[b]
        with torch.cuda.stream(s_in):
            if started[b]:
                s_in.wait_event(comp_done[b])  # step i - 2 has finished reading this input set
            for src, dst in ((hq, qi), (hk, ki), (hv, vi), (hdo, doi)):
                dst.copy_(src, non_blocking=True)
            in_done[b].record(s_in)
        stream.wait_event(in_done[b])
        if started[b]:
            stream.wait_event(out_done[b])  # step i - 2's outputs have been read back
        fa.fwd(qi, ki, vi, causal=True, out=o_, lse=lse_, residual=True, o_lo=lo_)
        fa.bwd(qi, ki, vi, o_, lse_, doi, causal=True, workspace=ws, dq=dq_, dk=dk_, dv=dv_, o_lo=lo_,
               dq_mode=args.dq_mode)
        comp_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            for src, dst in zip((o_, lse_, dq_, dk_, dv_), hsets[b]):
                dst.copy_(src, non_blocking=True)
            out_done[b].record(s_out)
        started[b] = True

    for i in range(max(3, args.warmup // 2)):
        e2e_step(i)
    torch.cuda.synchronize()
    started[0] = started[1] = False
    e2e_steps = max(3, min(K, 50))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    s_in.wait_event(ev0)
    s_out.wait_event(ev0)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(s_in)
    stream.wait_stream(s_out)
    ev1.record(stream)
    torch.cuda.synchronize()
    t_e2e = ev0.elapsed_time(ev1) / 1e3
    if dist:
        tt = torch.tensor([t_e2e], device=dev, dtype=torch.float64)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        t_e2e = tt.item()
    e2e_value = job_step_flops * e2e_steps / t_e2e / 1e12

    # The same copies alone, in and out at once on the same two streams: the time the host link needs per
    # step, so that e2e can be read against max(this, the device step time).
    def copies_only(b):
        (qi, ki, vi, doi), (o_, lse_, lo_, dq_, dk_, dv_) = dsets[b]
        with torch.cuda.stream(s_in):
            for src, dst in ((hq, qi), (hk, ki), (hv, vi), (hdo, doi)):
                dst.copy_(src, non_blocking=True)
        with torch.cuda.stream(s_out):
            for src, dst in zip((o_, lse_, dq_, dk_, dv_), hsets[b]):
                dst.copy_(src, non_blocking=True)

    copies_only(0)
    torch.cuda.synchronize()
    n_copy = 10
    ev0.record(stream)
    s_in.wait_event(ev0)
    s_out.wait_event(ev0)
    for i in range(n_copy):
        copies_only(i % 2)
    stream.wait_stream(s_in)
    stream.wait_stream(s_out)
    ev1.record(stream)
    torch.cuda.synchronize()
    t_copy = ev0.elapsed_time(ev1) / 1e3 / n_copy
    t_e2e_step = t_e2e / e2e_steps
    e2e_bound = max(t_copy, total / K)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    main_avg = t_main
    main_flops = 2.5 * F
    achieved = main_flops / main_avg / 1e12
    peak = peaks["bf16_tflops"]
    fwd_avg = t_fwd
    traffic = None if args.shape else recorded_traffic(roof_kernel)  # recorded for the bench workload only
    # secondary roofline of the softmax: exponentials (B*H*N^2, halved when causal: the FLOP count's
    # convention) per second in the forward and in the backward main kernel (which rebuilds P)
    ex2_peak = measure_ex2_rate(torch, L, dev)
    exps = B * H * N * N / 2
    exp_roof = None
    if ex2_peak:
        exp_roof = {"unit": "exp/s", "peak": ex2_peak, "peak_source": "measured (fa_selftest_ex2_rate)",
                    "fa_fwd_kernel": {"achieved": exps / fwd_avg, "frac": exps / fwd_avg / ex2_peak},
                    roof_kernel: {"achieved": exps / main_avg, "frac": exps / main_avg / ex2_peak}}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / K, "higher_is_better": True, "scaling": "strong" if sharded else "weak",
        "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name(), "B": B, "H": H, "N": N, "d": d, "causal": True, "seed": 0,
                   "dq": "separate pass" if sep else "accumulated (global reductions from registers)",
                   "l2": "flushed before every step (256 MiB write, then a 256 MiB read of another buffer so the write-back is not charged to the step; outside the timed interval)",
                   "timing": "value: whole step between two events; kernels_ms/roofline: a second pass of "
                             f"{K2} steps with events between kernels",
                   "parallelism": (f"heads: {job_heads} heads in contiguous ranges over {world} rank(s), no "
                                   "data-path collective" if sharded else f"weak: {world} independent replica(s)")},
        "pct_of_peak": value / (world * peak), "peak_tflops": peak, "peak_source": f"{peak_src} (bf16 burst)",
        "pct_of_published_peak": value / (world * PUBLISHED_DENSE_BF16_TFLOPS),
        "published_peak_tflops": PUBLISHED_DENSE_BF16_TFLOPS,
        "published_peak_source": "NVIDIA's GB300 dense bf16 tensor-core figure, 2.25 PFLOP/s per GPU (its "
                                 "larger per-system figures assume 2:4 sparsity)",
        "kernels_ms": {"fa_fwd_kernel": 1e3 * fwd_avg, "fa_bwd_preprocess_kernel": 1e3 * t_pre,
                       roof_kernel: 1e3 * main_avg,
                       ("fa_bwd_dq_kernel" if sep else "fa_bwd_dq_convert_kernel"): 1e3 * t_conv},
        "fwd_tflops": F / fwd_avg / 1e12,
        "bwd_tflops": 2.5 * F / (t_pre + t_main + t_conv) / 1e12,
        "roofline": {"kernel": roof_kernel, "bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_src} bf16 burst"},
        "exp_roofline": exp_roof,
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": 1e3 * t_e2e_step,
                "copies_alone_ms_per_step": 1e3 * t_copy,
                "h2d_gbs_concurrent": h2d / t_copy / 1e9, "d2h_gbs_concurrent": d2h / t_copy / 1e9,
                "bound": "host copies" if t_copy > total / K else "device step",
                "frac_of_bound": e2e_bound / t_e2e_step},
        "gpu_launches": 4 * K,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_sweep(args):
    """One JSON line per sweep point: forward and forward+backward, each timed between two events on the
    launching stream (L2 flushed before every step), TFLOP/s, % of the measured bf16 peak, and % of the
    attainable min(peak, HBM bandwidth x algorithmic intensity) with the algorithmic bytes per head
    8Nd + 4N (forward) and 16Nd + 8N more (backward), at 2 bytes per element and 4 per LSE / D value.
    For N <= 2048 also fwd_bwd_graph: the same step replayed from a CUDA graph."""
    import torch
    import tiled_attention_09_gb300 as fa
    from tiled_attention_09_gb300.inputs import Workload, cast_inputs, make_inputs_fp32
    from tiled_attention_09_gb300 import _lib
    L = _lib.load()
    peaks, peak_src = load_peaks()
    peak, bw = peaks["bf16_tflops"], peaks["hbm_gbs"]
    dev = torch.device("cuda", 0)
    flush = L2Flush(torch, dev)
    steps, warmup = max(3, min(args.steps, 20)), max(3, args.warmup)
    dtypes = ("bf16",) if args.sweep_bf16 else ("bf16", "fp16")
    for d in (64, 128, 256):
        for N in (512, 1024, 2048, 4096, 8192, 16384):
            fp32 = make_inputs_fp32(Workload(2, 12, N, d, "bf16", True))
            for dtype in dtypes:
                for causal in (True, False):
                    w = Workload(2, 12, N, d, dtype, causal)
                    q, k, v, do = (t.to(dev) for t in cast_inputs(w, fp32))
                    o, lse, o_lo = fa.fwd(q, k, v, causal=causal, residual=True)
                    ws = torch.empty(fa.workspace_size(w.B, w.H, N, d), dtype=torch.uint8, device=dev)
                    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

                    def fwd():
                        fa.fwd(q, k, v, causal=causal, out=o, lse=lse, residual=True, o_lo=o_lo)

                    # the split-key forward where the library would split this grid (kv_splits = 0)
                    n_split = int(L.fa_fwd_kv_splits(w.B, w.H, N, d, int(causal)))
                    fws = (torch.empty(int(L.fa_fwd_workspace_size(w.B, w.H, N, d, n_split)), dtype=torch.uint8,
                                       device=dev) if n_split > 1 else None)

                    def fwd_split():
                        fa.fwd(q, k, v, causal=causal, out=o, lse=lse, residual=True, o_lo=o_lo, kv_splits=n_split,
                               workspace=fws)

                    def step(mode):
                        fwd()
                        fa.bwd(q, k, v, o, lse, do, causal=causal, workspace=ws, dq=dq, dk=dk, dv=dv, o_lo=o_lo,
                               dq_mode=mode)

                    # both ways of forming dQ where the separate pass exists (d = 64, 128); the point's
                    # fwd_bwd is the library's default choice
                    modes = ("accumulate", "separate") if d in (64, 128) else ("accumulate",)
                    default = "separate" if dq_separate(L, "default", d, causal) else "accumulate"
                    times = {}
                    fns = [("fwd", fwd)] + [(f"fwd_bwd_{m}", (lambda m=m: step(m))) for m in modes]
                    if n_split > 1:
                        fns.append(("fwd_split", fwd_split))
                    for name, fn in fns:
                        for _ in range(warmup):
                            flush()
                            fn()
                        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                               for _ in range(steps)]
                        for e0, e1 in evs:
                            flush()
                            e0.record()
                            fn()
                            e1.record()
                        torch.cuda.synchronize()
                        times[name] = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3
                    if N <= 2048:
                        # short rows are launch-bound: the same step replayed from a CUDA graph (its four
                        # kernels captured once), timed the same way, shows what the launches cost
                        side = torch.cuda.Stream()
                        side.wait_stream(torch.cuda.current_stream())
                        with torch.cuda.stream(side):
                            step(default)
                        torch.cuda.current_stream().wait_stream(side)
                        graph = torch.cuda.CUDAGraph()
                        with torch.cuda.graph(graph):
                            step(default)
                        for _ in range(warmup):
                            flush()
                            graph.replay()
                        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                               for _ in range(steps)]
                        for e0, e1 in evs:
                            flush()
                            e0.record()
                            graph.replay()
                            e1.record()
                        torch.cuda.synchronize()
                        times["fwd_bwd_graph"] = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3
                        del graph
                    code, info = fa.device_status()
                    if code != "FA_OK":
                        raise RuntimeError(f"{w.name()}: {code} {info}")
                    F = w.fwd_flops()
                    heads = w.B * w.H
                    bytes_fwd = heads * (4 * N * d * 2 + 4 * N)  # Q, K, V in, O out; LSE
                    bytes_bwd = heads * (8 * N * d * 2 + 8 * N)  # Q, K, V, dO in; dQ, dK, dV out (+ O); LSE, D
                    line = {"point": w.name(), "N": N, "d": d, "dtype": dtype, "causal": causal, "dq_default": default}
                    times["fwd_bwd"] = times[f"fwd_bwd_{default}"]
                    line["fwd_kv_splits"] = n_split
                    for name, flops, nbytes in [("fwd", F, bytes_fwd)] + [
                            (f"fwd_bwd{x}", 3.5 * F, bytes_fwd + bytes_bwd)
                            for x in [""] + [f"_{m}" for m in modes] + (["_graph"] if N <= 2048 else [])] + (
                            [("fwd_split", F, bytes_fwd)] if n_split > 1 else []):
                        tf = flops / times[name] / 1e12
                        attainable = min(peak, bw * 1e9 * flops / nbytes / 1e12)
                        line[name] = {"ms": 1e3 * times[name], "tflops": tf, "pct_of_peak": tf / peak,
                                      "pct_of_attainable": tf / attainable}
                    line["peak_tflops"] = peak
                    line["peak_source"] = peak_src
                    print(json.dumps(line), flush=True)
                    del q, k, v, do, o, lse, o_lo, ws, dq, dk, dv, fws
            torch.cuda.empty_cache()


SPLIT_POINTS = [  # (B, H, N, d, causal): few query blocks, each with a long key range
    (1, 1, 4096, 128, True), (1, 1, 8192, 128, True), (1, 1, 16384, 128, True), (1, 1, 32768, 128, True),
    (1, 2, 16384, 128, True), (1, 1, 8192, 128, False), (1, 4, 4096, 128, True), (1, 1, 16384, 64, True),
    (1, 1, 8192, 256, True), (2, 2, 8192, 128, True), (2, 12, 4096, 128, True),
]


def run_split_sweep(args):
    """One JSON line per SPLIT_POINTS shape (bf16): the forward's median time at kv_splits 1, 2, 4, 8 (each
    between two events on the launching stream, L2 flushed before every call) and the library's choice."""
    import torch
    import tiled_attention_09_gb300 as fa
    from tiled_attention_09_gb300.inputs import Workload, make_inputs
    from tiled_attention_09_gb300 import _lib
    L = _lib.load()
    dev = torch.device("cuda", 0)
    flush = L2Flush(torch, dev)
    steps, warmup = max(3, min(args.steps, 20)), max(3, args.warmup)
    for B, H, N, d, causal in SPLIT_POINTS:
        w = Workload(B, H, N, d, "bf16", causal)
        q, k, v, _ = (t.to(dev) for t in make_inputs(w))
        o, lse = torch.empty_like(q), torch.empty(B, H, N, device=dev)
        us = {}
        for n_split in (1, 2, 4, 8):
            ws = (torch.empty(int(L.fa_fwd_workspace_size(B, H, N, d, n_split)), dtype=torch.uint8, device=dev)
                  if n_split > 1 else None)

            def call():
                fa.fwd(q, k, v, causal=causal, out=o, lse=lse, kv_splits=n_split, workspace=ws)

            for _ in range(warmup):
                flush()
                call()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
            for e0, e1 in evs:
                flush()
                e0.record()
                call()
                e1.record()
            torch.cuda.synchronize()
            us[n_split] = 1e3 * statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)
        code, info = fa.device_status()
        if code != "FA_OK":
            raise RuntimeError(f"{w.name()}: {code} {info}")
        best = min(us, key=us.get)
        choice = int(L.fa_fwd_kv_splits(B, H, N, d, int(causal)))
        print(json.dumps({"point": w.name(), "us": us, "fastest": best, "library_choice": choice,
                          "choice_vs_fastest": us[choice] / us[best] if choice in us else None,
                          "tflops_plain": w.fwd_flops() / us[1] / 1e6,
                          "tflops_choice": w.fwd_flops() / us[choice] / 1e6 if choice in us else None}), flush=True)
        del q, k, v, o, lse
        torch.cuda.empty_cache()


DECODE_POINTS = [  # (B, H, Hkv, Mq, d, page_size, ctx)
    (16, 32, 8, 1, 128, 64, 8192),
    (1, 32, 8, 1, 128, 64, 65536),
    (64, 8, 1, 4, 128, 16, 4096),
    (32, 16, 2, 1, 64, 128, 8192),
    (8, 64, 8, 2, 128, 256, 16384),
    (8, 32, 8, 1, 256, 64, 8192),
]


def run_decode(args):
    """One JSON line per paged-decode point: fa_decode (split kernel + merge) timed between two events on the
    launching stream, L2 flushed before every step, median of the timed steps. The C function is called
    with prepared arguments (no Python-side checks or allocation), so the host enqueues it while the L2
    flush still runs and the events time the device work. HBM-bound: the algorithmic bytes are the
    sequences' K and V (2 * keys * Hkv * d * 2) plus q in and O out; the fraction divides by the measured
    copy bandwidth."""
    import torch
    import tiled_attention_09_gb300 as fa
    from tiled_attention_09_gb300 import _lib
    from tiled_attention_09_gb300.inputs import DecodeWorkload, make_paged_inputs
    peaks, peak_src = load_peaks()
    bw = peaks["hbm_gbs"]
    dev = torch.device("cuda", 0)
    flush = L2Flush(torch, dev)  # ~80 us of device work: longer than the host takes to enqueue the call
    steps, warmup = max(3, min(args.steps, 30)), max(3, args.warmup)
    points = DECODE_POINTS if args.decode_point < 0 else [DECODE_POINTS[args.decode_point]]
    split_list = [int(x) for x in args.decode_splits.split(",")]
    for B, H, Hkv, Mq, d, ps, ctx in points:
        w = DecodeWorkload(B, H, Hkv, Mq, d, ps, ctx // ps, (ctx,) * B, spare=0, poison=False)
        q, kp, vp, table, cl = (t.to(dev) for t in make_paged_inputs(w))
        o, lse = fa.decode(q, kp, vp, table, cl)
        L = _lib.load()
        for forced in split_list:
            n_split = forced if forced > 0 else fa.decode_splits(B, Hkv, d, ps, w.max_pages)
            ws = torch.empty(int(L.fa_decode_workspace_size(B, H, Hkv, Mq, d, ps, w.max_pages, n_split)),
                             dtype=torch.uint8, device=dev)
            stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
            cargs = (q.data_ptr(), kp.data_ptr(), vp.data_ptr(), table.data_ptr(), cl.data_ptr(), o.data_ptr(),
                     lse.data_ptr(), ws.data_ptr(), ws.numel(), B, H, Hkv, Mq, d, ps, w.n_pages, w.max_pages, n_split,
                     w.scale, 0, 1, stream)

            def call():
                rc = L.fa_decode(*cargs)
                if rc != 0:
                    raise RuntimeError(f"fa_decode returned {rc}")

            for _ in range(warmup):
                flush()
                call()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
            host = []
            for e0, e1 in evs:
                flush()
                e0.record()
                h0 = time.perf_counter()
                call()
                host.append(time.perf_counter() - h0)
                e1.record()
            torch.cuda.synchronize()
            code, info = fa.device_status()
            if code != "FA_OK":
                raise RuntimeError(f"{w.name()}: {code} {info}")
            t = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3
            nbytes = w.kv_bytes() + 2 * q.numel() * 2 + 4 * lse.numel()
            gbs = nbytes / t / 1e9
            print(json.dumps({"point": w.name(), "us": 1e6 * t, "host_us": 1e6 * statistics.median(host),
                              "n_split": n_split, "library_choice": forced <= 0, "ctas": B * Hkv * n_split,
                              "algorithmic_bytes": nbytes, "gbs": gbs, "frac_of_hbm": gbs / bw, "hbm_peak_gbs": bw,
                              "peak_source": peak_src, "tflops": w.flops() / t / 1e12}), flush=True)
            del ws
        del q, kp, vp, table, cl, o, lse
        torch.cuda.empty_cache()


def cpu_model():
    """The host CPU's name from /proc/cpuinfo (x86 "model name"; Arm "CPU part" code), else the machine type."""
    import platform
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read().splitlines()
        for key in ("model name", "Model", "CPU part"):
            for line in info:
                if line.split(":")[0].strip() == key:
                    return f"{key}: {line.split(':', 1)[1].strip()} ({platform.machine()})"
    except OSError:
        pass
    return platform.machine()


def run_oracle_timing(args):
    """The fp64 oracle as it stands (numpy, BLAS threads = host cores), timed on the host: the small
    (B1 H2 N256 d64), pages (B2 H12 N1024 d64) and causal 4k (B2 H12 N4096 d128) workloads in full,
    forward and backward timed apart; the small one again with one BLAS thread (a child process, since
    the thread count is fixed when numpy loads); the 32k workload (B1 H8 N32768 d128) on the sampled
    query rows the parity tests check (O, LSE and dQ of those rows). GFLOP/s use the metric's count
    (forward 4BHN^2d, halved when causal; backward 2.5x), or for sampled rows 8 d (visible keys) a row."""
    import numpy as np
    import oracle
    from tiled_attention_09_gb300.inputs import CAUSAL_4K, LONG_32K, PAGES_SHAPE, SMALL, make_inputs, sample_rows
    cores, cpu = cpu_cores(), cpu_model()
    f64 = lambda t: t.double().numpy()

    def full(label, w):
        q, k, v, do = (f64(t) for t in make_inputs(w))
        t0 = time.perf_counter()
        oracle.attention_fwd(q, k, v, w.scale, w.causal)
        t_f = time.perf_counter() - t0
        t0 = time.perf_counter()
        oracle.attention_bwd(q, k, v, do, w.scale, w.causal)
        t_b = time.perf_counter() - t0
        F = w.fwd_flops()
        print(json.dumps({"oracle_timing": label, "workload": w.name(), "mode": "full", "threads": cores,
                          "cpu": cpu, "fwd_s": t_f, "bwd_s": t_b, "fwd_gflops": F / t_f / 1e9,
                          "bwd_gflops": 2.5 * F / t_b / 1e9}), flush=True)

    if args.oracle_single:
        full("small, 1 thread", SMALL)
        return
    for label, w in (("small", SMALL), ("pages", PAGES_SHAPE), ("causal 4k", CAUSAL_4K)):
        full(label, w)
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-timing", "--oracle-single"], env=env,
                   check=True)
    w = LONG_32K
    q, k, v, do = (f64(t) for t in make_inputs(w))
    rows = np.asarray(sample_rows(w.N))
    t0 = time.perf_counter()
    oracle.attention_rows(q, k, v, do, w.scale, w.causal, rows)
    dt = time.perf_counter() - t0
    visible = (rows + 1).sum() if w.causal else len(rows) * w.N
    flops = w.B * w.H * 8.0 * w.d * visible
    print(json.dumps({"oracle_timing": "long 32k", "workload": w.name(), "mode": "sampled rows",
                      "rows_per_head": int(len(rows)), "heads": w.B * w.H, "threads": cores, "cpu": cpu,
                      "s": dt, "gflops": flops / dt / 1e9}), flush=True)


def run_sdpa(args):
    """Context, not a target: torch.nn.functional.scaled_dot_product_attention, forward then backward
    with the same dO, on the headline workload, timed like the headline step (L2 flushed before every
    step, CUDA events around it); each backend torch offers is tried on its own and reported with its
    TFLOP/s (metric's FLOP count) or the error it raised. The library is only run."""
    import torch
    import torch.nn.functional as F
    from torch.nn.attention import SDPBackend, sdpa_kernel
    from tiled_attention_09_gb300.inputs import make_inputs
    w = bench_workload(args)
    dev = torch.device("cuda", 0)
    q, k, v, do = (t.to(dev) for t in make_inputs(w))
    q, k, v = (t.requires_grad_() for t in (q, k, v))
    flush = L2Flush(torch, dev)
    steps, warmup = max(3, min(args.steps, 50)), max(3, args.warmup)
    flops = 3.5 * w.fwd_flops()
    res = {}
    for name, be in (("cudnn", SDPBackend.CUDNN_ATTENTION), ("flash", SDPBackend.FLASH_ATTENTION),
                     ("efficient", SDPBackend.EFFICIENT_ATTENTION)):
        try:
            with sdpa_kernel([be]):
                def step():
                    q.grad = k.grad = v.grad = None
                    o = F.scaled_dot_product_attention(q, k, v, is_causal=w.causal, scale=w.scale)
                    o.backward(do)

                def fwd_only():
                    with torch.no_grad():
                        F.scaled_dot_product_attention(q, k, v, is_causal=w.causal, scale=w.scale)

                times = []
                for fn in (step, fwd_only):
                    for _ in range(warmup):
                        flush()
                        fn()
                    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                           for _ in range(steps)]
                    for e0, e1 in evs:
                        flush()
                        e0.record()
                        fn()
                        e1.record()
                    torch.cuda.synchronize()
                    times.append(statistics.median(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3)
            t, t_f = times
            res[name] = {"ms_per_step": 1e3 * t, "tflops": flops / t / 1e12, "fwd_ms": 1e3 * t_f,
                         "fwd_tflops": w.fwd_flops() / t_f / 1e12}
        except Exception as e:  # a backend that does not run on this GPU or shape
            torch.cuda.synchronize()
            res[name] = {"error": f"{type(e).__name__}: {str(e).splitlines()[0][:160] if str(e) else ''}"}
    print(json.dumps({"impl": "torch scaled_dot_product_attention (context)", "torch": torch.__version__,
                      "workload": w.name(), "steps": steps, "warmup": warmup,
                      "timing": "median step between two events, L2 flushed before each step", "backends": res}),
          flush=True)


def main():
    args = parse()
    if args.warmup < 3:
        args.warmup = 3
    if args.oracle_timing:
        run_oracle_timing(args)
        return
    if args.sdpa:
        run_sdpa(args)
        return
    if args.decode:
        run_decode(args)
    elif args.split_sweep:
        run_split_sweep(args)
    elif args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
