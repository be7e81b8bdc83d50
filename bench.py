"""Benchmark of the block-scaled FP8 video-attention hot path on GB300.

One step = stage 1 (fp8attn_prep: Q/K block quantisation, V-Smooth prep) +
stage 2 (fp8attn_fwd: the tcgen05 FP8 attention mainloop) over one batch of
seeded synthetic input already resident in HBM.  The default workload is the
Wan2.1-1.3B-shaped dense problem (B=1, H=12, T=32760 = 21x30x52, d=128,
exp2+cvt P-cast, S=256).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                       [--impl reference] [--no-cpu-baseline] [--smooth 0/1/2] [--v-bias]
                       [--cluster [--clusters K] [--cluster-dims r] [--cluster-iters n]] [--splits S]
                       [--tail-split {0,1}]
                       [--pv-fp4] [--pcast 0/1] [--vsmooth 0/1] [--reverse] [--S S] [--beta B]
For N > 1 launch under torch.distributed.run: every rank runs the same
workload on its own GPU (independent replicas of the per-head-parallel
problem, no collective on the data path); value = FLOPs of all ranks / the
slowest rank's time.  --impl reference times the CPU oracle (the plain numpy
restatement of the method) on a bounded sample of the same workload, one
head per host core in a process pool.  --pcast, --vsmooth, --reverse, --S
and --beta override the workload's P-cast variant (to isolate ExpCast,
V-Smooth or the KV order on one workload).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np

METRIC = "FP8 attention TFLOPS and fraction of GB300 FP8 dense peak; ms per call"
UNIT = "TFLOP/s"
NOMINAL_FP8_DENSE_TFLOPS = 4500.0
FP8_OVER_BF16 = 2.0          # nominal dense fp8 / bf16 tensor-core ratio

WORKLOAD_TEXT = {
    "wan21": "Wan2.1-1.3B-shaped dense attention: B=1 H=12 T=32760 (21x30x52) d=128, "
             "Q/K N(0,1)+4 offset channels, exp2+cvt P-cast S=256, no V-Smooth, forward",
    "wan22": "Wan2.2-14B-720p-shaped V-Smooth+ExpCast: B=1 H=40 T=75600 (21x45x80) d=128, "
             "16-cluster V with 0.5% x20 outliers, cluster-sorted permutation, S=256 beta=-0.35",
    "sta": "sliding-tile sparse: B=1 H=24 T=69120 (18x48x80), 6x8x8 tiles, 3x5x5 window (22.8% kept), "
           "exp2+cvt S=256",
    "tiny": "tiny dense: B=1 H=2 T=1024 d=128, exp2+cvt S=256, V-Smooth",
    "pcollapse": "P-collapse stress: B=1 H=8 T=16384, 4 sinks Delta=7, S=256, forward",
    "short4k": "single short head: B=1 H=1 T=4096 d=128, N(0,1), exp2+cvt S=256, no V-Smooth (32 query tiles)",
}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("nccl")
        return dist, dist.get_rank(), ws
    return None, 0, 1


def max_over_ranks(dist, values, device):
    """Element-wise maximum of `values` over all ranks (the slowest rank's times);
    the values themselves with one process."""
    if not dist:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


# B, T, H of each workload at full size (the GPU arm's shapes)
WORKLOAD_SHAPES = {"tiny": (1, 1024, 2), "wan21": (1, 32760, 12), "wan22": (1, 75600, 40),
                   "sta": (1, 69120, 24), "pcollapse": (1, 16384, 8), "short4k": (1, 4096, 1)}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def make(name, device, heads=None):
    from bit_attention_video_e4m3_gb300.workloads import make_workload
    return make_workload(name, device=device, H=heads)


def _oracle_head_job(job):
    """One head of the CPU oracle (runs in a pool worker): full stage-1 prep of
    the head, then emulated stage-2 attention for the sampled query rows; the
    exact fp64 attention of the same rows comes after the timed part, for the
    accuracy report.  Returns (emulated rows, exact rows or None, seconds,
    algorithmic FLOPs of the rows)."""
    from oracle import attention as OA
    from oracle import prep as OP
    from oracle.bf16 import bf16_from_bits
    qb, kb, vb, perm, rows, T, var, rp, cl, want_exact = job
    t0 = time.perf_counter()
    q, k, v = bf16_from_bits(qb), bf16_from_bits(kb), bf16_from_bits(vb)
    qc, sq = OP.quantize_qk_head(q)
    kc, sk = OP.quantize_qk_head(k if perm is None else k[perm])
    pv = OP.prep_v_head(v, perm, var["vsmooth"])
    out, _ = OA.emulated_attention_head(qc, sq, kc, sk, pv["vq"], pv["sv"], pv["mean"], T, rows,
                                        pcast=var["pcast"], S=var["S"], beta=var["beta"],
                                        reverse=var["reverse"], row_ptr=rp, col=cl)
    dt = time.perf_counter() - t0
    n_t = -(-T // 128)
    masks = None
    if rp is None:
        keys = len(rows) * T
    else:
        masks = {}
        keys = 0
        for r in rows:
            qt = int(r) // 128
            if qt not in masks:
                masks[qt] = OA.kept_key_mask(T, OA.tile_list_for_qtile(qt, n_t, False, rp, cl))
            keys += int(masks[qt].sum())
    exact = None
    if want_exact:
        kk = k if perm is None else k[perm]
        vv = v if perm is None else v[perm]
        mf = None if masks is None else (lambda r: masks[int(r) // 128])
        exact = OA.exact_attention_rows(q, kk, vv, rows, key_mask_for_row=mf)
    return out, exact, dt, 4.0 * keys * 128


def _pool_warm(_):
    # import the oracle in the worker before the timed map
    import oracle.attention  # noqa: F401
    import oracle.prep  # noqa: F401
    return os.getpid()


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


class OraclePool:
    """Process pool (spawn start method: safe next to a CUDA context) that runs
    the unchanged oracle one head per worker, each worker on one BLAS thread."""

    def __init__(self, workers: int):
        import concurrent.futures as cf
        import multiprocessing as mp
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        self.workers = max(1, workers)
        self.ex = cf.ProcessPoolExecutor(max_workers=self.workers, mp_context=mp.get_context("spawn"))
        pids = set(self.ex.map(_pool_warm, range(4 * self.workers)))
        self.started = len(pids)

    def run(self, jobs):
        """Wall time of the whole map and the per-job results."""
        t0 = time.perf_counter()
        res = list(self.ex.map(_oracle_head_job, jobs))
        return time.perf_counter() - t0, res

    def close(self):
        self.ex.shutdown()


def variant_of(w) -> dict:
    return dict(pcast=int(w.pcast), S=float(w.S), beta=float(w.beta), reverse=bool(w.reverse),
                vsmooth=bool(w.vsmooth))


def oracle_jobs(w, heads, rows_per_head: int, want_exact: bool):
    """Pool jobs for the given heads of workload ``w`` (device tensors are copied
    to the host as bf16 bits): rows 0.. of the head plus its last rows,
    including the ragged tail tile."""
    from bit_attention_video_e4m3_gb300.workloads import bf16_bits
    rows_per_head = min(rows_per_head, w.T)
    tail = min(128, rows_per_head // 2)
    rows = np.unique(np.concatenate([np.arange(rows_per_head - tail), np.arange(w.T - tail, w.T)]))
    rp = None if w.row_ptr is None else w.row_ptr.cpu().numpy()
    cl = None if w.col is None else w.col.cpu().numpy()
    var = variant_of(w)
    jobs = []
    for h in heads:
        perm = None if w.perm is None else w.perm[0, h].cpu().numpy().astype(np.int64)
        jobs.append((bf16_bits(w.q[0, :, h, :]), bf16_bits(w.k[0, :, h, :]), bf16_bits(w.v[0, :, h, :]),
                     perm, rows, w.T, var, rp, cl, want_exact))
    return jobs, rows


def sample_text(w, heads, rows, workers):
    return (f"oracle (numpy, fp64, unchanged) on {len(heads)} heads of the workload, one head per "
            f"process on {workers} host cores: full stage-1 prep of each head ({w.T} tokens) + "
            f"emulated stage-2 attention for {len(rows)} query rows per head (rows 0.. and the last "
            f"rows incl. the ragged tail tile) over all visited keys; value = 4*rows*keys*128 summed "
            f"over heads / wall time of the pool")


def measure_fp8_peak(n: int = 8192, seconds: float = 3.0):
    """cuBLASLt FP8 (E4M3 x E4M3 -> bf16) GEMM throughput through torch._scaled_mm:
    the best of 10 timed calls (burst) and the mean over a back-to-back loop of
    `seconds` (sustained, under the power cap).  A context figure for the
    attention kernel's roofline; the roofline itself uses the measured
    bf16 peak times the nominal fp8/bf16 ratio."""
    import torch
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(7)
    a = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn).t()    # column-major
    one = torch.ones((), device=dev)
    flop = 2.0 * n ** 3

    def mm():
        return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

    for _ in range(5):
        mm()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        mm()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    reps = max(1, int(seconds * 1e3 / best))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(0)
    clocks.start()
    e0.record()
    for _ in range(reps):
        mm()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    sustained_ms = e0.elapsed_time(e1) / reps
    print(json.dumps({"measure": "fp8 _scaled_mm peak", "n": n, "burst_tflops": flop / (best * 1e-3) / 1e12,
                      "sustained_tflops": flop / (sustained_ms * 1e-3) / 1e12, "reps": reps,
                      "clocks": clk}), flush=True)


def bench_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    from bit_attention_video_e4m3_gb300.workloads import make_workload
    B, T, H = WORKLOAD_SHAPES[args.workload]
    cores = host_cores()
    nh = max(1, min(H, cores))
    # the sampled heads only (the generator draws the same distributions as the
    # full workload; its values differ since fewer heads are drawn)
    w = make_workload(args.workload, device="cpu", H=nh)
    apply_variant(w, args)
    pool = OraclePool(nh)
    jobs, rows = oracle_jobs(w, list(range(nh)), ROWS_PER_HEAD, want_exact=False)
    for _ in range(args.warmup):
        pool.run(jobs[:1])
    vals, times = [], []
    for _ in range(args.steps):
        dt, res = pool.run(jobs)
        vals.append(sum(r[3] for r in res) / dt / 1e12)
        times.append(dt)
    pool.close()
    value = float(np.mean(vals))
    desc = sample_text(w, list(range(nh)), rows, pool.workers)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * float(np.mean(times)), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[args.workload], "B": B, "T": T, "H": H, "d": 128,
                       "seed": w.seed, "flops_per_step": w.flops() * H / nh, **variant_config(args),
                       "l2": L2_TEXT[args.workload]},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.workers, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


ROWS_PER_HEAD = 256


def apply_variant(w, args):
    """--pcast / --vsmooth / --reverse / --S / --beta override the workload's variant."""
    if args.pcast is not None:
        w.pcast = args.pcast
    if args.vsmooth is not None:
        w.vsmooth = bool(args.vsmooth)
    if args.reverse:
        w.reverse = True
    if args.S is not None:
        w.S = float(args.S)
    if args.beta is not None:
        w.beta = float(args.beta)


def variant_config(args) -> dict:
    out = {}
    if args.pcast is not None:
        out["pcast"] = ["exp2+cvt", "ExpCast"][args.pcast]
    if args.vsmooth is not None:
        out["vsmooth"] = bool(args.vsmooth)
    if args.reverse:
        out["kv_order"] = "reverse"
    if args.S is not None:
        out["S"] = float(args.S)
    if args.beta is not None:
        out["beta"] = float(args.beta)
    return out


def _l2_text(shape):
    B, T, H = shape
    mb = 3 * B * T * H * 128 * 2 / 1e6
    if mb > 129:
        return "inputs larger than L2: bf16 Q,K,V = %.0f MB per step (L2 = 129 MB); no explicit flush" % mb
    return "inputs smaller than L2: bf16 Q,K,V = %.1f MB per step (L2 = 129 MB); not flushed" % mb


L2_TEXT = {k: _l2_text(v) for k, v in WORKLOAD_SHAPES.items()}


def bench_gpu(args):
    import torch

    import bit_attention_video_e4m3_gb300 as fa
    from bit_attention_video_e4m3_gb300.build import build_library
    dist, rank, world = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    # the CPU oracle's process pool (rank 0 at N=1 only) starts before the first GPU call
    pool = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        pool = OraclePool(min(args.heads or WORKLOAD_SHAPES[args.workload][2], host_cores()))
    torch.cuda.set_device(local)
    build_library()
    dev = torch.device("cuda", local)
    w = make(args.workload, dev, args.heads)
    apply_variant(w, args)
    B, T, H = w.B, w.T, w.H
    flops = w.flops()
    stream = torch.cuda.Stream(device=dev)
    vf = 1 if args.pv_fp4 else 0
    pp = fa.Prepped.empty(B, T, H, dev, with_offset=(args.smooth == 2 or args.v_bias), v_format=vf)
    sm = dict(smooth=args.smooth, v_bias=args.v_bias, v_format=vf)
    if args.pv_fp4:
        w.pcast = fa.PCAST_EXP2_CVT        # the 4-bit PV product casts P with exp2
    out = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device=dev)
    ws_p = torch.empty(fa.prep_workspace_bytes(B, T, H), dtype=torch.uint8, device=dev)
    n_splits = args.splits if args.splits > 0 else fa.auto_splits(B, T, H)
    # the last wave of query tiles split with the unsplit P codes (dense, 8-bit PV)
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    tail = (args.tail_split and w.row_ptr is None and not args.pv_fp4 and n_splits == 1
            and fa.tail_plan(B, T, H, num_sms)[0] >= 2)
    tail_plan = fa.tail_plan(B, T, H, num_sms) if tail else None
    ws_f = torch.empty(fa.fwd_tail_workspace_bytes(B, T, H, num_sms) if tail
                       else fa.fwd_split_workspace_bytes(B, T, H, n_splits), dtype=torch.uint8, device=dev)
    kw = dict(row_ptr=w.row_ptr, col=w.col, reverse=w.reverse, pcast=w.pcast, S=w.S, beta=w.beta,
              vsmooth=w.vsmooth, out=out, workspace=ws_f, stream=stream, n_splits=n_splits,
              **({"tail_split": True, "num_sms": num_sms} if tail else {}))
    # online V clustering inside the step: its permutation replaces the workload's
    ck = dict(n_clusters=args.clusters, n_dims=args.cluster_dims, iters=args.cluster_iters)
    perm_c = torch.empty((B, H, T), dtype=torch.int32, device=dev) if args.cluster else None
    ws_c = (torch.empty(fa.cluster_workspace_bytes(B, T, H, args.cluster_dims), dtype=torch.uint8,
                        device=dev) if args.cluster else None)
    perm_used = perm_c if args.cluster else w.perm

    def step(ev=None):
        if args.cluster:
            fa.v_cluster(w.v, perm=perm_c, workspace=ws_c, stream=stream, **ck)
            if ev is not None:
                ev[2].record(stream)
        fa.prep(w.q, w.k, w.v, perm=perm_used, vsmooth=w.vsmooth, out=pp, workspace=ws_p, stream=stream,
                **sm)
        if ev is not None:
            ev[0].record(stream)
        fa.fwd(pp, **kw)
        if ev is not None:
            ev[1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    if fa.check_status(ws_f, stream=stream) != 0:
        raise RuntimeError("attention kernel reported a device error during warm-up")

    # ---- device-timed region: K steps, inputs resident in HBM
    attn_ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    starts = []
    for i in range(args.steps):
        starts.append(torch.cuda.Event(enable_timing=True))
        starts[-1].record(stream)
        step(attn_ev[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    ms_total = t_start.elapsed_time(t_end)
    attn_ms = [ev[0].elapsed_time(ev[1]) for ev in attn_ev]
    step_ms = [s0.elapsed_time(ev[1]) for s0, ev in zip(starts, attn_ev)]
    prep_only_ms = [s0.elapsed_time(ev[0]) for s0, ev in zip(starts, attn_ev)]
    cluster_ms = (float(np.mean([s0.elapsed_time(ev[2]) for s0, ev in zip(starts, attn_ev)]))
                  if args.cluster else 0.0)
    ms_total, = max_over_ranks(dist, [ms_total], dev)
    ms_step = ms_total / args.steps
    value = flops * world * args.steps / (ms_total * 1e-3) / 1e12
    attn_ms_avg = float(np.mean(attn_ms))
    prep_ms = ms_step - attn_ms_avg - cluster_ms

    # ---- end to end through the public API with HOST buffers
    hq = torch.empty_like(w.q, device="cpu").pin_memory()
    hk = torch.empty_like(w.k, device="cpu").pin_memory()
    hv = torch.empty_like(w.v, device="cpu").pin_memory()
    hq.copy_(w.q)
    hk.copy_(w.k)
    hv.copy_(w.v)
    hout = torch.empty((B, T, H, 128), dtype=torch.bfloat16).pin_memory()
    dq, dk, dv = torch.empty_like(w.q), torch.empty_like(w.k), torch.empty_like(w.v)
    h2d = 3 * hq.numel() * hq.element_size()
    d2h = hout.numel() * hout.element_size()
    e2e_steps = max(3, min(args.steps, 10))

    def e2e_step():
        with torch.cuda.stream(stream):
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            if args.cluster:
                fa.v_cluster(dv, perm=perm_c, workspace=ws_c, stream=stream, **ck)
            fa.prep(dq, dk, dv, perm=perm_used, vsmooth=w.vsmooth, out=pp, workspace=ws_p, stream=stream,
                    **sm)
            fa.fwd(pp, **kw)
            hout.copy_(out, non_blocking=True)

    e2e_step()
    stream.synchronize()
    if dist:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    stream.synchronize()
    e2e_serial_ms = e0.elapsed_time(e1) / e2e_steps

    # Pipelined end to end, as a serving loop runs it: step k's inputs go up on
    # one copy stream while step k-1 computes, and step k-1's output comes down on
    # another while step k computes (double-buffered device inputs and outputs,
    # ordered by events).  Every step's copies are inside the timed region.
    # one upload stream per input tensor, so that the three copies can run on
    # separate copy engines at once
    ups = [torch.cuda.Stream(device=dev) for _ in range(3)]
    down = torch.cuda.Stream(device=dev)
    dbuf = [(torch.empty_like(w.q), torch.empty_like(w.k), torch.empty_like(w.v)) for _ in range(2)]
    obuf = [torch.empty((B, T, H, 128), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    hobuf = [hout, torch.empty_like(hout).pin_memory()]
    n_pipe = e2e_steps + 2
    ev = {key: [torch.cuda.Event() for _ in range(n_pipe)] for key in ("comp", "down")}
    ev_up = [[torch.cuda.Event() for _ in range(n_pipe)] for _ in range(3)]

    def pipe_step(k):
        sl = k % 2
        for u, dst, src, evs in zip(ups, dbuf[sl], (hq, hk, hv), ev_up):
            with torch.cuda.stream(u):
                if k >= 2:
                    u.wait_event(ev["comp"][k - 2])     # the inputs of step k-2 are consumed
                dst.copy_(src, non_blocking=True)
                evs[k].record(u)
        bq, bk, bv = dbuf[sl]
        with torch.cuda.stream(stream):
            for evs in ev_up:
                stream.wait_event(evs[k])
            if k >= 2:
                stream.wait_event(ev["down"][k - 2])    # the output of step k-2 has been read back
            if args.cluster:
                fa.v_cluster(bv, perm=perm_c, workspace=ws_c, stream=stream, **ck)
            fa.prep(bq, bk, bv, perm=perm_used, vsmooth=w.vsmooth, out=pp, workspace=ws_p, stream=stream, **sm)
            fa.fwd(pp, **dict(kw, out=obuf[sl]))
            ev["comp"][k].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(ev["comp"][k])
            hobuf[sl].copy_(obuf[sl], non_blocking=True)
            ev["down"][k].record(down)

    pipe_step(0)
    pipe_step(1)
    torch.cuda.synchronize()
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    p0.record(ups[0])
    for u in ups[1:]:
        u.wait_event(p0)
    for k in range(2, n_pipe):
        pipe_step(k)
    p1.record(down)
    torch.cuda.synchronize()
    e2e_ms = p0.elapsed_time(p1) / e2e_steps
    e2e_ms, e2e_serial_ms = max_over_ranks(dist, [e2e_ms, e2e_serial_ms], dev)
    if fa.check_status(ws_f, stream=stream) != 0:
        raise RuntimeError("attention kernel reported a device error")

    if rank != 0:
        return
    peaks, src = _peaks()
    # the attention kernel is timed on its own (a few-millisecond launch), so the
    # burst figure applies: 2 x the measured cuBLAS bf16 burst (nominal fp8/bf16 ratio)
    peak_fp8 = FP8_OVER_BF16 * peaks["bf16_tflops"]
    attn_tflops = flops / (attn_ms_avg * 1e-3) / 1e12
    profile_traffic = _ncu_traffic(args.workload, w)
    context = context_peaks(clk)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "B": B, "T": T, "H": H, "d": 128,
                   "seed": w.seed, "flops_per_step": flops,
                   **({"smooth": ["none", "k", "kv"][args.smooth], "v_bias": bool(args.v_bias)}
                      if (args.smooth or args.v_bias) else {}),
                   **({"v_cluster": dict(ck, permutation="online V clustering in every step")}
                      if args.cluster else {}),
                   **({"n_splits": n_splits} if n_splits > 1 else {}),
                   **({"last_wave_split": {"parts": tail_plan[0], "query_tiles": tail_plan[1],
                                           "part_bounds_kv_tiles": tail_plan[2], "num_sms": num_sms}}
                      if tail else {}),
                   **({"pv": "NVFP4 (E2M1 P and V, UE4M3 scale per 16), exp2 P cast"} if args.pv_fp4 else {}),
                   **variant_config(args),
                   **({"heads_override": args.heads} if args.heads else {}),
                   "l2": L2_TEXT[args.workload] if not args.heads else _l2_text((B, T, H))},
        "clocks": clk,
        "e2e": {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipelined": "inputs of step k+1 uploaded on three copy streams (one per tensor) and output of step k-1 "
                             "read back on a fourth while step k computes (double-buffered, event-ordered)",
                "serial_value": flops * world / (e2e_serial_ms * 1e-3) / 1e12,
                "serial_ms_per_step": e2e_serial_ms},
        "gpu_launches": (4 + (3 if args.smooth else 0) + (1 if pp.v_offset is not None else 0)
                         + ((5 + 2 * args.cluster_iters) if args.cluster else 0)
                         + (1 if n_splits > 1 else 0) + (2 if tail else 0)) * args.steps,
        "kernel_source_sha256": kernel_source_hash(),
        "attn_ms": attn_ms_avg, "prep_ms": prep_ms, "attn_tflops": attn_tflops,
        **({"cluster_ms": cluster_ms} if args.cluster else {}),
        "median_ms": {"attention": float(np.median(attn_ms)), "prep": float(np.median(prep_only_ms)),
                      "step": float(np.median(step_ms)), "calls": args.steps},
        "frac_of_nominal_fp8_dense": attn_tflops / NOMINAL_FP8_DENSE_TFLOPS,
        "roofline": {"kernel": "attn_fwd_kernel", "bound": "tensor", "achieved": attn_tflops,
                     "peak": peak_fp8, "unit": "TFLOP/s", "frac": attn_tflops / peak_fp8,
                     "peak_source": f"{src}: 2 x bf16_tflops (burst; fp8/bf16 nominal dense ratio)",
                     "traffic": profile_traffic,
                     "context": context},
        "variant": variant_of(w),
    }
    if pool is not None:
        # CPU baseline: the oracle on min(H, cores) heads in parallel, timed; its
        # outputs double as the accuracy report of this run's GPU output
        heads = list(range(pool.workers))
        jobs, rows = oracle_jobs(w, heads, ROWS_PER_HEAD, want_exact=True)
        dt, res = pool.run(jobs)
        pool.close()
        line["cpu_baseline"] = {"value": sum(r[3] for r in res) / dt / 1e12, "unit": UNIT,
                                "cores": pool.workers, "kind": "oracle",
                                "sample": sample_text(w, heads, rows, pool.workers), "seconds": dt}
        if args.pv_fp4 or args.smooth or args.v_bias or n_splits > 1 or args.cluster:
            line["accuracy"] = {"skipped": "this variant's parity is checked by the GPU tests; the sampled-row "
                                           "report covers the plain E4M3 path"}
        else:
            line["accuracy"] = accuracy_report(out, heads, rows, res)
    print(json.dumps(line), flush=True)


def accuracy_report(out, heads, rows, res) -> dict:
    """GPU output rows against the oracle: rel-L2 to the emulated-quantisation
    result (the parity bar, per head and worst single row) and cosine / rel-L2 to
    exact fp64 attention, beside the emulation's own cosine to exact."""
    def cos(a, b):
        return float(np.sum(a * b) / (np.linalg.norm(a) * np.linalg.norm(b)))

    per = []
    for h, (emu, exact, _, _) in zip(heads, res):
        got = out[0, :, h, :].float().cpu().numpy().astype(np.float64)[rows]
        d = got - emu
        rn = np.linalg.norm(emu, axis=1)
        row_rel = np.linalg.norm(d, axis=1) / np.where(rn > 0, rn, 1.0)
        per.append({"head": h,
                    "rel_l2_vs_oracle": float(np.linalg.norm(d) / np.linalg.norm(emu)),
                    "row_rel_l2_max_vs_oracle": float(row_rel.max()),
                    "cos_vs_exact": cos(got, exact),
                    "rel_l2_vs_exact": float(np.linalg.norm(got - exact) / np.linalg.norm(exact)),
                    "oracle_cos_vs_exact": cos(emu, exact)})
    return {"rows_per_head": int(len(rows)), "heads": len(per),
            "rel_l2_vs_oracle_max": max(p["rel_l2_vs_oracle"] for p in per),
            "row_rel_l2_max_vs_oracle": max(p["row_rel_l2_max_vs_oracle"] for p in per),
            "cos_vs_exact_min": min(p["cos_vs_exact"] for p in per),
            "cos_vs_exact_mean": float(np.mean([p["cos_vs_exact"] for p in per])),
            "oracle_cos_vs_exact_min": min(p["oracle_cos_vs_exact"] for p in per),
            "oracle_cos_vs_exact_mean": float(np.mean([p["oracle_cos_vs_exact"] for p in per])),
            "per_head": per}


def context_peaks(clk) -> dict:
    """Other denominators, for context: NVIDIA's nominal dense FP8 figure and the
    measured per-instruction tcgen05 E4M3 rate (an M128 N128 K32 MMA every 64 SM
    cycles = 16384 flop per clock per SM, 152 SMs) at the SM clock sampled
    during the timed region."""
    mhz = clk.get("sm_mhz") or 2070.0
    return {"nominal_fp8_dense_tflops": NOMINAL_FP8_DENSE_TFLOPS,
            "tcgen05_e4m3_instruction_rate_tflops": 16384.0 * 152 * mhz * 1e6 / 1e12,
            "at_sm_mhz": mhz}


def kernel_source_hash() -> str:
    """sha256 over what the attention kernel is compiled from (attn.cu, ptx.cuh and the
    AttnParams struct of kernels.cuh), to tell whether a profile is current."""
    import hashlib
    import re
    hsh = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_attention_video_e4m3_gb300", "csrc")
    for name in ("attn.cu", "ptx.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            hsh.update(f.read())
    with open(os.path.join(csrc, "kernels.cuh")) as f:
        m = re.search(r"struct AttnParams \{.*?\n\};", f.read(), re.S)
    hsh.update(m.group(0).encode() if m else b"")
    return hsh.hexdigest()[:16]


def _ncu_traffic(workload, w=None):
    """DRAM bytes per launch of the attention kernel from the committed ncu summary.

    The summary (profiles/attn_fwd_<workload>[_expcast].md) records the kernel
    source hash it was taken with; if the sources changed since, the figure is
    stale -> None.
    """
    suffix = "_expcast" if (w is not None and w.pcast == 1 and workload == "wan21") else ""
    path = os.path.join(ROOT, "profiles", f"attn_fwd_{workload}{suffix}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_source_sha256") != kernel_source_hash():
        return None
    if w is not None and "heads" in fields and int(fields["heads"]) != w.H:
        return None                     # the figure is for the workload's full head count
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="wan21", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--smooth", type=int, default=0, choices=[0, 1, 2],
                    help="sequence-mean smoothing in the prep: 0 none, 1 K, 2 K and V")
    ap.add_argument("--v-bias", action="store_true", help="compensate the measured E4M3 mean bias of V")
    ap.add_argument("--cluster", action="store_true",
                    help="compute the permutation by online V clustering inside every step")
    ap.add_argument("--clusters", type=int, default=32)
    ap.add_argument("--cluster-dims", type=int, default=8)
    ap.add_argument("--cluster-iters", type=int, default=4)
    ap.add_argument("--measure-fp8-peak", action="store_true",
                    help="time cuBLASLt FP8 GEMMs (torch._scaled_mm) instead of the workload")
    ap.add_argument("--pv-fp4", action="store_true",
                    help="4-bit PV product: NVFP4 V residual and P (exp2 P cast)")
    ap.add_argument("--splits", type=int, default=1,
                    help="split-KV parts per query tile (1: none, 0: the library's automatic choice)")
    ap.add_argument("--tail-split", type=int, choices=[0, 1], default=1,
                    help="split the last wave of query tiles into parts that keep the unsplit P codes "
                         "(dense attention, 8-bit PV, no --splits; 0: plain kernel)")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="omit the CPU oracle leg (baseline timing and accuracy report), e.g. under a profiler")
    ap.add_argument("--pcast", type=int, choices=[0, 1], default=None,
                    help="override the workload's P cast: 0 exp2+cvt, 1 ExpCast")
    ap.add_argument("--vsmooth", type=int, choices=[0, 1], default=None,
                    help="override the workload's V-Smooth setting")
    ap.add_argument("--reverse", action="store_true", help="visit the KV tiles in reverse order")
    ap.add_argument("--S", type=float, default=None, help="override the static P scale S")
    ap.add_argument("--beta", type=float, default=None, help="override the ExpCast beta")
    ap.add_argument("--heads", type=int, default=None,
                    help="fewer heads than the workload's (small cases for profiling; not a bench line)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.measure_fp8_peak:
        measure_fp8_peak()
    elif args.impl == "reference":
        bench_reference(args)
    else:
        bench_gpu(args)


if __name__ == "__main__":
    main()
