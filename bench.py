"""Benchmark of the MXFP4 MoE expert FFN on GB300 (one JSON line on stdout).

A step is one routed MoE forward (routing permutation, MX quantisation of x, L1 grouped
GEMM with fused SiLU-gate + re-quant, L2 grouped GEMM, top-k weighted combine) over the
prefill workload: 8192 tokens, hidden 7168, intermediate 3072, 48 experts, top-8 with
Zipf(1.0)-skewed routing, MXFP4 weights (1.68 GB), synthetic seeded inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs N independent replicas (one process per GPU under torchrun, weak scaling):
each rank processes its own batch; the timed region is bracketed by a barrier and a
device synchronisation and the slowest rank's time is used.

`value` is the algorithmic TFLOP/s of the forward (132,120,576 FLOP per routed pair) with
every input resident in HBM and the weight scales in the GEMM's tile layout (converted
once, at weight load, like the weights themselves); `e2e` is the same metric through the C ABI with the step's
inputs copied from pinned host memory and the output copied back inside the timed region.
`roofline` reports the L1 GEMM, timed live with CUDA events recorded by the library at
its phase boundaries, against the measured burst BF16 tensor rate times the nominal
FP4:BF16 ratio (and, beside it, against the FP4 MMA issue rate at the sampled SM clock).
`cpu_baseline` times the CPU oracle on a bounded token sample: one process per host core
(spawned, each single-threaded), with the single-core figure beside it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mp
import os
import subprocess
import sys
import time

# Every oracle process runs on one host core: pin BLAS before numpy loads (spawned oracle
# workers inherit this).
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import (CONFIGS, make_config_inputs, make_dequant_inputs, make_gemm_inputs,  # noqa: E402
                       make_moe_inputs, make_nvfp4_config_inputs, make_nvfp4_scales)

METRIC = "MoE fwd TFLOP/s (MXFP4 grouped GEMM) & dequant GB/s, % of roofline, 1 GB300"
WORKLOAD = ("routed MoE prefill forward: T=8192 tokens, hidden 7168, intermediate 3072, 48 experts, "
            "top-8, Zipf(1.0) expert skew, MXFP4 (E2M1 + E8M0/32) weights")
FP4_OVER_BF16 = 13.5 / 2.25       # nominal dense FP4 : BF16 tensor-core ratio on GB300
# FP4 MMA issue rate measured on every SM of a GB300: one 128 x 256 x 64 kind::mxf4 MMA
# (2 * 128 * 256 * 64 FLOP) per 128 cycles, i.e. 32,768 FLOP per cycle per SM.
MMA_FLOP_PER_CYCLE_SM = 2 * 128 * 256 * 64 / 128
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "l1_gemm_prefill_traffic.json")
GEMM_SRC = os.path.join(ROOT, "fp4_block_scaled_mxfp4_gb300", "csrc", "mx_gemm.cu")


def flops_per_pair(H, I):
    return 2 * H * 2 * I + 2 * I * H


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world, device=None):
    """The slowest rank's figure, on every rank (all-reduce MAX); x itself when world == 1."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flop_per_rank_step, ms_per_step):
    """Whole-job throughput: every rank runs its own batch (replicas), timed by the slowest."""
    return world * flop_per_rank_step / (ms_per_step * 1e-3) / 1e12


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def fp4_peak_tflops(peaks):
    """The FP4 roofline denominator: the measured burst BF16 tensor rate (the GEMMs here are
    timed in sub-second regions) times the nominal FP4:BF16 ratio."""
    return peaks["bf16_tflops"] * FP4_OVER_BF16


def mma_rate_tflops(num_sms, sm_mhz):
    """FP4 MMA issue rate of all SMs at the given SM clock (TFLOP/s)."""
    return MMA_FLOP_PER_CYCLE_SM * num_sms * sm_mhz * 1e6 / 1e12


def l1_traffic_per_launch():
    """DRAM bytes per L1 launch from the committed ncu summary, if it matches this kernel."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    with open(GEMM_SRC, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    if d.get("kernel_source_sha256") != sha:
        return None
    return d.get("dram_bytes_per_full_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def time_oracle_sample(inp, tokens):
    import oracle
    t0 = time.perf_counter()
    oracle.moe_forward(inp.x, inp.topk_ids, inp.topk_w, inp.w13, inp.s13, inp.w2, inp.s2, inp.I,
                       tokens=tokens)
    dt = time.perf_counter() - t0
    ids = inp.topk_ids[tokens]
    pairs = int(((ids >= 0) & (ids < inp.E)).sum())
    return dt, pairs


# ---- the oracle on every host core: one spawned, single-threaded process per core, each
# holding its own copy of the seeded prefill inputs and computing whole tokens ----
_ORACLE_INP = None


def _oracle_worker_init():
    global _ORACLE_INP
    _ORACLE_INP = make_config_inputs("prefill")


def _oracle_worker_token(t):
    dt, pairs = time_oracle_sample(_ORACLE_INP, [int(t)])
    return pairs


def oracle_processes():
    """Host cores to use, limited so each process's copy of the inputs (~1.8 GB) and its
    per-expert float64 temporaries (~1.2 GB) fit in the available memory."""
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    avail = None
    try:
        with open("/proc/meminfo") as f:
            for ln in f:
                if ln.startswith("MemAvailable:"):
                    avail = int(ln.split()[1]) * 1024
    except OSError:
        pass
    if avail is not None:
        cores = min(cores, max(1, int(avail // (4 << 30))))
    return max(1, cores)


class OraclePool:
    """A spawn-started pool of single-threaded oracle processes (spawn: the parent may
    already hold a CUDA context, which a forked child must not inherit)."""

    def __init__(self, procs):
        self.procs = procs
        self.pool = mp.get_context("spawn").Pool(procs, initializer=_oracle_worker_init)
        # every worker has built its inputs before anything is timed
        self.pool.map(_oracle_worker_token, [0] * procs, chunksize=1)

    def run(self, tokens):
        """Wall time and routed pairs of the oracle over `tokens`, spread over the processes."""
        t0 = time.perf_counter()
        pairs = sum(self.pool.map(_oracle_worker_token, list(tokens), chunksize=1))
        return time.perf_counter() - t0, pairs

    def close(self):
        self.pool.terminate()
        self.pool.join()


def run_reference(args):
    """The reference arm: the CPU oracle on every host core, one prefill token per core and
    step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    c = CONFIGS["prefill"]
    fpp = flops_per_pair(c["H"], c["I"])
    procs = oracle_processes()
    pool = OraclePool(procs)
    rng = np.random.default_rng(1234)
    try:
        for _ in range(args.warmup):
            pool.run(rng.integers(c["T"], size=procs))
        total_t, total_pairs = 0.0, 0
        for _ in range(args.steps):
            dt, pairs = pool.run(rng.integers(c["T"], size=procs))
            total_t += dt
            total_pairs += pairs
    finally:
        pool.close()
    value = total_pairs * fpp / total_t / 1e12
    sample = (f"{procs} prefill tokens per step (one per process, {procs * 8} routed pairs), numpy float64, "
              f"{procs} single-threaded processes")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": procs, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from fp4_block_scaled_mxfp4_gb300 import build as _build
    _build.build()
    import fp4_block_scaled_mxfp4_gb300 as mx

    c = dict(CONFIGS["prefill"])
    if args.tokens:
        c["T"] = args.tokens
    T, H, I, E, K = c["T"], c["H"], c["I"], c["E"], c["K"]
    inp = make_moe_inputs(**c) if args.tokens else make_config_inputs("prefill")
    pairs = int(((inp.topk_ids >= 0) & (inp.topk_ids < E)).sum())
    flop_step = pairs * flops_per_pair(H, I)
    flop_l1 = pairs * 2 * H * 2 * I

    def d(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    x = d(inp.x).view(torch.bfloat16)
    ids = d(inp.topk_ids)
    w = d(inp.topk_w)
    w13, s13, w2, s2 = (d(a) for a in (inp.w13, inp.s13, inp.w2, inp.s2))
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(mx.moe_mxfp4_workspace_size(T, H, I, E, K, True), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    n_phase = 6
    # weight load: the weight scales go into the tile layout once (a weight-format transform)
    s13t = torch.empty(mx.mxfp4_tiled_scales_bytes(E * 2 * I, H), dtype=torch.uint8, device=dev)
    s2t = torch.empty(mx.mxfp4_tiled_scales_bytes(E * H, I), dtype=torch.uint8, device=dev)
    mx.mxfp4_scales_to_tiled(s13.view(-1, H // 32), s13t)
    mx.mxfp4_scales_to_tiled(s2.view(-1, I // 32), s2t)

    def step(evs=None, tiled=True):
        if tiled:
            mx.moe_mxfp4_forward(x, ids, w, w13, s13t, w2, s2t, out, ws, stream=stream, events=evs,
                                 scales_tiled=True)
        else:
            mx.moe_mxfp4_forward(x, ids, w, w13, s13, w2, s2, out, ws, stream=stream, events=evs)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    if mx.device_status() != 0:
        raise RuntimeError("device status set during warm-up")

    # ---------------- device-resident timed region ----------------
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_phase)] for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for row in ev:
            for e in row:
                e.record(stream)          # create the underlying CUDA events
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clocks:
        with torch.cuda.stream(stream):
            start.record(stream)
            for i in range(args.steps):
                step(ev[i])
            stop.record(stream)
        torch.cuda.synchronize()
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), world, dev)
    if mx.device_status() != 0:
        raise RuntimeError("device status set during the timed region")
    phase_names = ["route", "quant_gather", "l1_gemm", "l2_gemm", "combine"]
    phase_ms = {n: 0.0 for n in phase_names}
    for row in ev:
        for j, n in enumerate(phase_names):
            phase_ms[n] += row[j].elapsed_time(row[j + 1])
    phase_ms = {n: v / args.steps for n, v in phase_ms.items()}
    ms_per_step = elapsed_ms / args.steps
    value = job_tflops(world, flop_step, ms_per_step)

    # ---------------- end-to-end through the C ABI with host buffers ----------------
    # A serving loop: every step uploads its inputs from pinned host memory, runs the
    # forward and downloads its result. Uploads and downloads run on their own streams,
    # double-buffered, so step i+1's upload and step i-1's download overlap step i's forward.
    e2e_steps = max(4, min(args.steps, 20))
    hx = torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True)
    hx.view(torch.int16).numpy()[:] = inp.x.view(np.int16)
    hids = torch.from_numpy(inp.topk_ids.copy()).pin_memory()
    hw = torch.from_numpy(inp.topk_w.copy()).pin_memory()
    nbuf = 2
    hout = [torch.empty((T, H), dtype=torch.bfloat16, pin_memory=True) for _ in range(nbuf)]
    xin = [torch.empty_like(x) for _ in range(nbuf)]
    idin = [torch.empty_like(ids) for _ in range(nbuf)]
    win = [torch.empty_like(w) for _ in range(nbuf)]
    outb = [torch.empty_like(out) for _ in range(nbuf)]
    s_up, s_down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_up = [torch.cuda.Event() for _ in range(nbuf)]      # inputs of buffer b uploaded
    ev_fwd = [torch.cuda.Event() for _ in range(nbuf)]     # forward of buffer b done
    ev_down = [torch.cuda.Event() for _ in range(nbuf)]    # result of buffer b downloaded
    for b in range(nbuf):
        for e in (ev_fwd[b], ev_down[b]):
            e.record(stream)

    def e2e_run(n):
        for i in range(n):
            b = i % nbuf
            s_up.wait_event(ev_fwd[b])                      # the forward two steps back read xin[b]
            with torch.cuda.stream(s_up):
                xin[b].copy_(hx, non_blocking=True)
                idin[b].copy_(hids, non_blocking=True)
                win[b].copy_(hw, non_blocking=True)
                ev_up[b].record(s_up)
            stream.wait_event(ev_up[b])
            stream.wait_event(ev_down[b])                   # outb[b] downloaded two steps back
            mx.moe_mxfp4_forward(xin[b], idin[b], win[b], w13, s13t, w2, s2t, outb[b], ws, stream=stream,
                                 scales_tiled=True)
            ev_fwd[b].record(stream)
            s_down.wait_event(ev_fwd[b])
            with torch.cuda.stream(s_down):
                hout[b].copy_(outb[b], non_blocking=True)
                ev_down[b].record(s_down)

    e2e_run(2)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_up.wait_event(e0)
    s_down.wait_event(e0)
    e2e_run(e2e_steps)
    for b in range(nbuf):
        stream.wait_event(ev_down[b])                       # every result is on the host
    e1.record(stream)
    torch.cuda.synchronize()
    if not np.array_equal(hout[(e2e_steps - 1) % nbuf].view(torch.int16).numpy(), out.cpu().view(torch.int16).numpy()):
        raise RuntimeError("end-to-end result differs from the device-resident forward")
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
    h2d = hx.numel() * 2 + hids.numel() * 4 + hw.numel() * 4
    d2h = hout[0].numel() * 2

    # ---------------- context figures measured outside the timed step ----------------
    extra = {}
    if rank == 0:
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            step(tiled=False)
            p0.record(stream)
            for _ in range(10):
                step(tiled=False)
            p1.record(stream)
        torch.cuda.synchronize()
        extra["forward_row_major_scales_ms"] = p0.elapsed_time(p1) / 10
    if rank == 0 and not args.no_extra:
        extra.update(measure_extra(mx, torch, dev, stream))

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    peaks, peak_kind = measured_peaks()
    fp4_peak = fp4_peak_tflops(peaks)
    l1_tflops = flop_l1 / (phase_ms["l1_gemm"] * 1e-3) / 1e12
    traffic = l1_traffic_per_launch()
    clk = clocks.summary()
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mma_peak = mma_rate_tflops(num_sms, clk["sm_mhz"] or peaks.get("sm_max_mhz", 2070.0))

    cpu = None
    if not args.no_cpu_baseline and not args.tokens:
        cpu = cpu_baseline(inp, H, I)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e2m1", "data": "synthetic",
        "config": {"workload": WORKLOAD if not args.tokens else WORKLOAD.replace("T=8192", f"T={T}"),
                   "routed_pairs_per_step": pairs, "flop_per_step": flop_step,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (1.68 GB MXFP4 weights + 117 MB activations per step)"},
        "roofline": {"kernel": "L1 grouped GEMM (gate/up, fused SiLU + MX re-quant)", "bound": "tensor",
                     "achieved": l1_tflops, "peak": fp4_peak, "unit": "TFLOP/s", "frac": l1_tflops / fp4_peak,
                     "traffic": traffic,
                     "peak_source": f"{peak_kind} bf16_tflops (burst) x {FP4_OVER_BF16:g} (nominal FP4:BF16)",
                     "mma_rate_peak": mma_peak, "frac_mma_rate": l1_tflops / mma_peak,
                     "mma_rate_source": f"one 128x256x64 kind::mxf4 MMA per 128 cycles per SM, {num_sms} SMs, "
                                        f"median sampled SM clock"},
        "phases_ms": phase_ms,
        "cpu_baseline": cpu,
        "e2e": {"value": job_tflops(world, flop_step, e2e_ms), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": 6 * args.steps,
        "clocks": clk,
        "extra": extra,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def cpu_baseline(inp, H, I):
    """The oracle on a bounded sample of the step's tokens: on every host core (one
    single-threaded process per core, two tokens each), and on one core (two tokens)."""
    fpp = flops_per_pair(H, I)
    rng = np.random.default_rng(7)
    dt1, p1 = time_oracle_sample(inp, sorted(rng.choice(inp.T, size=2, replace=False).tolist()))
    single = {"value": p1 * fpp / dt1 / 1e12, "unit": "TFLOP/s", "cores": 1,
              "sample": f"2 prefill tokens ({p1} routed pairs), {dt1:.1f} s"}
    procs = oracle_processes()
    pool = OraclePool(procs)
    try:
        dt, p = pool.run(rng.integers(inp.T, size=2 * procs))
    finally:
        pool.close()
    return {"value": p * fpp / dt / 1e12, "unit": "TFLOP/s", "cores": procs, "kind": "oracle",
            "sample": f"{2 * procs} prefill tokens ({p} routed pairs) over {procs} single-threaded processes, "
                      f"numpy float64, {dt:.1f} s",
            "single_core": single}


def measure_extra(mx, torch, dev, stream):
    """Dequant sweep GB/s and the decode / shared-expert forwards (context, same GPU)."""
    res = {}
    peaks, _ = measured_peaks()
    hbm = peaks["hbm_gbs"]

    def timeit(fn, reps=10, warm=3):
        with torch.cuda.stream(stream):
            for _ in range(warm):
                fn()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                fn()
            b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    # For inputs that fit in L2 (129 MB): write a 256 MB buffer before every repetition and
    # subtract the time of the writes alone, so each repetition starts from a cold L2.
    l2_flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timeit_cold(fn, reps=10):
        def body():
            l2_flush.zero_()
            fn()
        return timeit(body, reps=reps) - timeit(l2_flush.zero_, reps=reps)

    w13, s13, w2, s2, q, fsf = make_dequant_inputs()
    t = {k: torch.from_numpy(v).to(dev) for k, v in (("w13", w13), ("s13", s13), ("w2", w2), ("s2", s2),
                                                        ("q", q), ("fsf", fsf))}
    o13 = torch.empty((w13.shape[0], 2 * w13.shape[1]), dtype=torch.bfloat16, device=dev)
    o2 = torch.empty((w2.shape[0], 2 * w2.shape[1]), dtype=torch.bfloat16, device=dev)

    def deq():
        mx.mxfp4_dequant(t["w13"], t["s13"], o13, stream=stream)
        mx.mxfp4_dequant(t["w2"], t["s2"], o2, stream=stream)

    ms = timeit(deq)
    nbytes = w13.nbytes + s13.nbytes + w2.nbytes + s2.nbytes + (o13.numel() + o2.numel()) * 2
    res["mxfp4_dequant"] = {"GB/s": nbytes / ms / 1e6, "frac_hbm": nbytes / ms / 1e6 / hbm, "ms": ms,
                            "bytes": nbytes}
    # the same expert codes as NVFP4 (E4M3 per 16 columns + float32 global scale)
    n13, n2, g = make_nvfp4_scales()
    t["n13"], t["n2"] = torch.from_numpy(n13).to(dev), torch.from_numpy(n2).to(dev)

    def nvdeq():
        mx.nvfp4_dequant(t["w13"], t["n13"], g, o13, stream=stream)
        mx.nvfp4_dequant(t["w2"], t["n2"], g, o2, stream=stream)

    ms = timeit(nvdeq)
    nbytes = w13.nbytes + n13.nbytes + w2.nbytes + n2.nbytes + (o13.numel() + o2.numel()) * 2
    res["nvfp4_dequant"] = {"GB/s": nbytes / ms / 1e6, "frac_hbm": nbytes / ms / 1e6 / hbm, "ms": ms,
                            "bytes": nbytes}
    del o13, o2
    of = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    ms = timeit_cold(lambda: mx.fp8_block_dequant_128x128(t["q"], t["fsf"], of, stream=stream), reps=50)
    nbytes = q.nbytes + fsf.nbytes + of.numel() * 2
    res["fp8_dequant"] = {"GB/s": nbytes / ms / 1e6, "frac_hbm": nbytes / ms / 1e6 / hbm, "ms": ms,
                          "bytes": nbytes, "l2": "flushed before every repetition"}
    del t, of
    torch.cuda.empty_cache()
    # one dense GEMM (a projection) in both formats, against the FP4 tensor peak
    a, b, mx_sa, mx_sb, nv_sa, nv_sb, ga, gb = make_gemm_inputs()
    M, N, K = a.shape[0], b.shape[0], 2 * a.shape[1]
    g = {k: torch.from_numpy(v).to(dev) for k, v in (("a", a), ("b", b), ("mx_sa", mx_sa), ("nv_sa", nv_sa))}
    g["mx_sbt"] = torch.empty(mx.mxfp4_tiled_scales_bytes(N, K), dtype=torch.uint8, device=dev)
    mx.mxfp4_scales_to_tiled(torch.from_numpy(mx_sb).to(dev), g["mx_sbt"])
    g["nv_sbt"] = torch.empty(mx.nvfp4_tiled_scales_bytes(N, K), dtype=torch.uint8, device=dev)
    mx.nvfp4_scales_to_tiled(torch.from_numpy(nv_sb).to(dev), g["nv_sbt"])
    d = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    fp4_peak = fp4_peak_tflops(peaks)
    for name, fn in (("gemm_mxfp4", lambda: mx.mxfp4_gemm_bf16(g["a"], g["mx_sa"], g["b"], g["mx_sbt"], d,
                                                               stream=stream)),
                     ("gemm_nvfp4", lambda: mx.nvfp4_gemm_bf16(g["a"], g["nv_sa"], ga, g["b"], g["nv_sbt"], gb, d,
                                                               stream=stream))):
        ms = timeit_cold(fn, reps=20)
        tflops = 2.0 * M * N * K / ms / 1e9
        res[name] = {"shape": [M, N, K], "ms": ms, "TFLOP/s": tflops, "frac_fp4_peak": tflops / fp4_peak,
                     "l2": "flushed before every repetition"}
    # the fused q_a + kv projection: two weight matrices stacked along N, one global each
    seg = [1536, 576]
    Nf = sum(seg)
    df = torch.empty((M, Nf), dtype=torch.bfloat16, device=dev)
    bf = g["b"][:Nf]
    sbf = torch.empty(mx.nvfp4_tiled_scales_bytes(Nf, K), dtype=torch.uint8, device=dev)
    mx.nvfp4_scales_to_tiled(torch.from_numpy(np.ascontiguousarray(nv_sb[:Nf])).to(dev), sbf)
    ms = timeit_cold(lambda: mx.nvfp4_gemm_bf16_multi(g["a"], g["nv_sa"], ga, bf, sbf, [gb, 0.5 * gb], seg, df,
                                                      stream=stream), reps=20)
    tflops = 2.0 * M * Nf * K / ms / 1e9
    res["gemm_nvfp4_fused_projection"] = {"shape": [M, Nf, K], "segments": seg, "ms": ms, "TFLOP/s": tflops,
                                          "frac_fp4_peak": tflops / fp4_peak, "l2": "flushed before every repetition"}
    del g, d, df, sbf
    torch.cuda.empty_cache()
    for name in ("decode", "shared"):
        inp = make_config_inputs(name)
        c = CONFIGS[name]
        x = torch.from_numpy(inp.x).to(dev).view(torch.bfloat16)
        routed = inp.topk_ids is not None
        ids = torch.from_numpy(inp.topk_ids).to(dev) if routed else None
        w = torch.from_numpy(inp.topk_w).to(dev) if routed else None
        W = [torch.from_numpy(a).to(dev) for a in (inp.w13, inp.s13, inp.w2, inp.s2)]
        s13t = torch.empty(mx.mxfp4_tiled_scales_bytes(c["E"] * 2 * c["I"], c["H"]), dtype=torch.uint8, device=dev)
        s2t = torch.empty(mx.mxfp4_tiled_scales_bytes(c["E"] * c["H"], c["I"]), dtype=torch.uint8, device=dev)
        mx.mxfp4_scales_to_tiled(W[1].view(-1, c["H"] // 32), s13t)
        mx.mxfp4_scales_to_tiled(W[3].view(-1, c["I"] // 32), s2t)
        W = [W[0], s13t, W[2], s2t]
        out = torch.empty((c["T"], c["H"]), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(max(256, mx.moe_mxfp4_workspace_size(c["T"], c["H"], c["I"], c["E"], inp.K, routed)),
                         dtype=torch.uint8, device=dev)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

        def fwd(fused=False):
            flush.zero_()          # keep the weights out of L2 between repetitions
            mx.moe_mxfp4_forward(x, ids, w, *W, out, ws, stream=stream, scales_tiled=True, fused=fused)

        def fwd_fused():
            fwd(True)

        def only_flush():
            flush.zero_()

        ms = timeit(fwd, reps=20) - timeit(only_flush, reps=20)
        ms_fused = timeit(fwd_fused, reps=20) - timeit(only_flush, reps=20)
        # The same forwards replayed as CUDA graphs (the API is capture-safe), which removes
        # the host launch gaps between the multi-kernel forward's few short kernels.
        graphs = []
        for body in (fwd, fwd_fused, only_flush):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                body()
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=stream):
                body()
            graphs.append(g)
        t_flush = timeit(graphs[2].replay, reps=20)
        ms_graph = timeit(graphs[0].replay, reps=20) - t_flush
        ms_fused_graph = timeit(graphs[1].replay, reps=20) - t_flush
        pairs = int(((inp.topk_ids >= 0) & (inp.topk_ids < c["E"])).sum()) if routed else c["T"]
        touched = np.unique(inp.topk_ids).size if routed else 1
        wbytes = touched * (inp.w13[0].nbytes + inp.s13[0].nbytes + inp.w2[0].nbytes + inp.s2[0].nbytes)
        nbytes = wbytes + inp.x.nbytes * 2
        res[name] = {"ms": ms, "TFLOP/s": pairs * flops_per_pair(c["H"], c["I"]) / ms / 1e9,
                     "GB/s": nbytes / ms / 1e6, "frac_hbm": nbytes / ms / 1e6 / hbm, "algorithmic_bytes": nbytes,
                     "graph_ms": ms_graph, "graph_frac_hbm": nbytes / ms_graph / 1e6 / hbm,
                     "single_launch_ms": ms_fused, "single_launch_frac_hbm": nbytes / ms_fused / 1e6 / hbm,
                     "single_launch_graph_ms": ms_fused_graph,
                     "single_launch_graph_frac_hbm": nbytes / ms_fused_graph / 1e6 / hbm}
        del graphs
        del x, ids, w, W, out, ws, flush
        torch.cuda.empty_cache()
    res.update(measure_nvfp4_forward(mx, torch, dev, stream, timeit))
    res.update(measure_mxfp8_forward(mx, torch, dev, stream, timeit))
    return res


def measure_mxfp8_forward(mx, torch, dev, stream, timeit):
    """The routed prefill forward with MXFP8 activations over the same MXFP4 weights (the
    step's workload), against the FP8 tensor rate: kind::mxf8f6f4 runs at the E4M3 rate, one
    third of the FP4 one (nominal 4.5 : 13.5)."""
    inp = make_config_inputs("prefill")
    c = CONFIGS["prefill"]
    T, H, I, E, K = c["T"], c["H"], c["I"], c["E"], c["K"]
    x = torch.from_numpy(inp.x).to(dev).view(torch.bfloat16)
    ids = torch.from_numpy(inp.topk_ids).to(dev)
    w = torch.from_numpy(inp.topk_w).to(dev)
    w13, w2 = torch.from_numpy(inp.w13).to(dev), torch.from_numpy(inp.w2).to(dev)
    s13t = torch.empty(mx.mxfp4_tiled_scales_bytes(E * 2 * I, H), dtype=torch.uint8, device=dev)
    s2t = torch.empty(mx.mxfp4_tiled_scales_bytes(E * H, I), dtype=torch.uint8, device=dev)
    mx.mxfp4_scales_to_tiled(torch.from_numpy(inp.s13.reshape(-1, H // 32)).to(dev), s13t)
    mx.mxfp4_scales_to_tiled(torch.from_numpy(inp.s2.reshape(-1, I // 32)).to(dev), s2t)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(mx.moe_mxfp4w_mxfp8a_workspace_size(T, H, I, E, K, True), dtype=torch.uint8, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in ev:
        e.record(stream)              # create the underlying CUDA events

    def fwd(events=None):
        mx.moe_mxfp4w_mxfp8a_forward(x, ids, w, w13, s13t, w2, s2t, out, ws, stream=stream, events=events)

    ms = timeit(fwd, reps=20)
    fwd(ev)
    torch.cuda.synchronize()
    pairs = int(((inp.topk_ids >= 0) & (inp.topk_ids < E)).sum())
    flop = pairs * flops_per_pair(H, I)
    l1_ms = ev[2].elapsed_time(ev[3])
    l1_tflops = pairs * 2 * H * 2 * I / l1_ms / 1e9
    fp8_peak = fp4_peak_tflops(measured_peaks()[0]) / 3.0
    r = {"mxfp8_activation_forward": {
        "workload": "routed prefill T=8192, H=7168, I=3072, 48 experts, top-8, MXFP8 activations x MXFP4 weights",
        "ms": ms, "TFLOP/s": flop / ms / 1e9,
        "phases_ms": {k: ev[i].elapsed_time(ev[i + 1]) for i, k in
                      enumerate(("route", "quant_gather", "l1_gemm", "l2_gemm", "combine"))},
        "l1_TFLOP/s": l1_tflops, "l1_frac_fp8_peak": l1_tflops / fp8_peak,
        "fp8_peak_source": "measured bf16_tflops (burst) x 2 (nominal FP8:BF16)"}}
    del x, ids, w, w13, w2, s13t, s2t, out, ws
    torch.cuda.empty_cache()
    return r


def measure_nvfp4_forward(mx, torch, dev, stream, timeit):
    """The routed prefill forward with NVFP4 weights and activations (the same shapes, routing
    and x recipe as the MXFP4 step; E4M3 scales per 16, gate/up/down globals)."""
    inp = make_nvfp4_config_inputs("prefill")
    c = CONFIGS["prefill"]
    x = torch.from_numpy(inp.x).to(dev).view(torch.bfloat16)
    ids = torch.from_numpy(inp.topk_ids).to(dev)
    w = torch.from_numpy(inp.topk_w).to(dev)
    w13, w2, g13, g2 = (torch.from_numpy(a).to(dev) for a in (inp.w13, inp.w2, inp.g13, inp.g2))
    s13t = torch.empty(mx.nvfp4_tiled_scales_bytes(c["E"] * 2 * c["I"], c["H"]), dtype=torch.uint8, device=dev)
    s2t = torch.empty(mx.nvfp4_tiled_scales_bytes(c["E"] * c["H"], c["I"]), dtype=torch.uint8, device=dev)
    mx.nvfp4_scales_to_tiled(torch.from_numpy(inp.s13.reshape(-1, c["H"] // 16)).to(dev), s13t)
    mx.nvfp4_scales_to_tiled(torch.from_numpy(inp.s2.reshape(-1, c["I"] // 16)).to(dev), s2t)
    out = torch.empty((c["T"], c["H"]), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(mx.moe_nvfp4_workspace_size(c["T"], c["H"], c["I"], c["E"], c["K"], True), dtype=torch.uint8,
                     device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in ev:
        e.record(stream)              # create the underlying CUDA events

    def fwd(events=None):
        mx.moe_nvfp4_forward(x, ids, w, w13, s13t, g13, w2, s2t, g2, inp.x_global, inp.h_global, out, ws,
                             stream=stream, events=events)

    ms = timeit(fwd, reps=20)
    fwd(ev)
    torch.cuda.synchronize()
    pairs = int(((inp.topk_ids >= 0) & (inp.topk_ids < c["E"])).sum())
    flop = pairs * flops_per_pair(c["H"], c["I"])
    l1_ms = ev[2].elapsed_time(ev[3])
    l1_tflops = pairs * 2 * c["H"] * 2 * c["I"] / l1_ms / 1e9
    fp4_peak = fp4_peak_tflops(measured_peaks()[0])
    r = {"nvfp4_forward": {"workload": "routed prefill T=8192, H=7168, I=3072, 48 experts, top-8, NVFP4",
                           "ms": ms, "TFLOP/s": flop / ms / 1e9,
                           "phases_ms": {k: ev[i].elapsed_time(ev[i + 1]) for i, k in
                                         enumerate(("route", "quant_gather", "l1_gemm", "l2_gemm", "combine"))},
                           "l1_TFLOP/s": l1_tflops, "l1_frac_fp4_peak": l1_tflops / fp4_peak}}
    del x, ids, w, w13, w2, g13, g2, s13t, s2t, out, ws
    torch.cuda.empty_cache()
    return r


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the dequant/decode/shared context figures")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip timing the CPU oracle sample")
    ap.add_argument("--tokens", type=int, default=0,
                    help="prefill batch size other than 8192 (smaller cases for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
