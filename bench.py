"""Throughput of exact attention fwd+bwd on GB300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the whole hot path over one batch: fa_fwd (forward
kernel) then the three backward kernels (fa_bwd_preprocess, fa_bwd_main,
fa_bwd_dq_convert, which together are fa_bwd).  Workload: causal bf16
attention, B=2, H=16, N=8192, d=128, scale 1/sqrt(d), seeded N(0,1) inputs.
FLOPs per step follow the convention fwd = 4 B H N^2 d (halved for causal),
bwd = 2.5 x fwd.  Q, K, V and dO (256 MiB) exceed the 129 MB L2, so no flush.

--gpus N > 1 runs under torchrun, one process per GPU: the attention path has
no exchange step, so each rank runs an independent replica (weak scaling) and
`value` is the work of all ranks over the slowest rank's time.

--impl reference times the float64 CPU oracle on the host cores, one head of
the same workload per step (a bounded sample).

After the timed steps, the line's "side" object times the other training
shapes one by one (GPT-2-small-like layer, the fixed-16384-token sweep, the
FP8 forward); --no-side skips them.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = dict(name="long_causal_B2_H16_N8192_d128", B=2, H=16, N=8192, d=128, causal=True, seed=3)
METRIC = "attention fwd+bwd TFLOPS (bf16, causal, d=128, 1xGB300)"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


def flops_step(B, H, N, d, causal):
    fwd = 4.0 * B * H * N * N * d / (2.0 if causal else 1.0)
    return fwd, 2.5 * fwd


def window_pairs(N, W):
    """(query, key) pairs a sliding window of W keys leaves visible over N
    rows: row i sees keys i - W + 1 .. i that exist, min(i + 1, W) of them."""
    return N * W - W * (W - 1) // 2 if N >= W else N * (N + 1) // 2


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# Source files each timed kernel is compiled from (its translation unit and
# the headers it includes).
KERNEL_SOURCES = {
    "fa_fwd": ["fa_fwd.cu", "fa_common.cuh", "fa_host.h"],
    "fa_bwd_preprocess": ["fa_bwd.cu", "fa_common.cuh", "fa_host.h"],
    "fa_bwd_main": ["fa_bwd.cu", "fa_common.cuh", "fa_host.h"],
    "fa_bwd_dq_convert": ["fa_bwd.cu", "fa_common.cuh", "fa_host.h"],
}


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_76_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's sources changed since those counters were taken."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        rec = json.load(f)
    ent = rec.get("kernels", {}).get(kernel)
    if not ent or kernel not in KERNEL_SOURCES or ent.get("source_hash") != kernel_source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}


def max_over_ranks(x: float, device) -> float:
    """The largest value of x over all ranks (x itself on one process)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_step: float, steps: int, ms_slowest: float) -> float:
    """Work of all ranks (independent replicas) over the slowest rank's time."""
    return world * flops_per_step * steps / (ms_slowest * 1e-3) / 1e12


def cpu_oracle_sample(heads, N, d, causal, seed):
    """Times the float64 oracle (forward + backward) on `heads` heads of the
    workload; returns (seconds, flops of those heads)."""
    import oracle
    from exact_attention_76_gb300 import inputs

    q, k, v, do = inputs.draw_bf16(1, heads, N, d, seed)
    scale = 1.0 / math.sqrt(d)
    t0 = time.perf_counter()
    oracle.forward(q, k, v, causal, scale)
    oracle.backward(q, k, v, do, causal, scale)
    dt = time.perf_counter() - t0
    f, b = flops_step(1, heads, N, d, causal)
    return dt, f + b


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    W = WORKLOAD
    for _ in range(args.warmup):
        cpu_oracle_sample(1, W["N"], W["d"], W["causal"], W["seed"])
    times, fl = [], 0.0
    for _ in range(args.steps):
        dt, fl = cpu_oracle_sample(1, W["N"], W["d"], W["causal"], W["seed"])
        times.append(dt)
    tot = sum(times)
    value = fl * args.steps / tot / 1e12
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": W["name"], "B": W["B"], "H": W["H"], "N": W["N"], "d": W["d"],
                   "causal": W["causal"], "sample": "1 of 32 heads per step"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "one (batch, head) of the workload per step, fwd+bwd in float64"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_ours(args):
    import torch
    import torch.distributed as dist

    from exact_attention_76_gb300 import api, inputs
    from exact_attention_76_gb300 import build as _build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if rank == 0:
        _build.build()
    if world > 1:
        dist.barrier()
    W = dict(WORKLOAD)
    if args.shape:  # profiling cases only; the default is the workload above
        W["B"], W["H"], W["N"], W["d"] = (int(x) for x in args.shape.split(","))
        W["name"] = f"causal_B{W['B']}_H{W['H']}_N{W['N']}_d{W['d']}"
    B, H, N, d, causal = W["B"], W["H"], W["N"], W["d"], W["causal"]
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = inputs.draw_bf16(B, H, N, d, W["seed"])
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    Dv = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    acc = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    kernels = ["fa_fwd", "fa_bwd_preprocess", "fa_bwd_main", "fa_bwd_dq_convert"]

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        api.fa_fwd(qd, kd, vd, causal, scale, o=o, lse=lse)
        if ev is not None:
            ev[1].record(stream)
        api.fa_bwd_preprocess(o, dod, D=Dv, dq_acc=acc)
        if ev is not None:
            ev[2].record(stream)
        api.fa_bwd_main(qd, kd, vd, lse, dod, Dv, acc, causal, scale, dk=dk, dv=dv)
        if ev is not None:
            ev[3].record(stream)
        api.fa_bwd_dq_convert(acc, scale, dq=dq)
        if ev is not None:
            ev[4].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if api.fa_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    # ---- timed region: K steps, CUDA events on the launching stream
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        stop.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms_total = start.elapsed_time(stop)
    per_kernel = {n: sum(e[j].elapsed_time(e[j + 1]) for e in evs) / args.steps for j, n in enumerate(kernels)}
    ms_total = max_over_ranks(ms_total, "cuda")
    if api.fa_device_error() != 0:
        raise RuntimeError("device error word set during the timed region")

    fwd_fl, bwd_fl = flops_step(B, H, N, d, causal)
    step_fl = fwd_fl + bwd_fl
    ms_step = ms_total / args.steps
    value = whole_job_tflops(world, step_fl, args.steps, ms_total)

    # ---- end to end through the same API with pinned host buffers
    # Every step copies its inputs (Q, K, V, dO) from pinned host memory and
    # its results (O, L, dQ, dK, dV) back, inside the timed region.  Three
    # streams pipeline consecutive steps: step i+1's inputs go in and step
    # i-1's results come out while step i computes; device buffers alternate.
    hq, hk, hv, hdo = (t.pin_memory() for t in (q, k, v, do))
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    e2e_steps = max(3, min(args.steps, 20))
    ms_e2e = float("nan")
    d2h = 0
    if not args.no_e2e:
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        bufs = []
        for _ in range(2):
            ins = [torch.empty_like(t) for t in (qd, kd, vd, dod)]
            outs = [torch.empty_like(o), torch.empty_like(lse), torch.empty_like(dq), torch.empty_like(dk),
                    torch.empty_like(dv)]
            ws = torch.empty(api.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
            bufs.append((ins, outs, ws))
        hout = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in bufs[0][1]] for _ in range(2)]
        d2h = sum(t.numel() * t.element_size() for t in hout[0])

        def run_pipeline(n):
            in_ready = [torch.cuda.Event() for _ in range(n)]
            done = [torch.cuda.Event() for _ in range(n)]
            out_done = [torch.cuda.Event() for _ in range(n)]
            for i in range(n):
                ins, outs, ws = bufs[i % 2]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(done[i - 2])      # compute i-2 finished with these inputs
                    for h_, d_ in zip((hq, hk, hv, hdo), ins):
                        d_.copy_(h_, non_blocking=True)
                    in_ready[i].record(s_in)
                with torch.cuda.stream(s_cmp):
                    s_cmp.wait_event(in_ready[i])
                    if i >= 2:
                        s_cmp.wait_event(out_done[i - 2])  # results of i-2 copied out of these outputs
                    api.fa_fwd(ins[0], ins[1], ins[2], causal, scale, o=outs[0], lse=outs[1], stream=s_cmp)
                    api.fa_bwd(ins[0], ins[1], ins[2], outs[0], outs[1], ins[3], causal, scale, dq=outs[2],
                               dk=outs[3], dv=outs[4], workspace=ws, stream=s_cmp)
                    done[i].record(s_cmp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done[i])
                    for h_, d_ in zip(hout[i % 2], outs):
                        h_.copy_(d_, non_blocking=True)
                    out_done[i].record(s_out)
            return out_done[n - 1]

        run_pipeline(2)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        s_cmp.wait_event(e0)
        s_out.wait_event(e0)
        last = run_pipeline(e2e_steps)
        s_in.wait_event(last)
        e1.record(s_in)
        torch.cuda.synchronize()
        ms_e2e = e0.elapsed_time(e1)
    ms_e2e = max_over_ranks(ms_e2e, "cuda") if not args.no_e2e else ms_e2e
    e2e_value = None if args.no_e2e else whole_job_tflops(world, step_fl, e2e_steps, ms_e2e)

    # ---- roofline of the dominant kernel
    # The timed region lasts tens of milliseconds at full clock, so a kernel's
    # fraction is taken against the burst bf16 figure (cuBLAS timed alone);
    # the sustained one (seconds under the power cap) is reported beside it.
    peaks, peak_src = measured_peaks()
    fl_per_kernel = {"fa_fwd": fwd_fl, "fa_bwd_main": bwd_fl}
    dom = max(per_kernel, key=per_kernel.get)
    peak = peaks["bf16_tflops"]
    peak_sus = peaks.get("bf16_tflops_sustained", peak)
    if dom in fl_per_kernel:
        achieved = fl_per_kernel[dom] / (per_kernel[dom] * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": recorded_traffic(dom), "kernel": dom,
                "peak_source": f"{peak_src} bf16 burst (the timed region is tens of ms at full clock)",
                "peak_sustained": peak_sus, "frac_of_sustained": achieved / peak_sus,
                "step_frac": value / world / peak}
    else:
        roof = {"bound": "hbm", "achieved": None, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": None,
                "traffic": recorded_traffic(dom), "kernel": dom}
    # secondary figures: every kernel's share and the memory-bound kernels' GB/s
    rows = B * H * N
    hbm_bytes = {"fa_bwd_preprocess": rows * (2 * d * 2 + 4 + 4 * d), "fa_bwd_dq_convert": rows * (4 * d + 2 * d)}
    kernel_stats = {}
    for n, ms in per_kernel.items():
        ent = {"ms": ms, "share": ms / sum(per_kernel.values())}
        if n in fl_per_kernel:
            ent["tflops"] = fl_per_kernel[n] / (ms * 1e-3) / 1e12
            ent["frac_of_bf16_burst"] = ent["tflops"] / peak
        if n in hbm_bytes:
            ent["gbs"] = hbm_bytes[n] / (ms * 1e-3) / 1e9
            ent["frac_of_hbm"] = ent["gbs"] / peaks["hbm_gbs"]
        kernel_stats[n] = ent

    # ---- the other training shapes (outside the timed region above)
    side = None
    if not args.no_side and rank == 0:
        side = side_measurements(peaks, peak_src)

    in_bytes = 4 * B * H * N * d * 2
    l2_note = (f"no flush: Q,K,V,dO are {in_bytes / 2**20:.0f} MiB, larger than L2" if in_bytes > L2_BYTES else
               f"no flush: Q,K,V,dO are {in_bytes / 2**20:.0f} MiB and fit in L2 (a profiling shape)")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": W["name"], "B": B, "H": H, "N": N, "d": d, "causal": causal,
                   "scale": "1/sqrt(d)", "l2": l2_note,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roof,
        "kernels": kernel_stats,
        "e2e": None if e2e_value is None else {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                                               "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": 4 * args.steps,
        "clocks": clk.summary(),
    }
    if side is not None:
        line["side"] = side
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        heads = 2
        dt, fl = cpu_oracle_sample(heads, N, d, causal, W["seed"])
        line["cpu_baseline"] = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
                                "kind": "oracle",
                                "sample": f"{heads} of {B * H} heads, fwd+bwd in float64 ({dt:.1f} s)"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def _time_iters(fn, iters, flush=None, warmup=3):
    """Mean device time (ms) of fn() over `iters` calls, each bracketed by CUDA
    events on the current stream; flush() (an L2 flush) runs between calls,
    outside the events, when the call's inputs fit in L2."""
    import torch

    stream = torch.cuda.current_stream()
    for _ in range(warmup):  # as the timed calls run, flush included
        if flush is not None:
            flush()
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for e0, e1 in evs:
        if flush is not None:
            flush()
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return sum(e0.elapsed_time(e1) for e0, e1 in evs) / iters


L2_BYTES = 129 * 1000 * 1000


def side_measurements(peaks, peak_src, iters=8):
    """The other training shapes of the workload set, each timed on its own
    (not part of the step above): the GPT-2-small-like layer (B=4, H=12,
    N=1024, d=64), the fixed-16384-token sweep (N = 512 .. 16384 at H=32 d=64
    and H=16 d=128) and the FP8 forward (B=1, H=16, N=16384, d=128, Q and K
    Hadamard-rotated before per-tensor e4m3 storage, the configuration that
    passes the FP8 error gate).  Inputs are seeded N(0,1) draws made on the
    device; a 256 MiB write flushes L2 between iterations whenever a case's
    inputs fit in it."""
    import torch

    from exact_attention_76_gb300 import api, inputs

    bf16_peak = peaks["bf16_tflops"]
    fp8_peak = 2.0 * bf16_peak
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def flush():
        scratch.zero_()

    out = {"peak_bf16": bf16_peak, "peak_fp8": fp8_peak,
           "peak_source": f"{peak_src} bf16 burst; fp8 = 2 x bf16 (nominal ratio)", "cases": {}}

    def bf16_case(name, B, H, N, d, causal, seed):
        g = torch.Generator(device="cuda").manual_seed(seed)
        q, k, v, do = (torch.randn(B, H, N, d, device="cuda", generator=g).to(torch.bfloat16) for _ in range(4))
        scale = 1.0 / math.sqrt(d)
        o = torch.empty_like(q)
        lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(api.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
        fl = None if 4 * q.numel() * 2 > L2_BYTES else flush
        ms_f = _time_iters(lambda: api.fa_fwd(q, k, v, causal, scale, o=o, lse=lse), iters, fl)
        ms_b = _time_iters(lambda: api.fa_bwd(q, k, v, o, lse, do, causal, scale, dq=dq, dk=dk, dv=dv,
                                              workspace=ws), iters, fl)

        def step():
            api.fa_fwd(q, k, v, causal, scale, o=o, lse=lse)
            api.fa_bwd(q, k, v, o, lse, do, causal, scale, dq=dq, dk=dk, dv=dv, workspace=ws)

        ms_s = _time_iters(step, iters, fl)
        f, b = flops_step(B, H, N, d, causal)
        # fwd_ms and bwd_ms time each call on its own (L2 flushed before each
        # where the inputs fit in it); step_ms times the forward and backward
        # back to back in one region, as the headline step is timed (L2
        # flushed between steps only).
        out["cases"][name] = {
            "B": B, "H": H, "N": N, "d": d, "causal": causal, "l2_flush": fl is not None,
            "fwd_ms": ms_f, "bwd_ms": ms_b, "fwd_tflops": f / ms_f / 1e9, "bwd_tflops": b / ms_b / 1e9,
            "fwdbwd_tflops": (f + b) / (ms_f + ms_b) / 1e9, "fwdbwd_frac": (f + b) / (ms_f + ms_b) / 1e9 / bf16_peak,
            "step_ms": ms_s, "step_tflops": (f + b) / ms_s / 1e9, "step_frac": (f + b) / ms_s / 1e9 / bf16_peak}

    w = inputs.GPT2
    for causal in (True, False):
        bf16_case(f"gpt2small_B4_H12_N1024_d64_{'c' if causal else 'nc'}", w.B, w.H, w.N, w.d, causal, w.seed)
    for d in (64, 128):
        for causal in (True, False):
            for sw in inputs.sweep_workloads(causal, d):
                bf16_case(sw.name, sw.B, sw.H, sw.N, sw.d, causal, sw.seed)
    torch.cuda.synchronize()

    w = inputs.FP8
    q, k, v = (t.cuda() for t in inputs.draw_outlier_fp32(w.B, w.H, w.N, w.d, w.seed))
    (q8, dsq), (k8, dsk), (v8, dsv) = (api.fa_fp8_quantize(q, True), api.fa_fp8_quantize(k, True),
                                       api.fa_fp8_quantize(v, False))
    del q, k, v
    o = torch.empty(w.B, w.H, w.N, w.d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device="cuda")
    for causal in (True, False):
        ms = _time_iters(lambda: api.fa_fwd_fp8(q8, k8, v8, dsq, dsk, dsv, causal, w.scale, o=o, lse=lse), iters,
                         flush)
        f, _ = flops_step(w.B, w.H, w.N, w.d, causal)
        out["cases"][f"fp8_hadamard_B1_H16_N16384_d128_{'c' if causal else 'nc'}"] = {
            "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": causal, "l2_flush": True, "fwd_ms": ms,
            "fwd_tflops": f / ms / 1e9, "fwd_frac": f / ms / 1e9 / fp8_peak}
    if api.fa_device_error() != 0:
        raise RuntimeError("device error word set during the side measurements")
    return out


def run_decode(args):
    """Decode against a key/value cache (a side measurement, not the bench's
    workload): K/V read bandwidth of fa_decode, timed with CUDA events on the
    launching stream; the cache (2 B H_kv N d bf16) is meant to exceed L2."""
    import torch

    from exact_attention_76_gb300 import api
    from exact_attention_76_gb300 import build as _build

    _build.build()
    B, H, Hkv, N, d = (int(x) for x in args.decode.split(","))
    g = torch.Generator(device="cuda").manual_seed(1)
    q = torch.randn(B, H, d, device="cuda", generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, N, d, device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, N, d, device="cuda", generator=g).to(torch.bfloat16)
    ws = torch.empty(api.fa_decode_workspace_size(B, H, Hkv, N, d), dtype=torch.uint8, device="cuda")
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, dtype=torch.float32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    stream = torch.cuda.current_stream()
    for _ in range(max(args.warmup, 3)):
        api.fa_decode(q, k, v, scale, o=o, lse=lse, workspace=ws, stream=stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        api.fa_decode(q, k, v, scale, o=o, lse=lse, workspace=ws, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    kv_bytes = 2.0 * B * Hkv * N * d * 2
    gbs = kv_bytes / ms / 1e6
    peaks, src = measured_peaks()
    print(json.dumps({"metric": "decode K/V read bandwidth", "value": gbs, "unit": "GB/s", "steps": args.steps,
                      "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
                      "config": {"workload": f"decode_B{B}_H{H}_Hkv{Hkv}_N{N}_d{d}", "kv_bytes": kv_bytes},
                      "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                   "frac": gbs / peaks["hbm_gbs"], "peak_source": src}}), flush=True)
    return 0


def run_fp8(args):
    """FP8 e4m3 forward on the FP8 workload (a side measurement, not the bench's
    workload): B=1, H=16, N=16384, d=128, Q, K, V drawn N(0,1) with 0.1 % of the
    entries scaled by 10, stored as e4m3 by the library's quantiser with Q and
    K Hadamard-rotated first (the configuration that passes the FP8 error
    gate): one scale per tensor, or with --fp8-blocks one per 128 rows of Q
    and per 64 rows of K and V.  --fp8-shape B,H,N,d replaces the shape.  The
    default shape's codes (100 MB) fit in L2, so a 256 MiB write flushes it
    between calls; each call is timed with CUDA events on the launching
    stream, against the fp8 peak (the measured bf16 figure times 2, the
    nominal fp8:bf16 ratio)."""
    import torch

    from exact_attention_76_gb300 import api, inputs
    from exact_attention_76_gb300 import build as _build

    _build.build()
    causal = args.fp8 == "causal"
    B, H, N, d = (int(x) for x in args.fp8_shape.split(","))
    q, k, v = (t.cuda() for t in inputs.draw_outlier_fp32(B, H, N, d, seed=4))
    if args.fp8_blocks:
        (q8, dq), (k8, dk), (v8, dv) = (api.fa_fp8_quantize_blocks(q, True, api.FP8_BLOCK_Q),
                                        api.fa_fp8_quantize_blocks(k, True, api.FP8_BLOCK_KV),
                                        api.fa_fp8_quantize_blocks(v, False, api.FP8_BLOCK_KV))
        fwd, scales = api.fa_fwd_fp8_blocks, "block scales (128 rows of Q, 64 of K and V)"
    else:
        (q8, dq), (k8, dk), (v8, dv) = (api.fa_fp8_quantize(q, True), api.fa_fp8_quantize(k, True),
                                        api.fa_fp8_quantize(v, False))
        fwd, scales = api.fa_fwd_fp8, "per-tensor scales"
    del q, k, v
    o = torch.empty(B, H, N, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    stream = torch.cuda.current_stream()
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    ms = _time_iters(lambda: fwd(q8, k8, v8, dq, dk, dv, causal, scale, o=o, lse=lse, stream=stream), args.steps,
                     flush=scratch.zero_, warmup=max(args.warmup, 3))
    fl, _ = flops_step(B, H, N, d, causal)
    tflops = fl / ms / 1e9
    peaks, src = measured_peaks()
    peak = 2.0 * peaks["bf16_tflops"]
    tag = f"fp8_B{B}_H{H}_N{N}_d{d}_{args.fp8}" + ("_blocks" if args.fp8_blocks else "")
    print(json.dumps({"metric": f"attention fwd TFLOPS (fp8 e4m3, {scales}, d={d}, 1xGB300)",
                      "value": tflops, "unit": "TFLOP/s", "steps": args.steps, "ms_per_step": ms,
                      "higher_is_better": True, "dtype": "e4m3", "data": "synthetic",
                      "config": {"workload": tag, "l2": "flushed"},
                      "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                                   "frac": tflops / peak, "peak_source": src + " bf16 burst x 2 (fp8:bf16)"}}),
          flush=True)
    return 0


def run_quant(args):
    """The FP8 quantisers on the FP8 workload's tensor shape (a side
    measurement, not the bench's workload): B=1, H=16, N=16384, d=128, the
    outlier draws of Q as fp32 and as bf16 input, per tensor and per 128-row
    block, each with and without the Hadamard rotation.  Bytes per call: the
    input read once and the e4m3 codes written (the per-tensor form reads its
    input twice, for max|y| and for the codes, so its ceiling lies below the
    copy figure).  A 256 MiB write flushes L2 between calls; each call is
    timed with CUDA events on the launching stream."""
    import torch

    from exact_attention_76_gb300 import api, inputs
    from exact_attention_76_gb300 import build as _build

    _build.build()
    B, H, N, d, block_rows = 1, 16, 16384, 128, 128
    x32 = inputs.draw_outlier_fp32(B, H, N, d, seed=4)[0].cuda()
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    peaks, src = measured_peaks()
    cases = {}
    for x in (x32, x32.to(torch.bfloat16)):
        codes = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
        desc = torch.empty(1, dtype=torch.float32, device="cuda")
        desc_b = torch.empty(B * H, N // block_rows, dtype=torch.float32, device="cuda")
        nbytes = x.numel() * (x.element_size() + 1)
        for rot in (False, True):
            for form, fn in (("tensor", lambda: api.fa_fp8_quantize(x, rot, codes=codes, descale=desc,
                                                                    stream=stream)),
                             ("blocks128", lambda: api.fa_fp8_quantize_blocks(x, rot, block_rows, codes=codes,
                                                                              descale=desc_b, stream=stream))):
                ms = _time_iters(fn, args.steps, flush=scratch.zero_, warmup=max(args.warmup, 3))
                gbs = nbytes / ms / 1e6
                name = f"{form}_{'fp32' if x.dtype == torch.float32 else 'bf16'}{'_rot' if rot else ''}"
                cases[name] = {"ms": ms, "GB/s": gbs, "frac": gbs / peaks["hbm_gbs"]}
    best = max(c["GB/s"] for c in cases.values())
    print(json.dumps({"metric": "fp8 quantiser throughput (input read once + codes written)", "value": best,
                      "unit": "GB/s", "steps": args.steps, "higher_is_better": True, "dtype": "f32",
                      "data": "synthetic", "config": {"workload": f"fp8q_B{B}_H{H}_N{N}_d{d}", "l2": "flushed"},
                      "cases": cases, "peak": peaks["hbm_gbs"], "peak_source": src}), flush=True)
    return 0


def run_variant(args):
    """Grouped-query or sliding-window attention, forward + backward (a side
    measurement, not the bench's workload): --gqa B,H,Hkv,N,d (causal) or
    --window B,H,N,d,W.  Inputs are seeded N(0,1) draws made on the device;
    the forward, the backward and the two back to back are each timed with
    CUDA events on the launching stream, and a 256 MiB write flushes L2
    between calls when the inputs fit in it.  FLOPs: grouped-query attention
    counts as H full heads under the causal convention; the window counts its
    visible pairs only (row i sees min(i + 1, W) keys), backward 2.5 x
    forward."""
    import torch

    from exact_attention_76_gb300 import api
    from exact_attention_76_gb300 import build as _build

    _build.build()
    if args.gqa:
        B, H, Hkv, N, d = (int(x) for x in args.gqa.split(","))
        W = 0
    else:
        B, H, N, d, W = (int(x) for x in args.window.split(","))
        Hkv = H
    g = torch.Generator(device="cuda").manual_seed(1)
    q, do = (torch.randn(B, H, N, d, device="cuda", generator=g).to(torch.bfloat16) for _ in range(2))
    k, v = (torch.randn(B, Hkv, N, d, device="cuda", generator=g).to(torch.bfloat16) for _ in range(2))
    scale = 1.0 / math.sqrt(d)
    o, lse = torch.empty_like(q), torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if W:
        ws = torch.empty(api.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")

        def fwd():
            api.fa_fwd_window(q, k, v, W, scale, o=o, lse=lse)

        def bwd():
            api.fa_bwd_window(q, k, v, o, lse, do, W, scale, dq=dq, dk=dk, dv=dv, workspace=ws)

        f = 4.0 * B * H * d * window_pairs(N, W)
        name = f"window{W}_B{B}_H{H}_N{N}_d{d}"
    else:
        ws = torch.empty(api.fa_bwd_gqa_workspace_size(B, H, Hkv, N, d), dtype=torch.uint8, device="cuda")

        def fwd():
            api.fa_fwd_gqa(q, k, v, True, scale, o=o, lse=lse)

        def bwd():
            api.fa_bwd_gqa(q, k, v, o, lse, do, True, scale, dq=dq, dk=dk, dv=dv, workspace=ws)

        f, _ = flops_step(B, H, N, d, True)
        name = f"gqa_B{B}_H{H}_Hkv{Hkv}_N{N}_d{d}_c"
    b = 2.5 * f
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    in_bytes = (2 * B * H + 2 * B * Hkv) * N * d * 2
    fl = scratch.zero_ if in_bytes <= L2_BYTES else None
    warm = max(args.warmup, 3)
    ms_f = _time_iters(fwd, args.steps, fl, warm)
    ms_b = _time_iters(bwd, args.steps, fl, warm)
    ms_s = _time_iters(lambda: (fwd(), bwd()), args.steps, fl, warm)
    peaks, src = measured_peaks()
    step_tflops = (f + b) / ms_s / 1e9
    print(json.dumps({"metric": "attention fwd+bwd TFLOPS (bf16)", "value": step_tflops, "unit": "TFLOP/s",
                      "steps": args.steps, "ms_per_step": ms_s, "higher_is_better": True, "dtype": "bf16",
                      "data": "synthetic", "config": {"workload": name, "l2": "flushed" if fl else "inputs > L2"},
                      "fwd_ms": ms_f, "bwd_ms": ms_b, "fwd_tflops": f / ms_f / 1e9, "bwd_tflops": b / ms_b / 1e9,
                      "roofline": {"bound": "tensor", "achieved": step_tflops, "peak": peaks["bf16_tflops"],
                                   "unit": "TFLOP/s", "frac": step_tflops / peaks["bf16_tflops"],
                                   "peak_source": src + " bf16 burst"}}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling runs)")
    ap.add_argument("--no-side", action="store_true", help="skip the other training shapes (profiling runs)")
    ap.add_argument("--shape", default="", help="B,H,N,d of a causal profiling case instead of the workload")
    ap.add_argument("--decode", default="", help="B,H,Hkv,N,d: time fa_decode instead (side measurement)")
    ap.add_argument("--mufu", action="store_true", help="measure the special-function unit's exp2 rate")
    ap.add_argument("--fp8", choices=["full", "causal"], default="",
                    help="time the FP8 forward on B=1 H=16 N=16384 d=128 instead (side measurement)")
    ap.add_argument("--fp8-blocks", action="store_true", help="with --fp8: block-scaled codes and fa_fwd_fp8_blocks")
    ap.add_argument("--fp8-shape", default="1,16,16384,128", help="with --fp8: B,H,N,d")
    ap.add_argument("--gqa", default="", help="B,H,Hkv,N,d: time grouped-query fwd+bwd instead (side measurement)")
    ap.add_argument("--window", default="", help="B,H,N,d,W: time sliding-window fwd+bwd instead (side measurement)")
    ap.add_argument("--quant", action="store_true",
                    help="time the FP8 quantisers on the FP8 workload's tensor shape instead (side measurement)")
    args = ap.parse_args()
    if args.quant:
        return run_quant(args)
    if args.gqa or args.window:
        return run_variant(args)
    if args.decode:
        return run_decode(args)
    if args.fp8:
        return run_fp8(args)
    if args.mufu:
        from exact_attention_76_gb300 import api
        from exact_attention_76_gb300 import build as _build
        _build.build()
        rate = api.fa_measure_ex2_rate()
        print(json.dumps({"metric": "ex2 rate", "value": rate, "unit": "results/clock/SM",
                          "note": "2 CTAs x 512 threads per SM, 8 independent ex2->FMA chains per thread"}))
        return 0
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
