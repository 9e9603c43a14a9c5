#!/usr/bin/env python
"""Benchmark of the quantised mixed-precision hot path on GB300.

A step is one INT8 x INT4 GEMM with the fused per-column dequantisation at
M = N = K = 4096 (A int8 uniform in [-128, 127], B int4 uniform in [-8, 7]
packed in the interleaved layout, fp16 scale uniform in [1e-3, 1e-2], fp16
output), called through the library's C ABI.  Inputs are resident in HBM.
The K timed steps cycle through 3 distinct input sets (168 MiB together,
more than the 129 MB L2), are captured once as a CUDA graph and replayed
inside the timed region (so the time is device time, not Python launch
overhead); CUDA events on the launching stream bracket the replay.

The M = 1 fp16 x INT4 GEMV of an N = 11008, K = 4096 layer ("gemv") is timed
the same way as a stack of 8 layers with distinct weights (180 MB, read from
HBM), as a decode step streams them; single-launch times with an L2 flush
before each launch are reported beside it, and the other workloads follow
("paths").

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl bq|reference]

With N > 1 (launched by torch.distributed.run) every rank runs its own copy of
the workload (independent problems, no collective on the data path) and the
reported value is the work of all ranks divided by the slowest rank's time.
--impl reference times the CPU oracle (the plain definition of the method)
on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "INT8xINT4 GEMM TOPS & f16xINT4 GEMV GB/s at 1 GB300; % of int8/HBM roofline"
WORKLOAD = ("INT8xINT4 GEMM with fused per-column fp16 dequant, M=N=K=4096 "
            "(A int8 U[-128,127], B int4 U[-8,7] interleaved-packed, scale fp16 U[1e-3,1e-2], C fp16), seed 0")
GEMV_WORKLOAD = "fp16 x INT4 GEMV, M=1, N=11008, K=4096 (X fp16 N(0,1), W int4 packed, scale = absmax/7 of N(0,0.02))"
M2 = N2 = K2 = 4096
OPS2 = 2 * M2 * N2 * K2
FLUSH_BYTES = 512 * 2 ** 20
GEMV_LAYERS = 8


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["bq", "reference"], default="bq")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-paths", action="store_true")
    p.add_argument("--profile", choices=sorted(PROFILES),
                   help="run one workload a few times through the C ABI and exit (for ncu captures)")
    return p.parse_args()


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def source_sha(*rel):
    h = hashlib.sha256()
    for r in rel:
        with open(os.path.join(ROOT, r), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """Per-launch DRAM traffic from the committed ncu summary, only if the
    kernel's sources are unchanged since it was taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f).get(kernel)
    if not t:
        return None
    if t.get("source_sha") != source_sha(*t["sources"]):
        return None
    return t.get("traffic_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.proc or not self.tmp:
            return None
        with open(self.tmp.name) as f:
            rows = [r for r in csv.reader(f) if len(r) >= 9]
        os.unlink(self.tmp.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip() == "Active"})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def flush_l2(flush):
    """Write one buffer larger than L2, then read another one: the write evicts
    whatever the previous step left in L2, and the read evicts (writes back)
    the dirty lines of that write, so the timed step starts from a cold L2
    without paying for someone else's write-backs."""
    w, r = flush
    w.zero_()
    r.max()


def time_steps(torch, fn, steps, warmup, flush, stream):
    """Per-step device time (ms) with CUDA events on the launching stream; L2
    flushed before every step, outside the events."""
    for _ in range(warmup):
        flush_l2(flush)
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s, e in evs:
        flush_l2(flush)
        s.record(stream)
        fn()
        e.record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


def e2e_pipelined(torch, bq, A_h, Bp_h, sc_h, dev, steps, warmup):
    """End-to-end time of `steps` GEMM steps whose inputs start on the host and
    whose result ends on the host, in a three-stage software pipeline (upload,
    GEMM, download on their own streams, three device buffer sets), and the
    same steps run one after another on one stream.  Returns both totals (ms)."""
    nset = 3
    A = [torch.empty_like(A_h, device=dev) for _ in range(nset)]
    B = [torch.empty_like(Bp_h, device=dev) for _ in range(nset)]
    S = [torch.empty_like(sc_h, device=dev) for _ in range(nset)]
    C = [torch.empty((A_h.shape[0], Bp_h.shape[0]), dtype=torch.float16, device=dev) for _ in range(nset)]
    C_h = [torch.empty((A_h.shape[0], Bp_h.shape[0]), dtype=torch.float16).pin_memory() for _ in range(nset)]
    up, comp, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    up_done, comp_done, down_done = ([ev() for _ in range(nset)] for _ in range(3))
    used = [False] * nset

    def run(n):
        for i in range(n):
            j = i % nset
            if used[j]:
                up.wait_event(comp_done[j])          # the GEMM that read set j is done
            with torch.cuda.stream(up):
                A[j].copy_(A_h, non_blocking=True)
                B[j].copy_(Bp_h, non_blocking=True)
                S[j].copy_(sc_h, non_blocking=True)
                up_done[j].record(up)
            comp.wait_event(up_done[j])
            if used[j]:
                comp.wait_event(down_done[j])        # set j's previous result has left the device
            with torch.cuda.stream(comp):
                bq.bq_gemm_i8xi4(A[j], B[j], "interleaved", col_scale=S[j], out=C[j])
                comp_done[j].record(comp)
            down.wait_event(comp_done[j])
            with torch.cuda.stream(down):
                C_h[j].copy_(C[j], non_blocking=True)
                down_done[j].record(down)
            used[j] = True

    run(warmup)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(up)
    run(steps)
    up.wait_stream(comp)
    up.wait_stream(down)
    end.record(up)
    torch.cuda.synchronize()
    pipelined = start.elapsed_time(end)

    s = torch.cuda.current_stream()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(s)
    for _ in range(steps):
        A[0].copy_(A_h, non_blocking=True)
        B[0].copy_(Bp_h, non_blocking=True)
        S[0].copy_(sc_h, non_blocking=True)
        bq.bq_gemm_i8xi4(A[0], B[0], "interleaved", col_scale=S[0], out=C[0])
        C_h[0].copy_(C[0], non_blocking=True)
    s1.record(s)
    torch.cuda.synchronize()
    return pipelined, s0.elapsed_time(s1)


def capture(torch, fn):
    """Capture fn's launches (on a side stream) into a CUDA graph."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g.replay()                       # first replay (untimed)
    torch.cuda.synchronize()
    return g


def time_graph(torch, g, reps, stream):
    """Median device time (ms) of one replay of g."""
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def max_over_ranks(torch, values, device, world):
    """Per-rank timings -> the slowest rank's, element by element (MAX
    all-reduce over the default process group); unchanged for one rank."""
    values = [float(v) for v in values]
    if world <= 1:
        return values
    t = torch.tensor(values, dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_rate(world, units_per_rank_step, steps, slowest_ms, scale=1e12):
    """Units processed by all ranks (each does the same work) divided by the
    slowest rank's time, per second, in multiples of `scale`."""
    return world * units_per_rank_step * steps / (slowest_ms * 1e-3) / scale


def run_gpu(args, rank, world, local_rank):
    import torch

    import quantized_mixed_precision_gb300 as bq
    from quantized_mixed_precision_gb300 import roofline, workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    bq.lib()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    stream = torch.cuda.current_stream()
    flush = (torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev),
             torch.zeros(FLUSH_BYTES, dtype=torch.uint8, device=dev))

    # ---- headline workload: INT8 x INT4 4096^3 with per-column dequant ----
    d = W.cfg2()
    A = torch.from_numpy(d["A"]).to(dev)
    Bq = torch.from_numpy(d["B"]).to(dev)
    Bp = bq.bq_pack_weights(Bq, 4, "interleaved")       # offline packing, not timed
    sc = torch.from_numpy(d["scale"]).to(dev)
    C = torch.empty((M2, N2), dtype=torch.float16, device=dev)
    del Bq
    # two more input sets (rotations of the first) so consecutive steps miss L2
    sets = [(A, Bp, sc, C)]
    for r in (1, 2):
        sets.append((torch.roll(A, r * 1031, 0).contiguous(), torch.roll(Bp, r * 977, 0).contiguous(), sc,
                     torch.empty_like(C)))

    def step(i):
        a, b, s_, c = sets[i % len(sets)]
        bq.bq_gemm_i8xi4(a, b, "interleaved", col_scale=s_, out=c)

    gemm_launches_per_step = 1
    hbm_peak, tc_peak, tc_sust, peak_src = load_peaks()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    graph = capture(torch, lambda: [step(i) for i in range(args.steps)])

    with ClockSampler(local_rank) as clk:
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t_wall0 = time.perf_counter()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        t_wall = time.perf_counter() - t_wall0
    clocks = clk.summary()
    (total_ms,) = max_over_ranks(torch, [e0.elapsed_time(e1)], dev, world)
    ms_step = total_ms / args.steps
    value = whole_job_rate(world, OPS2, args.steps, total_ms)
    single = time_steps(torch, lambda: step(0), 5, 2, flush, stream)
    del graph, sets

    # ---- end to end: pinned host buffers, H2D + C ABI call + D2H every step ----
    A_h = torch.from_numpy(d["A"]).pin_memory()
    Bp_h = Bp.cpu().pin_memory()
    sc_h = torch.from_numpy(d["scale"]).pin_memory()
    h2d_bytes = A_h.numel() + Bp_h.numel() + 2 * sc_h.numel()
    d2h_bytes = 2 * M2 * N2
    e2e_ms, e2e_serial_ms = max_over_ranks(torch, e2e_pipelined(torch, bq, A_h, Bp_h, sc_h, dev, args.steps,
                                                                  args.warmup), dev, world)
    e2e = {"value": whole_job_rate(world, OPS2, args.steps, e2e_ms), "unit": "TOPS",
           "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes, "ms_per_step": e2e_ms / args.steps,
           "method": "every step copies its A, B and scale host->device and its C device->host (pinned buffers) "
                     "around one C-ABI call; three buffer sets on three streams, so step i's GEMM overlaps step "
                     "i+1's upload and step i-1's download; events bracket all K steps",
           "serialized_ms_per_step": e2e_serial_ms / args.steps}
    del A_h, Bp_h

    # ---- the M = 1 GEMV (a memory-bound kernel): a stack of 8 layers ----
    d3 = W.cfg3(M=1)
    S = torch.from_numpy(d3["S"]).to(dev)
    _, s3 = bq.bq_quantize_sym(S, 4)                 # per-channel scale = absmax / 7 of the source matrix
    del S
    X3 = torch.from_numpy(d3["X"]).to(dev)
    W3 = bq.bq_pack_weights(torch.from_numpy(d3["W"]).to(dev), 4, "interleaved")
    layers = [W3] + [torch.roll(W3, i * 977, 0).contiguous() for i in range(1, GEMV_LAYERS)]
    Y3 = [torch.empty((1, 11008), dtype=torch.float16, device=dev) for _ in layers]

    def gemv_stack():
        for i, wl in enumerate(layers):
            bq.bq_gemm_f16xi4(X3, wl, s3, "interleaved", out=Y3[i])

    gemv_stack()
    torch.cuda.synchronize()
    reps = max(1, args.steps // 4)
    g3 = capture(torch, lambda: [gemv_stack() for _ in range(reps)])
    (gemv_ms,) = max_over_ranks(torch, [time_graph(torch, g3, 5, stream) / (reps * GEMV_LAYERS)], dev, world)
    gemv_single = statistics.median(time_steps(torch, lambda: bq.bq_gemm_f16xi4(X3, W3, s3, "interleaved", out=Y3[0]),
                                               args.steps, args.warmup, flush, stream))
    gemv_bytes = roofline.matmul_min_bytes(1, 4096, 11008, 16, 4, 16, extra_bytes=2 * 11008)
    gbs = gemv_bytes / (gemv_ms * 1e-3) / 1e9
    gemv = {"value": gbs, "unit": "GB/s", "ms": gemv_ms, "workload": GEMV_WORKLOAD,
            "method": f"{GEMV_LAYERS} layers with distinct weights ({GEMV_LAYERS * 22.5:.0f} MB) back to back in a "
                      f"CUDA graph, {reps} rounds; per GPU, the slowest rank's time",
            "single_launch_ms_l2_flushed": gemv_single,
            "single_launch_GB/s": gemv_bytes / (gemv_single * 1e-3) / 1e9,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                         "peak_source": f"{peak_src} hbm_gbs"}}
    del g3, layers, X3, W3, Y3

    paths = {} if args.no_paths else measure_paths(torch, bq, W, roofline, dev, flush, stream, hbm_peak, tc_peak)
    achieved = OPS2 / (ms_step * 1e-3) / 1e12
    traffic = ncu_traffic("gemm_pair_kernel")
    line = {
        "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD,
                   "l2": "inputs larger than L2: steps cycle through 3 input sets (168 MiB); K steps replayed as one "
                         "CUDA graph between two events",
                   "single_launch_ms_l2_flushed": statistics.median(single),
                   "mma": "tcgen05.mma cta_group::2 kind::f16 on CTA pairs (int8/int4 converted exactly to fp16), fp32 accumulation",
                   "per_gpu": "independent replica of the workload on every rank"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": achieved / tc_peak, "traffic": traffic,
                     "peak_source": f"{peak_src} bf16_tflops (burst; fp16 dense rate equals bf16)",
                     "kernel": "gemm_pair_kernel"},
        "e2e": e2e, "gpu_launches": gemm_launches_per_step * args.steps, "clocks": clocks,
        "wall_s_timed_region": t_wall, "gemv": gemv, "paths": paths,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(d, Bp.cpu().numpy())
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure_paths(torch, bq, W, roofline, dev, flush, stream, hbm_peak, tc_peak, steps=10, warmup=3):
    """The other workloads, each timed with the same protocol (median ms)."""
    out = {}

    def med(fn):
        return statistics.median(time_steps(torch, fn, steps, warmup, flush, stream))

    # quantise + INT8 x INT8, 1024 x 4096 x 4096
    d1 = W.cfg1()
    Wt, Xt = torch.from_numpy(d1["W"]).to(dev), torch.from_numpy(d1["X"]).to(dev)
    wq = torch.empty((4096, 4096), dtype=torch.int8, device=dev)
    sw = torch.empty((4096,), dtype=torch.float16, device=dev)
    ms = med(lambda: bq.bq_quantize_sym(Wt, 8, q=wq, scale=sw))
    qb = roofline.quantize_bytes(4096, 4096)
    out["quantize_w_4096x4096"] = {"ms": ms, "GB/s": qb / (ms * 1e-3) / 1e9, "hbm_frac": qb / (ms * 1e-3) / 1e9 / hbm_peak}
    xq, sx = bq.bq_quantize_sym(Xt, 8)
    ms = med(lambda: bq.bq_gemm_i8xi8(xq, wq, row_scale=sx, col_scale=sw))
    ops = roofline.matmul_ops(1024, 4096, 4096)
    out["i8xi8_rowcol_1024x4096x4096"] = {"ms": ms, "TOPS": ops / (ms * 1e-3) / 1e12,
                                          "tc_frac": ops / (ms * 1e-3) / 1e12 / tc_peak}
    # the fused quantised linear (fp16 X quantised inside the GEMM) beside the two-call path
    # (bq_quantize_sym of X, then the integer GEMM with both scales), for 8- and 4-bit weights
    Y = torch.empty((1024, 4096), dtype=torch.float16, device=dev)
    sxf = torch.empty((1024,), dtype=torch.float16, device=dev)
    q = torch.empty((1024, 4096), dtype=torch.int8, device=dev)
    w4q, sw4 = bq.bq_quantize_sym(Wt, 4)
    w4 = bq.bq_pack_weights(w4q, 4, "interleaved")
    for bits, wd, swd, gemm in ((8, wq, sw, lambda: bq.bq_gemm_i8xi8(q, wq, row_scale=sxf, col_scale=sw, out=Y)),
                                (4, w4, sw4, lambda: bq.bq_gemm_i8xi4(q, w4, "interleaved", row_scale=sxf,
                                                                      col_scale=sw4, out=Y))):
        ms_f = med(lambda: bq.bq_quantized_linear(Xt, wd, bits, swd, layout="interleaved", out=Y, x_scale=sxf))

        def two_call():
            bq.bq_quantize_sym(Xt, 8, q=q, scale=sxf)
            gemm()

        ms_2 = med(two_call)
        out[f"linear_fused_w{bits}_1024x4096x4096"] = {
            "ms": ms_f, "TOPS": ops / (ms_f * 1e-3) / 1e12, "two_call_ms": ms_2,
            "two_call_TOPS": ops / (ms_2 * 1e-3) / 1e12, "launches": 2, "two_call_launches": 2}
    del Wt, Xt, wq, sw, xq, sx, Y, sxf, q, w4q, sw4, w4
    # INT8 x INT4 256^3 int32
    d0 = W.cfg0()
    A0 = torch.from_numpy(d0["A"]).to(dev)
    B0 = bq.bq_pack_weights(torch.from_numpy(d0["B"]).to(dev), 4, "plain")
    ms = med(lambda: bq.bq_gemm_i8xi4(A0, B0, "plain"))
    out["i8xi4_i32_256^3"] = {"ms": ms, "TOPS": roofline.matmul_ops(256, 256, 256) / (ms * 1e-3) / 1e12}
    # INT8 x INT4 4096^3 with the dequantisation followed by a fused activation
    d2 = W.cfg2()
    A2 = torch.from_numpy(d2["A"]).to(dev)
    B2 = bq.bq_pack_weights(torch.from_numpy(d2["B"]).to(dev), 4, "interleaved")
    s2 = torch.from_numpy(d2["scale"]).to(dev)
    C2 = torch.empty((4096, 4096), dtype=torch.float16, device=dev)
    for act in ("none", "relu", "gelu"):
        ms = med(lambda: bq.bq_gemm_i8xi4_act(A2, B2, act, "interleaved", col_scale=s2, out=C2))
        out[f"i8xi4_{act}_4096^3"] = {"ms": ms, "TOPS": OPS2 / (ms * 1e-3) / 1e12,
                                      "tc_frac": OPS2 / (ms * 1e-3) / 1e12 / tc_peak}
    # batched with a shared activation block: one 1024 x 4096 A against three stacked 4096 x 4096 int4
    # weights (a fused QKV projection), each item with its own column scales
    Aq = A2[:1024].unsqueeze(0).contiguous()
    Bq3 = torch.stack([B2, torch.roll(B2, 977, 0), torch.roll(B2, 1931, 0)]).contiguous()
    sq = torch.stack([s2, s2, s2]).contiguous()
    Cq = torch.empty((3, 1024, 4096), dtype=torch.float16, device=dev)
    ms = med(lambda: bq.bq_gemm_i8xi4_batched(Aq, Bq3, "interleaved", col_scale=sq, out=Cq))
    ops = 3 * roofline.matmul_ops(1024, 4096, 4096)
    out["qkv_i8xi4_batched_3x1024x4096x4096"] = {"ms": ms, "TOPS": ops / (ms * 1e-3) / 1e12,
                                                 "tc_frac": ops / (ms * 1e-3) / 1e12 / tc_peak}
    del A2, B2, s2, C2, Aq, Bq3, sq, Cq
    # fp16 x INT4, dynamic M
    d3 = W.cfg3(M=1024, source=False)
    W3 = bq.bq_pack_weights(torch.from_numpy(d3["W"]).to(dev), 4, "interleaved")
    s3 = torch.full((11008,), 0.01, dtype=torch.float16, device=dev)
    X3 = torch.from_numpy(d3["X"]).to(dev)
    for M in (1, 4, 16, 64, 256, 1024):
        Xm = X3[:M].contiguous()
        ms = med(lambda: bq.bq_gemm_f16xi4(Xm, W3, s3, "interleaved"))
        b = roofline.matmul_min_bytes(M, 4096, 11008, 16, 4, 16, extra_bytes=2 * 11008)
        f = roofline.matmul_ops(M, 4096, 11008)
        out[f"f16xi4_M{M}"] = {"ms": ms, "GB/s": b / (ms * 1e-3) / 1e9, "TFLOPS": f / (ms * 1e-3) / 1e12,
                               "hbm_frac": b / (ms * 1e-3) / 1e9 / hbm_peak, "tc_frac": f / (ms * 1e-3) / 1e12 / tc_peak}
    # fp16 x unsigned 4-bit with a per-column zero point (codes u = q + 8, zero points in [0, 15] with some
    # fractional), the same layer and activations
    rng = np.random.default_rng(0)
    U3 = bq.bq_pack_weights((torch.from_numpy(d3["W"]).to(dev).to(torch.int16) + 8).to(torch.int8), 4,
                            "interleaved")
    z3 = torch.from_numpy((rng.integers(0, 16, size=11008) + rng.uniform(-0.5, 0.5, size=11008))
                          .astype(np.float16)).to(dev)
    rs3 = torch.empty((1024,), dtype=torch.float32, device=dev)
    for M in (1, 64, 1024):
        Xm = X3[:M].contiguous()
        ms = med(lambda: bq.bq_gemm_f16xu4_zp(Xm, U3, s3, z3, "interleaved", row_sum=rs3[:M]))
        b = roofline.matmul_min_bytes(M, 4096, 11008, 16, 4, 16, extra_bytes=4 * 11008 + 4 * M)
        f = roofline.matmul_ops(M, 4096, 11008)
        out[f"f16xu4_zp_M{M}"] = {"ms": ms, "GB/s": b / (ms * 1e-3) / 1e9, "TFLOPS": f / (ms * 1e-3) / 1e12,
                                  "hbm_frac": b / (ms * 1e-3) / 1e9 / hbm_peak,
                                  "tc_frac": f / (ms * 1e-3) / 1e12 / tc_peak, "launches": 2}
    del W3, X3, U3, z3, rs3
    # INT8 x ternary, N = K = 8192
    d4 = W.cfg4(M=1024)
    B4 = bq.bq_pack_weights(torch.from_numpy(d4["B"]).to(dev), 2, "interleaved")
    s4 = torch.from_numpy(d4["scale"]).to(dev)
    A4 = torch.from_numpy(d4["A"]).to(dev)
    for M in (1, 128, 1024):
        Am = A4[:M].contiguous()
        ms = med(lambda: bq.bq_gemm_i8xi2(Am, B4, "interleaved", col_scale=s4))
        b = roofline.matmul_min_bytes(M, 8192, 8192, 8, 2, 16, extra_bytes=2 * 8192)
        f = roofline.matmul_ops(M, 8192, 8192)
        out[f"i8xi2_M{M}"] = {"ms": ms, "GB/s": b / (ms * 1e-3) / 1e9, "TOPS": f / (ms * 1e-3) / 1e12,
                              "hbm_frac": b / (ms * 1e-3) / 1e9 / hbm_peak, "tc_frac": f / (ms * 1e-3) / 1e12 / tc_peak}
    return out


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------
def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_rows(O, a_rows, bp, scale):
    """The oracle's whole path for a block of A rows: unpack the packed
    weights, exact int32 GEMM, fp32 dequantisation to fp16."""
    b = O.unpack_interleaved(bp, K2, 4)
    return O.dequant(O.gemm_int(a_rows, b), scale)


def cpu_baseline(d, bp, budget_s=10.0, rows=512):
    from oracle import bq_oracle as O
    done, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        r0 = done % M2                      # cycle over A's row blocks until the budget is spent
        oracle_rows(O, d["A"][r0:r0 + rows], bp, d["scale"])
        done += rows
    el = time.perf_counter() - t0
    return {"value": 2 * done * N2 * K2 / el / 1e12, "unit": "TOPS", "cores": cores_used(), "kind": "oracle",
            "sample": f"{done} rows of A cycled over its {M2} rows ({rows}-row blocks, each unpacking B and running the exact "
                      f"float64-BLAS int32 GEMM + fp32 dequant), {el:.1f} s; numpy BLAS threads = all available cores"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    from oracle import bq_oracle as O
    from quantized_mixed_precision_gb300 import workloads as W
    d = W.cfg2()
    bp = O.pack_interleaved(d["B"], 4)
    rows = 256
    for i in range(args.warmup):
        oracle_rows(O, d["A"][:rows], bp, d["scale"])
    times = []
    for i in range(args.steps):
        r0 = (i * rows) % M2
        t0 = time.perf_counter()
        oracle_rows(O, d["A"][r0:r0 + rows], bp, d["scale"])
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = 2 * rows * N2 * K2 * args.steps / total / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": f"{rows} rows of A per step (full B, K)"},
            "cpu_baseline": {"value": value, "unit": "TOPS", "cores": cores_used(), "kind": "oracle",
                             "sample": f"{rows} of {M2} rows of A per step"},
            "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _profile_workloads():
    """Named single workloads, each a callable that sets up its inputs once and
    returns the step to launch."""
    def setup(name):
        import torch

        import quantized_mixed_precision_gb300 as bq
        from quantized_mixed_precision_gb300 import workloads as W
        dev = torch.device("cuda")
        bq.lib()
        if name in ("gemv_m1", "f16xi4_m64", "zp_m1024"):
            M = {"gemv_m1": 1, "f16xi4_m64": 64, "zp_m1024": 1024}[name]
            d = W.cfg3(M=M, source=False)
            X = torch.from_numpy(d["X"]).to(dev)
            s = torch.full((11008,), 0.01, dtype=torch.float16, device=dev)
            if name == "zp_m1024":
                U = bq.bq_pack_weights((torch.from_numpy(d["W"]).to(dev).to(torch.int16) + 8).to(torch.int8), 4,
                                       "interleaved")
                z = torch.full((11008,), 7.5, dtype=torch.float16, device=dev)
                return lambda: bq.bq_gemm_f16xu4_zp(X, U, s, z, "interleaved")
            Wp = bq.bq_pack_weights(torch.from_numpy(d["W"]).to(dev), 4, "interleaved")
            return lambda: bq.bq_gemm_f16xi4(X, Wp, s, "interleaved")
        if name == "quantize_4096":
            Wt = torch.from_numpy(W.cfg1(M=1)["W"]).to(dev)
            q = torch.empty((4096, 4096), dtype=torch.int8, device=dev)
            sc = torch.empty((4096,), dtype=torch.float16, device=dev)
            return lambda: bq.bq_quantize_sym(Wt, 8, q=q, scale=sc)
        if name == "linear_w8_1024":
            d = W.cfg1()
            wq, sw = bq.bq_quantize_sym(torch.from_numpy(d["W"]).to(dev), 8)
            X = torch.from_numpy(d["X"]).to(dev)
            return lambda: bq.bq_quantized_linear(X, wq, 8, sw)
        if name == "i8xi8_1024":
            d = W.cfg1()
            xq, sx = bq.bq_quantize_sym(torch.from_numpy(d["X"]).to(dev), 8)
            wq, sw = bq.bq_quantize_sym(torch.from_numpy(d["W"]).to(dev), 8)
            return lambda: bq.bq_gemm_i8xi8(xq, wq, row_scale=sx, col_scale=sw)
        if name == "pair_i8xi4_4096":
            d = W.cfg2()
            A = torch.from_numpy(d["A"]).to(dev)
            Bp = bq.bq_pack_weights(torch.from_numpy(d["B"]).to(dev), 4, "interleaved")
            sc = torch.from_numpy(d["scale"]).to(dev)
            return lambda: bq.bq_gemm_i8xi4(A, Bp, "interleaved", col_scale=sc)
        raise ValueError(name)
    return setup


PROFILES = ("gemv_m1", "f16xi4_m64", "quantize_4096", "linear_w8_1024", "zp_m1024", "pair_i8xi4_4096", "i8xi8_1024")


def run_profile(name, launches=3):
    import torch
    step = _profile_workloads()(name)
    for _ in range(2 + launches):
        step()
    torch.cuda.synchronize()
    import quantized_mixed_precision_gb300 as bq
    print(json.dumps({"profile": name, "launches": 2 + launches, "status": bq.bq_device_status(reset=True)}))


def main():
    args = parse()
    if args.profile:
        run_profile(args.profile)
        return
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
