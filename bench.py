"""Benchmark of the fine-grained FP8 hot path on GB300.

One step = one Fprop linear layer of the FP8 training path, computed online:
  1. 1x128 E4M3 quantization of the BF16 activations X[4096, 7168]
     (8 fixed outlier channels x50),
  2. 128x128 E4M3 quantization of the FP32 master weight W[18432, 7168],
  3. block-scaled FP8 GEMM Y = X W^T with FP32 promotion every 128 of K,
     BF16 output Y[4096, 18432].
value = 2*M*N*K / step time (TFLOP/s of the whole step, quantizers included),
aggregated over all ranks (each rank runs its own replica: weak scaling).
The JSON line also carries the per-kernel breakdown (quantizer GB/s against
HBM, GEMM TFLOP/s against the FP8 tensor peak), the roofline of the dominant
kernel, an end-to-end number through the C ABI with host buffers, the SM
clocks seen during the timed region, and the CPU oracle timed on a bounded
sample of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload fprop|tiny|dgrad|wgrad|grouped]

For N > 1 launch with torchrun (one rank per GPU); rank 0 prints the line.
--workload other than fprop times the same kernels on the other GEMMs of
the FP8 path (the tiny 256x256x512 Fprop; Dgrad dY[8192,2048] x
W[2048,7168]; Wgrad dY^T X with X[8192,7168], token-axis groups; grouped MoE
64 experts W_g[2048,7168] over 32768 tokens) on one GPU and prints a line of
the same metric for it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "block-scaled FP8 GEMM TFLOP/s & % of FP8 peak; quantizer GB/s vs HBM"
M, N, K = 4096, 18432, 7168
WORKLOAD = ("Fprop linear: X[4096,7168] bf16 N(0,1) with 8 fixed outlier channels x50, quantized 1x128; "
            "W[18432,7168] fp32 master N(0,0.02^2), quantized 128x128; Y = X W^T [4096,18432] bf16, "
            "FP32 promotion every 128 of K; seed 1")
FLOPS = 2.0 * M * N * K
ACT_BYTES = M * K * 2 + M * K + (K // 128) * M * 4                 # 3.031 B per element
W_BYTES = N * K * 4 + N * K + (N // 128) * (K // 128) * 4         # 5.0002 B per element
DUAL_BYTES = M * K * 2 + 2 * M * K + 2 * (K // 128) * M * 4        # 4.0625 B per element (one read, two outputs)
GEMM_MIN_BYTES = M * K + N * K + 4 * (M * K // 128 + N * K // 16384) + M * N * 2
FP8_OVER_BF16 = 4.5 / 2.25          # nominal dense FP8 : BF16 tensor ratio
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "gemm_blockscaled_fprop_4096x18432x7168.md")


# --------------------------------------------------------------- helpers ---

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, group=None) -> float:
    """Maximum of a per-rank float over the process group (identity when not
    distributed).  Uses the group's own backend."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return float(value)
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def rank_seed(rank: int) -> int:
    """Seed of each rank's replica: rank 0 draws the published workload (seed 1)."""
    return 1 + 1000 * rank


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK["hbm_gbs"], FALLBACK["bf16_tflops"], "fallback"


def gemm_source_sha() -> str:
    """Hash of the GEMM's code (gemm.cu + ptx.cuh) with // comments and blank
    lines left out, so that a comment edit does not orphan a profile."""
    h = hashlib.sha256()
    for rel in ("fp8_fine_grained_act_gb300/csrc/gemm.cu", "fp8_fine_grained_act_gb300/csrc/ptx.cuh"):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            for line in f:
                code = re.sub(r"//.*$", "", line).rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per GEMM launch from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    sha = re.search(r"kernel source sha256\[:16\]:\s*([0-9a-f]+)", text)
    tr = re.search(r"dram bytes per launch \(read \+ write\):\s*([0-9]+)", text)
    if not sha or not tr or sha.group(1) != gemm_source_sha():
        return None
    return int(tr.group(1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append({"sm": float(f[1]), "max": float(f[2]), "power": float(f[3]),
                             "hw_slowdown": f[5], "hw_thermal": f[6], "sw_thermal": f[7], "sw_power_cap": f[8]})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        busy = [r for r in rows if r["power"] > 200.0] or rows
        reasons = []
        for key, name in (("hw_slowdown", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                          ("sw_thermal", "sw_thermal_slowdown"), ("sw_power_cap", "sw_power_cap")):
            if any(r[key].lower().startswith("active") for r in busy):
                reasons.append(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": reasons, "samples": len(busy), "power_w_max": max(r["power"] for r in rows)}


# ------------------------------------------------------------- oracle CPU ---

def cpu_baseline(mb: int, nb: int, seed: int = 1):
    """The oracle, as it is, on a bounded sample of the workload: the first
    mb tokens and nb output channels of the Fprop layer (quantize both, then
    the double GEMM).  Returns (GEMM-equivalent TFLOP/s of the sample, cores,
    seconds)."""
    import oracle
    from fp8_fine_grained_act_gb300 import synth
    d = synth.fprop_linear(seed=seed, M=mb, N=nb, K=K)
    t0 = time.perf_counter()
    qx, sx = oracle.quant_act(d["x"])
    qw, sw = oracle.quant_w(d["w"])
    oracle.gemm(qx, sx, qw, sw)
    dt = time.perf_counter() - t0
    return 2.0 * mb * nb * K / dt / 1e12, oracle.num_threads(), dt


def run_reference(args):
    """The oracle arm: each step is a bounded sample of the workload, sized
    so that warm-up plus timed steps take about two minutes."""
    mb = 128
    _, _, t_small = cpu_baseline(mb, 256)
    per_step = min(5.0, 120.0 / (args.steps + args.warmup))
    nb = int(max(2, min(256, round(2 * per_step / max(t_small, 1e-6))))) * 128
    for _ in range(args.warmup):
        cpu_baseline(mb, nb)
    times = []
    cores = 1
    for _ in range(args.steps):
        _, cores, dt = cpu_baseline(mb, nb)
        times.append(dt)
    t = sum(times) / len(times)
    value = 2.0 * mb * nb * K / t / 1e12
    sample = f"Fprop sample per step: X[{mb},{K}] and W[{nb},{K}] quantized + {mb}x{nb}x{K} double GEMM"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU ---

def run_gpu(args):
    import torch
    import torch.distributed as dist

    from fp8_fine_grained_act_gb300 import binding as fb
    from fp8_fine_grained_act_gb300 import build as fbuild
    from fp8_fine_grained_act_gb300 import synth

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device; the FP8 path has no CPU fallback")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    fbuild.build()
    fb.load()
    dev = torch.device("cuda", local)

    d = synth.fprop_linear(seed=rank_seed(rank))
    x_h = torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    w_h = torch.from_numpy(d["w"]).pin_memory()
    del d
    x = x_h.to(dev)
    w = w_h.to(dev)
    qx = torch.empty((M, K), dtype=torch.uint8, device=dev)
    sx = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
    qw = torch.empty((N, K), dtype=torch.uint8, device=dev)
    sw = torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    y_h = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fb.fp8_quant_act_1x128(x, q=qx, scales=sx, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        fb.fp8_quant_w_128x128(w, q=qw, scales=sw, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        fb.fp8_gemm_blockscaled(qx, sx, qw, sw, out_dtype=fb.FP8FG_OUT_BF16, d=y, stream=stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert fb.fp8fg_last_device_status() == 0

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total_ms = start.elapsed_time(end)
    t_act = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    t_w = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps
    t_gemm = sum(e[2].elapsed_time(e[3]) for e in evs) / args.steps
    status = fb.fp8fg_last_device_status()
    if status != 0:
        raise SystemExit(f"device status {status}: {fb.fp8fg_status_string(status)}")

    # end to end through the C ABI with host buffers: H2D of X and W from pinned
    # memory, the three kernels, D2H of Y into pinned memory, every step
    e2e_steps = max(3, min(args.steps, 50))
    for _ in range(2):
        x.copy_(x_h, non_blocking=True)
        w.copy_(w_h, non_blocking=True)
        step()
        y_h.copy_(y, non_blocking=True)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        x.copy_(x_h, non_blocking=True)
        w.copy_(w_h, non_blocking=True)
        step()
        y_h.copy_(y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps)

    # the same, with step i+1's uploads and step i-1's download overlapping
    # step i's kernels: three streams, two device buffer sets
    s_up, s_cmp, s_dn = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    xs, ws = [x, torch.empty_like(x)], [w, torch.empty_like(w)]
    ys = [y, torch.empty_like(y)]
    yhs = [y_h, torch.empty_like(y_h).pin_memory()]
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_dn = [torch.cuda.Event() for _ in range(2)]

    def pipelined(n):
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_up):
                if i >= 2:
                    s_up.wait_event(ev_cmp[b])
                xs[b].copy_(x_h, non_blocking=True)
                ws[b].copy_(w_h, non_blocking=True)
                ev_up[b].record(s_up)
            s_cmp.wait_event(ev_up[b])
            if i >= 2:
                s_cmp.wait_event(ev_dn[b])
            fb.fp8_quant_act_1x128(xs[b], q=qx, scales=sx, stream=s_cmp)
            fb.fp8_quant_w_128x128(ws[b], q=qw, scales=sw, stream=s_cmp)
            fb.fp8_gemm_blockscaled(qx, sx, qw, sw, out_dtype=fb.FP8FG_OUT_BF16, d=ys[b], stream=s_cmp)
            ev_cmp[b].record(s_cmp)
            with torch.cuda.stream(s_dn):
                s_dn.wait_event(ev_cmp[b])
                yhs[b].copy_(ys[b], non_blocking=True)
                ev_dn[b].record(s_dn)

    pipelined(4)
    torch.cuda.synchronize()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(s_up)
    pipelined(e2e_steps)
    s_up.wait_stream(s_dn)
    p1.record(s_up)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(p0.elapsed_time(p1) / e2e_steps)
    del xs[1], ws[1], ys[1], yhs[1]

    # outside the step: the fused 1x128 + 128x1 quantizer on the same X (what a
    # training forward runs to cache X in FP8 for the weight gradient)
    qr, srw, qct, scl = fb.fp8_quant_act_dual(x, stream=stream)
    dual_iters = 50
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(dual_iters):
        fb.fp8_quant_act_dual(x, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    t_dual = max_over_ranks(e0.elapsed_time(e1) / dual_iters)
    del qr, srw, qct, scl

    ms_step = max_over_ranks(total_ms / args.steps)
    t_gemm = max_over_ranks(t_gemm)
    t_act = max_over_ranks(t_act)
    t_w = max_over_ranks(t_w)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    hbm, bf16, src = peaks()
    fp8_peak = bf16 * FP8_OVER_BF16
    gemm_tflops = FLOPS / (t_gemm * 1e-3) / 1e12
    clocks = clk.summary()
    line = {
        "metric": METRIC,
        "value": world * FLOPS / (ms_step * 1e-3) / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K,
                   "l2": "inputs larger than L2: each step reads X (58.7 MB) and W (528 MB)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": gemm_tflops, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": gemm_tflops / fp8_peak, "traffic": profiled_traffic(),
                     "kernel": "gemm_blockscaled_kernel<0>",
                     "peak_source": f"{src} bf16 burst {bf16} TFLOP/s x {FP8_OVER_BF16} (FP8:BF16 nominal)"},
        "kernels": {
            "quant_act_1x128": {"us": t_act * 1e3, "GB/s": ACT_BYTES / (t_act * 1e-3) / 1e9,
                                "frac_hbm": ACT_BYTES / (t_act * 1e-3) / 1e9 / hbm},
            "quant_w_128x128": {"us": t_w * 1e3, "GB/s": W_BYTES / (t_w * 1e-3) / 1e9,
                                "frac_hbm": W_BYTES / (t_w * 1e-3) / 1e9 / hbm},
            "quant_act_dual_1x128_128x1 (not in the step)": {
                "us": t_dual * 1e3, "GB/s": DUAL_BYTES / (t_dual * 1e-3) / 1e9,
                "frac_hbm": DUAL_BYTES / (t_dual * 1e-3) / 1e9 / hbm},
            "gemm_blockscaled": {"us": t_gemm * 1e3, "TFLOP/s": gemm_tflops, "frac_fp8_peak": gemm_tflops / fp8_peak},
            "hbm_peak_gbs": hbm, "hbm_peak_source": src,
        },
        "e2e": {"value": world * FLOPS / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": x_h.numel() * 2 + w_h.numel() * 4,
                "d2h_bytes_per_step": y_h.numel() * 2, "ms_per_step": e2e_ms, "steps": e2e_steps,
                "how": "copies of step i+1 (H2D) and i-1 (D2H) overlap step i's kernels on separate streams",
                "serial_ms_per_step": e2e_serial_ms},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        mb, nb = 1024, 4096
        v, cores, dt = cpu_baseline(mb, nb)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": f"first {mb} tokens x {nb} output channels of the workload: both "
                                          f"quantizers + {mb}x{nb}x{K} double GEMM, {dt:.1f} s"}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_other(args):
    """One step of another GEMM of the path (quantizers + GEMM), single GPU,
    CUDA events per kernel; the line has the same metric and a per-kernel
    breakdown."""
    import torch

    from fp8_fine_grained_act_gb300 import binding as fb
    from fp8_fine_grained_act_gb300 import build as fbuild
    from fp8_fine_grained_act_gb300 import synth

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device; the FP8 path has no CPU fallback")
    fbuild.build()
    fb.load()
    dev = torch.device("cuda", 0)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    kernels = []   # (name, fn, algorithmic bytes or None)
    extra = {}
    if args.workload == "tiny":
        d = synth.tiny_fprop(seed=0)
        x, w = bf(d["x"]), torch.from_numpy(d["w"]).to(dev)
        Mw, Kw = x.shape
        Nw = w.shape[0]
        qx = torch.empty((Mw, Kw), dtype=torch.uint8, device=dev)
        sx = torch.empty((Kw // 128, Mw), dtype=torch.float32, device=dev)
        qw = torch.empty((Nw, Kw), dtype=torch.uint8, device=dev)
        sw = torch.empty((Nw // 128, Kw // 128), dtype=torch.float32, device=dev)
        y = torch.empty((Mw, Nw), dtype=torch.float32, device=dev)

        def k_act():
            fb.fp8_quant_act_1x128(x, q=qx, scales=sx)

        def k_w():
            fb.fp8_quant_w_128x128(w, q=qw, scales=sw)

        def k_gemm():
            fb.fp8_gemm_blockscaled(qx, sx, qw, sw, out_dtype=fb.FP8FG_OUT_F32, d=y)

        # the same three calls captured once in a CUDA graph and replayed:
        # this shape is bound by launch overhead, which the graph removes
        for fn in (k_act, k_w, k_gemm):
            fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            k_act()
            k_w()
            k_gemm()
        extra["graph"] = graph

        kernels = [("quant_act_1x128 X", k_act, Mw * Kw * 3.031), ("quant_w_128x128 W", k_w, Nw * Kw * 5.0002),
                   ("gemm_blockscaled", k_gemm, None)]
        workload = ("Tiny Fprop: X[256,512] N(0,1) with 0.1% of entries x100, W[256,512] N(0,0.02^2), fp32 out; "
                    "seed 0 (launch-latency bound: two 128x256 tiles)")
    elif args.workload == "dgrad":
        d = synth.dgrad(seed=2)
        dy, w = bf(d["dy"]), torch.from_numpy(d["w"]).to(dev)
        Mw, Kw = dy.shape
        Nw = w.shape[1]
        qdy = torch.empty((Mw, Kw), dtype=torch.uint8, device=dev)
        sdy = torch.empty((Kw // 128, Mw), dtype=torch.float32, device=dev)
        out = {}

        def k_act():
            fb.fp8_quant_act_1x128(dy, q=qdy, scales=sdy)

        def k_w():
            out["w"] = fb.fp8_quant_w_128x128(w, transposed=True)

        k_w()
        y = torch.empty((Mw, Nw), dtype=torch.bfloat16, device=dev)

        def k_gemm():
            fb.fp8_gemm_blockscaled(qdy, sdy, out["w"][1], out["w"][2], sb_strides=(1, Nw // 128), d=y)

        kernels = [("quant_act_1x128 dY", k_act, Mw * Kw * 3.031),
                   ("quant_w_128x128 W + transposed copy", k_w, Kw * Nw * 6.0002), ("gemm_blockscaled", k_gemm, None)]
        workload = "Dgrad: dX[8192,7168] = dY[8192,2048] . W[2048,7168], block scales read transposed, bf16 out; seed 2"
    elif args.workload == "wgrad":
        d = synth.wgrad(seed=3)
        dy, x = bf(d["dy"]), bf(d["x"])
        T, Mw = dy.shape
        Nw = x.shape[1]
        Kw = T
        res = {}

        def k_dy():
            res["a"] = fb.fp8_quant_act_1x128(dy, axis=fb.FP8FG_AXIS_ROWS)

        def k_x():
            res["b"] = fb.fp8_quant_act_1x128(x, axis=fb.FP8FG_AXIS_ROWS)

        k_dy()
        k_x()
        y = torch.empty((Mw, Nw), dtype=torch.float32, device=dev)

        def k_gemm():
            fb.fp8_gemm_blockscaled(res["a"][0], res["a"][1], res["b"][0], res["b"][1], bscale=fb.FP8FG_BSCALE_ROW,
                                    out_dtype=fb.FP8FG_OUT_F32, d=y)

        kernels = [("quant_act_128x1 dY", k_dy, T * Mw * 3.031), ("quant_act_128x1 X", k_x, T * Nw * 3.031),
                   ("gemm_blockscaled (per-row B scales)", k_gemm, None)]
        workload = "Wgrad: dW[2048,7168] = dY^T . X over 8192 tokens, 128x1 groups, per-row B scales, fp32 out; seed 3"
    else:
        d = synth.grouped_moe(seed=4)
        x = bf(d["x"])
        G, Nw, Kw = d["w"].shape
        w = torch.from_numpy(d["w"].reshape(G * Nw, Kw)).to(dev)
        off = torch.from_numpy(d["offsets"]).to(dev)
        Mw = x.shape[0]
        del d
        res = {}

        def k_act():
            res["a"] = fb.fp8_quant_act_1x128(x)

        def k_w():
            res["b"] = fb.fp8_quant_w_128x128(w, transposed=False)

        k_act()
        k_w()
        y = torch.empty((Mw, Nw), dtype=torch.bfloat16, device=dev)

        def k_gemm():
            fb.fp8_gemm_grouped(res["a"][0], res["a"][1], res["b"][0].view(G, Nw, Kw),
                                res["b"][1].view(G, Nw // 128, Kw // 128), off, d=y)

        kernels = [("quant_act_1x128 X_all", k_act, Mw * Kw * 3.031),
                   ("quant_w_128x128 64 experts", k_w, G * Nw * Kw * 5.0002), ("gemm_grouped", k_gemm, None)]
        workload = (f"Grouped MoE Fprop: 64 experts W_g[2048,7168], Dirichlet(1)/multinomial counts over 32768 "
                    f"tokens padded to 128 (M_total {Mw}); bf16 out; seed 4")
    flops = 2.0 * Mw * Nw * Kw
    for _ in range(args.warmup):
        for _, fn, _ in kernels:
            fn()
    torch.cuda.synchronize()
    assert fb.fp8fg_last_device_status() == 0
    steps = min(args.steps, 200)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(kernels) + 1)] for _ in range(steps)]
    with ClockSampler(0) as clk:
        for i in range(steps):
            ev[i][0].record()
            for j, (_, fn, _) in enumerate(kernels):
                fn()
                ev[i][j + 1].record()
        torch.cuda.synchronize()
    if fb.fp8fg_last_device_status() != 0:
        raise SystemExit("device status not clean")
    hbm, bf16, src = peaks()
    fp8_peak = bf16 * FP8_OVER_BF16
    per = [sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)) / steps for j in range(len(kernels))]
    ms = sum(per)
    kd = {}
    for (name, _, nbytes), t in zip(kernels, per):
        if nbytes is None:
            tf = flops / (t * 1e-3) / 1e12
            kd[name] = {"us": t * 1e3, "TFLOP/s": tf, "frac_fp8_peak": tf / fp8_peak}
        else:
            kd[name] = {"us": t * 1e3, "GB/s": nbytes / (t * 1e-3) / 1e9, "frac_hbm": nbytes / (t * 1e-3) / 1e9 / hbm}
    if "graph" in extra:
        g = extra["graph"]
        for _ in range(10):
            g.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record()
        for _ in range(steps):
            g.replay()
        g1.record()
        torch.cuda.synchronize()
        graph_ms = g0.elapsed_time(g1) / steps
        kd["step as one CUDA graph (3 kernels)"] = {"us": graph_ms * 1e3, "TFLOP/s": flops / (graph_ms * 1e-3) / 1e12}
    line = {"metric": METRIC, "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1, "steps": steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": {"workload": workload, "M": Mw, "N": Nw, "K": Kw, "parallelism": "single GPU"},
            "kernels": kd, "peaks": {"fp8_tflops": fp8_peak, "hbm_gbs": hbm, "source": src},
            "clocks": clk.summary(), "gpu_launches": len(kernels) * steps}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["fprop", "tiny", "dgrad", "wgrad", "grouped"], default="fprop")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        rank, _, _ = dist_env()
        if rank == 0:
            run_reference(args)
        return
    if args.workload != "fprop":
        run_other(args)
        return
    run_gpu(args)


if __name__ == "__main__":
    main()
