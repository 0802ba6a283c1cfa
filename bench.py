"""Benchmark of the fine-grained FP8 hot path on GB300.

One step = one Fprop linear layer of the FP8 training path, computed online:
  1. 1x128 E4M3 quantization of the BF16 activations X[4096, 7168]
     (8 fixed outlier channels x50),
  2. 128x128 E4M3 quantization of the FP32 master weight W[18432, 7168],
  3. block-scaled FP8 GEMM Y = X W^T with FP32 promotion every 128 of K,
     BF16 output Y[4096, 18432].
value = 2*M*N*K / step time (TFLOP/s of the whole step, quantizers included),
aggregated over all ranks (each rank runs its own replica: weak scaling).

The JSON line also carries, under "kernels", one keyed record per
configuration of the path -- the Fprop step's own kernels, the tiny Fprop,
Dgrad, Wgrad and the grouped MoE GEMM, each with its quantizers -- with the
time, TFLOP/s or GB/s of every kernel and its fraction of the peak; the
roofline of the dominant kernel; the fused dual quantizer; the measured FP8
tensor rate (a probe of back-to-back MMAs); an end-to-end number through the
C ABI with host buffers; the SM clocks seen while each measured block ran
(every block lasts at least a second, so that nvidia-smi samples it under
load); and the CPU oracle timed on a bounded sample of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload fprop|tiny|dgrad|wgrad|grouped] [--configs all|none]

For N > 1 launch with torchrun (one rank per GPU); rank 0 prints the line.
The per-configuration records are single-GPU measurements, taken at N = 1.
--workload other than fprop prints a line for that configuration alone.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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
ROW_B_PER_ELT = 2 + 1 + 4 / 128          # 1x128 or 128x1 quantizer: read BF16, write a code, a scale per 128
W_B_PER_ELT = 4 + 1 + 4 / 16384          # 128x128 quantizer: read FP32, write a code, a scale per block
DUAL_B_PER_ELT = 2 + 2 + 8 / 128         # 1x128 and 128x1 from one read: two codes, two scales per 128
ACT_BYTES = M * K * ROW_B_PER_ELT
W_BYTES = N * K * W_B_PER_ELT
GEMM_MIN_BYTES = M * K + N * K + 4 * (M * K // 128 + N * K // 16384) + M * N * 2
FP8_OVER_BF16 = 4.5 / 2.25               # nominal dense FP8 : BF16 tensor ratio
NOMINAL_FP8_TFLOPS = 4500.0              # GB300 dense FP8, nominal
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
PROFILES = os.path.join(ROOT, "profiles")
PROFILE_SUMMARY = os.path.join(PROFILES, "gemm_blockscaled_fprop_4096x18432x7168.md")
L2_BYTES = 129 * 2 ** 20
MMA_TILE_FLOPS = 2.0 * 128 * 256 * 128   # one K chunk of one 128 x 256 tile


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


def sustained_bf16():
    """The measured BF16 rate of a seconds-long GEMM loop under the power cap
    (None if not measured)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except (OSError, KeyError, ValueError):
        return None


def rotations(bytes_per_set: float, floor: int = 1, cap: int = 8) -> int:
    """Input sets to rotate through so that consecutive uses of one set are
    separated by at least twice the L2 capacity of other inputs."""
    if bytes_per_set <= 0:
        return floor
    return int(max(floor, min(cap, math.ceil(2 * L2_BYTES / bytes_per_set) + 1)))


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


def profiled_traffic(path: str | None = None):
    """DRAM bytes per GEMM launch from a committed ncu summary, if it was
    taken on the current kernel source; else None."""
    try:
        text = open(path or PROFILE_SUMMARY).read()
    except OSError:
        return None
    sha = re.search(r"kernel source sha256\[:16\]:\s*([0-9a-f]+)", text)
    tr = re.search(r"dram bytes per launch \(read \+ write\):\s*([0-9]+)", text)
    if not sha or not tr or sha.group(1) != gemm_source_sha():
        return None
    return int(tr.group(1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a measured block."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = ""

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
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        return summarize_clocks(self.out)


def summarize_clocks(text: str, busy_watts: float = 250.0):
    """Median SM clock and throttle reasons over the samples taken under load
    (power above ``busy_watts``; all samples if none is)."""
    rows = []
    for line in (text or "").splitlines():
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
    busy = [r for r in rows if r["power"] > busy_watts]
    use = busy or rows
    reasons = []
    for key, name in (("hw_slowdown", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                      ("sw_thermal", "sw_thermal_slowdown"), ("sw_power_cap", "sw_power_cap")):
        if any(r[key].lower().startswith("active") for r in use):
            reasons.append(name)
    return {"sm_mhz": statistics.median(r["sm"] for r in use), "sm_max_mhz": max(r["max"] for r in rows),
            "reasons": reasons, "samples": len(rows), "samples_under_load": len(busy),
            "power_w_max": max(r["power"] for r in rows)}


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


def cpu_quantizers_1core(rows: int, seed: int = 1):
    """The oracle's two Fprop quantizers on one host core (the all-core
    figure is the GEMM-dominated cpu_baseline value): X[rows, K] 1x128 and
    W[rows, K] 128x128, as algorithmic GB/s.  The thread count is restored."""
    import oracle
    from fp8_fine_grained_act_gb300 import synth
    d = synth.fprop_linear(seed=seed, M=rows, N=rows, K=K)
    n0 = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        t0 = time.perf_counter()
        oracle.quant_act(d["x"])
        t1 = time.perf_counter()
        oracle.quant_w(d["w"])
        t2 = time.perf_counter()
    finally:
        oracle.set_num_threads(n0)
    act_b = rows * K * (2 + 1 + 4 / 128)
    w_b = rows * K * (4 + 1 + 4 / 16384)
    return {"cores": 1,
            "quant_act_1x128": {"GB/s": act_b / (t1 - t0) / 1e9, "sample": f"X[{rows},{K}] bf16", "s": t1 - t0},
            "quant_w_128x128": {"GB/s": w_b / (t2 - t1) / 1e9, "sample": f"W[{rows},{K}] fp32", "s": t2 - t1}}


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

def _gpu_setup(local: int):
    import torch
    from fp8_fine_grained_act_gb300 import binding as fb
    from fp8_fine_grained_act_gb300 import build as fbuild
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device; the FP8 path has no CPU fallback")
    torch.cuda.set_device(local)
    fbuild.build()
    fb.load()
    return torch.device("cuda", local)


def timed_rounds(kernels, rounds: int, stream):
    """Run `rounds` rounds of the kernels (list of (name, fn)), an event
    between consecutive kernels; returns the mean ms of each kernel and the
    wall ms of the whole block on the device."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(kernels) + 1)] for _ in range(rounds)]
    for i in range(rounds):
        ev[i][0].record(stream)
        for j, (_, fn) in enumerate(kernels):
            fn(i)
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    per = [sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(rounds)) / rounds for j in range(len(kernels))]
    return per, ev[0][0].elapsed_time(ev[-1][-1])


def b2b_ms(fn, stream, seconds: float, warmup: int = 3) -> float:
    """Mean ms per launch of `fn(i)` launched back to back (no event between
    launches) for at least `seconds` of GPU time; the caller rotates inputs
    over more than twice the L2 (or uses inputs larger than L2), so that no
    launch finds its input in L2."""
    import torch
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(5):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    n = int(min(20000, max(20, math.ceil(seconds * 1e3 / max(e0.elapsed_time(e1) / 5, 1e-3)))))
    e0.record(stream)
    for i in range(n):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


class L2Flush:
    """Reads a buffer of 3x the L2 capacity (a reduction, no writes): the L2
    then holds only clean lines of it, so the kernel timed next starts with
    cold inputs and with no dirty lines of earlier kernels left to write
    back (a flush by writing would leave its own dirty lines instead)."""

    def __init__(self, dev):
        import torch
        self.buf = torch.ones(3 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        import torch
        torch.amax(self.buf, dim=0, out=self.sink)


def isolated_times(kernels, flush: L2Flush, stream, seconds: float):
    """Each kernel alone: repeated launches, each after a read-only L2 flush,
    CUDA events around the kernel only.  Returns the mean ms per kernel."""
    import torch
    out = []
    for _, fn in kernels:
        fn(0)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(5):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        reps = int(min(2000, max(20, math.ceil(seconds * 1e3 / (e0.elapsed_time(e1) / 5 + 0.05)))))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for i in range(reps):
            flush()
            ev[i][0].record(stream)
            fn(i)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        out.append(statistics.median(a.elapsed_time(b) for a, b in ev))
    return out


def block_rounds(kernels, stream, seconds: float, warmup: int, cap: int = 20000) -> int:
    """Rounds needed for a measured block of at least `seconds` of GPU time."""
    import torch
    for i in range(max(warmup, 3)):
        for _, fn in kernels:
            fn(i)
    torch.cuda.synchronize()
    _, ms = timed_rounds(kernels, 5, stream)
    return int(min(cap, max(20, math.ceil(seconds * 1e3 / max(ms / 5, 1e-3)))))


def probe_tensor_rate(fb, stream, target_ms: float = 40.0, repeats: int = 5):
    """Measured FP8 tensor rate: the library's probe of back-to-back
    128x256x32 kind::f8f6f4 MMAs, one CTA per SM; the best of `repeats`."""
    import torch
    chunks = 2000
    ctas = fb.fp8fg_probe_mma_rate(chunks, stream=stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    fb.fp8fg_probe_mma_rate(chunks, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    chunks = int(max(2000, min(1 << 22, chunks * target_ms / max(e0.elapsed_time(e1), 1e-3))))
    best = 0.0
    for _ in range(repeats):
        e0.record(stream)
        fb.fp8fg_probe_mma_rate(chunks, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        best = max(best, ctas * chunks * MMA_TILE_FLOPS / (e0.elapsed_time(e1) * 1e-3) / 1e12)
    if fb.fp8fg_last_device_status() != 0:
        raise SystemExit("tensor-rate probe: device status not clean")
    return {"tflops": best, "ctas": ctas, "chunks_per_cta": chunks,
            "how": "one CTA per SM issuing back-to-back tcgen05.mma.kind::f8f6f4 128x256x32 (the GEMM's "
                   "instruction and operand layout), no data movement or promotion; best of 5 launches"}


class Peaks:
    def __init__(self, probe=None):
        self.hbm, self.bf16, self.src = peaks()
        self.fp8 = self.bf16 * FP8_OVER_BF16
        sus = sustained_bf16()
        self.fp8_sustained = sus * FP8_OVER_BF16 if sus else None
        self.probe = probe["tflops"] if probe else None

    def gemm(self, flops: float, ms: float, extra=None):
        tf = flops / (ms * 1e-3) / 1e12
        r = {"us": ms * 1e3, "TFLOP/s": tf, "frac_fp8_peak": tf / self.fp8,
             "frac_nominal_fp8": tf / NOMINAL_FP8_TFLOPS}
        if self.fp8_sustained:
            r["frac_sustained_fp8"] = tf / self.fp8_sustained
        if self.probe:
            r["frac_tensor_probe"] = tf / self.probe
        if extra:
            r.update(extra)
        return r

    def quant(self, nbytes: float, ms: float):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"us": ms * 1e3, "GB/s": gbs, "frac_hbm": gbs / self.hbm}

    def legend(self):
        d = {"fp8_tflops": self.fp8, "fp8_source": f"{self.src} bf16 burst {self.bf16} TFLOP/s x {FP8_OVER_BF16} "
                                                  "(FP8:BF16 nominal)",
             "nominal_fp8_tflops": NOMINAL_FP8_TFLOPS, "hbm_gbs": self.hbm, "hbm_source": self.src}
        if self.fp8_sustained:
            d["sustained_fp8_tflops"] = self.fp8_sustained
            d["sustained_source"] = (f"{self.src} bf16 sustained {self.fp8_sustained / FP8_OVER_BF16} TFLOP/s x "
                                     f"{FP8_OVER_BF16}; reported beside the burst-based peak, which stays the "
                                     "denominator: the GEMM's SM clock under load stays near its maximum")
        if self.probe:
            d["tensor_probe_tflops"] = self.probe
        return d


def measure_config(name: str, dev, stream, pk: Peaks, seconds: float, warmup: int, flush=None):
    """One configuration of the path: its quantizers and GEMM, repeated for
    at least `seconds` of GPU time with rotated inputs, CUDA events between
    kernels and nvidia-smi sampling the SM clocks (the step as training runs
    it: each kernel's time includes the write-back of what the previous one
    left dirty in L2); then each kernel alone after a read-only L2 flush (its
    own roofline).  Returns its record."""
    import torch

    from fp8_fine_grained_act_gb300 import binding as fb
    from fp8_fine_grained_act_gb300 import synth
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    rec = {}
    if name == "tiny":
        d = synth.tiny_fprop(seed=0)
        x, w = bf(d["x"]), torch.from_numpy(d["w"]).to(dev)
        Mw, Kw = x.shape
        Nw = w.shape[0]
        qx = torch.empty((Mw, Kw), dtype=torch.uint8, device=dev)
        sx = torch.empty((Kw // 128, Mw), dtype=torch.float32, device=dev)
        qw = torch.empty((Nw, Kw), dtype=torch.uint8, device=dev)
        sw = torch.empty((Nw // 128, Kw // 128), dtype=torch.float32, device=dev)
        y = torch.empty((Mw, Nw), dtype=torch.float32, device=dev)
        kernels = [("quant_act_1x128 X[256,512]", lambda i: fb.fp8_quant_act_1x128(x, q=qx, scales=sx, stream=stream)),
                   ("quant_w_128x128 W[256,512]", lambda i: fb.fp8_quant_w_128x128(w, q=qw, scales=sw, stream=stream)),
                   ("gemm_blockscaled 256x256x512 f32", lambda i: fb.fp8_gemm_blockscaled(
                       qx, sx, qw, sw, out_dtype=fb.FP8FG_OUT_F32, d=y, stream=stream))]
        nbytes = [Mw * Kw * ROW_B_PER_ELT, Nw * Kw * W_B_PER_ELT, None]
        flops = 2.0 * Mw * Nw * Kw
        workload = ("Tiny Fprop: X[256,512] N(0,1) with 0.1% of entries x100, W[256,512] N(0,0.02^2), fp32 out; "
                    "seed 0 (launch-latency bound: two 128x256 tiles)")
        sets = 1
    elif name == "dgrad":
        d = synth.dgrad(seed=2)
        Mw, Kw = d["dy"].shape
        Nw = d["w"].shape[1]
        sets = rotations(Mw * Kw * 2 + Kw * Nw * 4)
        dys = [bf(d["dy"]) for _ in range(sets)]
        ws = [torch.from_numpy(d["w"]).to(dev) for _ in range(sets)]
        del d
        qdy = torch.empty((Mw, Kw), dtype=torch.uint8, device=dev)
        sdy = torch.empty((Kw // 128, Mw), dtype=torch.float32, device=dev)
        qw = torch.empty((Kw, Nw), dtype=torch.uint8, device=dev)
        qwt = torch.empty((Nw, Kw), dtype=torch.uint8, device=dev)
        sw = torch.empty((Kw // 128, Nw // 128), dtype=torch.float32, device=dev)
        y = torch.empty((Mw, Nw), dtype=torch.bfloat16, device=dev)
        kernels = [("quant_act_1x128 dY[8192,2048]", lambda i: fb.fp8_quant_act_1x128(
                        dys[i % sets], q=qdy, scales=sdy, stream=stream)),
                   ("quant_w_128x128 W[2048,7168] + transposed copy", lambda i: fb.fp8_quant_w_128x128(
                       ws[i % sets], transposed=True, q=qw, q_t=qwt, scales=sw, stream=stream)),
                   ("gemm_blockscaled dgrad 8192x7168x2048 bf16", lambda i: fb.fp8_gemm_blockscaled(
                       qdy, sdy, qwt, sw, sb_strides=(1, Nw // 128), d=y, stream=stream))]
        nbytes = [Mw * Kw * ROW_B_PER_ELT, Kw * Nw * (W_B_PER_ELT + 1), None]
        flops = 2.0 * Mw * Nw * Kw
        workload = ("Dgrad: dX[8192,7168] = dY[8192,2048] . W[2048,7168]; dY = N(0,1) x exp(N(0,2)) per token, "
                    "quantized 1x128; W fp32 master quantized 128x128 with a transposed copy, block scales read "
                    "transposed; bf16 out; seed 2")
    elif name == "wgrad":
        d = synth.wgrad(seed=3)
        T, Mw = d["dy"].shape
        Nw = d["x"].shape[1]
        Kw = T
        sets = rotations(T * Mw * 2 + T * Nw * 2)
        dys = [bf(d["dy"]) for _ in range(sets)]
        xs = [bf(d["x"]) for _ in range(sets)]
        del d
        qa = torch.empty((Mw, T), dtype=torch.uint8, device=dev)
        sa = torch.empty((T // 128, Mw), dtype=torch.float32, device=dev)
        qb = torch.empty((Nw, T), dtype=torch.uint8, device=dev)
        sb = torch.empty((T // 128, Nw), dtype=torch.float32, device=dev)
        y = torch.empty((Mw, Nw), dtype=torch.float32, device=dev)
        kernels = [("quant_act_128x1 dY[8192,2048]", lambda i: fb.fp8_quant_act_1x128(
                        dys[i % sets], axis=fb.FP8FG_AXIS_ROWS, q=qa, scales=sa, stream=stream)),
                   ("quant_act_128x1 X[8192,7168]", lambda i: fb.fp8_quant_act_1x128(
                       xs[i % sets], axis=fb.FP8FG_AXIS_ROWS, q=qb, scales=sb, stream=stream)),
                   ("gemm_blockscaled wgrad 2048x7168x8192 per-row B scales f32", lambda i: fb.fp8_gemm_blockscaled(
                       qa, sa, qb, sb, bscale=fb.FP8FG_BSCALE_ROW, out_dtype=fb.FP8FG_OUT_F32, d=y, stream=stream))]
        nbytes = [T * Mw * ROW_B_PER_ELT, T * Nw * ROW_B_PER_ELT, None]
        flops = 2.0 * Mw * Nw * Kw
        workload = ("Wgrad: dW[2048,7168] = dY^T . X over 8192 tokens; dY as Dgrad, X as Fprop, both quantized in "
                    "128-token x 1-channel groups (transposed codes); per-row B scales; fp32 out; seed 3")
    elif name == "grouped":
        d = synth.grouped_moe(seed=4)
        G, Nw, Kw = d["w"].shape
        x = bf(d["x"])
        w = torch.from_numpy(d["w"].reshape(G * Nw, Kw)).to(dev)
        off = torch.from_numpy(d["offsets"]).to(dev)
        Mw = x.shape[0]
        del d
        sets = 1
        qx = torch.empty((Mw, Kw), dtype=torch.uint8, device=dev)
        sx = torch.empty((Kw // 128, Mw), dtype=torch.float32, device=dev)
        qw = torch.empty((G * Nw, Kw), dtype=torch.uint8, device=dev)
        sw = torch.empty((G * Nw // 128, Kw // 128), dtype=torch.float32, device=dev)
        y = torch.empty((Mw, Nw), dtype=torch.bfloat16, device=dev)
        qw3, sw3 = qw.view(G, Nw, Kw), sw.view(G, Nw // 128, Kw // 128)
        kernels = [(f"quant_act_1x128 X_all[{Mw},7168]", lambda i: fb.fp8_quant_act_1x128(
                        x, q=qx, scales=sx, stream=stream)),
                   ("quant_w_128x128 64 experts W_g[2048,7168]", lambda i: fb.fp8_quant_w_128x128(
                       w, q=qw, scales=sw, stream=stream)),
                   (f"gemm_grouped {Mw}x2048x7168 bf16", lambda i: fb.fp8_gemm_grouped(
                       qx, sx, qw3, sw3, off, d=y, stream=stream))]
        nbytes = [Mw * Kw * ROW_B_PER_ELT, G * Nw * Kw * W_B_PER_ELT, None]
        flops = 2.0 * Mw * Nw * Kw
        gemm_bytes = Mw * Kw + G * Nw * Kw + 4 * (Mw * Kw // 128 + G * Nw * Kw // 16384) + Mw * Nw * 2
        workload = (f"Grouped MoE Fprop: 64 experts W_g[2048,7168] fp32 N(0,0.02^2) quantized 128x128; "
                    f"Dirichlet(1)/multinomial counts over 32768 tokens padded to 128 (M_total {Mw}), X N(0,1) "
                    f"quantized 1x128; bf16 out; seed 4")
    else:
        raise ValueError(name)

    rounds = block_rounds(kernels, stream, seconds, warmup)
    with ClockSampler(dev.index or 0) as clk:
        per, block_ms = timed_rounds(kernels, rounds, stream)
    status = fb.fp8fg_last_device_status()
    if status != 0:
        raise SystemExit(f"{name}: device status {status}: {fb.fp8fg_status_string(status)}")
    alone = isolated_times(kernels, flush, stream, min(seconds, 0.5)) if flush is not None else [None] * len(kernels)
    for (kname, _), t, ta, nb in zip(kernels, per, alone, nbytes):
        if nb is None:
            extra = {}
            if name == "grouped":
                t_roof = max(flops / (pk.fp8 * 1e12), gemm_bytes / (pk.hbm * 1e9))
                extra = {"roofline_us": t_roof * 1e6, "frac_roofline": t_roof / (t * 1e-3),
                         "roofline": "max(2MNK / FP8 peak, minimum bytes / HBM)"}
            rec[kname] = pk.gemm(flops, t, extra)
            if ta is not None:
                rec[kname]["alone"] = pk.gemm(flops, ta)
        else:
            rec[kname] = pk.quant(nb, t)
            if ta is not None:
                rec[kname]["alone"] = pk.quant(nb, ta)
            if sets > 1 or name == "grouped":
                fn = dict(kernels)[kname]
                rec[kname]["b2b"] = pk.quant(nb, b2b_ms(fn, stream, min(seconds, 0.3)))
    rec["step"] = {"ms": sum(per), "TFLOP/s": flops / (sum(per) * 1e-3) / 1e12, "rounds": rounds,
                   "block_ms": block_ms, "input_sets": sets,
                   "l2": "inputs rotate over sets totalling > 2x L2" if sets > 1 else
                         ("one set larger than L2" if name == "grouped" else "launch-bound, fits in L2")}
    if name == "tiny":
        # the same three calls captured on the capture stream and replayed
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.graph(graph, stream=cap):
            fb.fp8_quant_act_1x128(x, q=qx, scales=sx, stream=cap)
            fb.fp8_quant_w_128x128(w, q=qw, scales=sw, stream=cap)
            fb.fp8_gemm_blockscaled(qx, sx, qw, sw, out_dtype=fb.FP8FG_OUT_F32, d=y, stream=cap)
        for _ in range(10):
            graph.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 2000
        g0.record(stream)
        for _ in range(reps):
            graph.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        gms = g0.elapsed_time(g1) / reps
        rec["step as one CUDA graph (3 kernels)"] = {"us": gms * 1e3, "TFLOP/s": flops / (gms * 1e-3) / 1e12}
    rec["clocks"] = clk.summary()
    rec["workload"] = workload
    rec["M_N_K"] = [int(Mw), int(Nw), int(Kw)]
    rec["gpu_launches"] = len(kernels) * rounds
    return rec, flops, sum(per)


def measure_dual(dev, stream, pk: Peaks, seconds: float):
    """The fused 1x128 + 128x1 quantizer on X[4096,7168] and X[8192,7168]
    (what a training forward runs to cache X in FP8 for the weight
    gradient), inputs rotated over more than twice the L2."""
    import torch

    from fp8_fine_grained_act_gb300 import binding as fb
    out = {}
    for rows in (4096, 8192):
        cols = 7168
        sets = rotations(rows * cols * 2)
        gen = torch.Generator(device=dev).manual_seed(5)
        base = torch.randn((rows, cols), device=dev, generator=gen, dtype=torch.float32).to(torch.bfloat16)
        xs = [base.clone() for _ in range(sets)]
        qr = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
        sr = torch.empty((cols // 128, rows), dtype=torch.float32, device=dev)
        qc = torch.empty((cols, rows), dtype=torch.uint8, device=dev)
        sc = torch.empty((rows // 128, cols), dtype=torch.float32, device=dev)
        kern = [("dual", lambda i: fb.fp8_quant_act_dual(xs[i % sets], q_row=qr, s_row=sr, q_col_t=qc, s_col=sc,
                                                         stream=stream))]
        rounds = block_rounds(kern, stream, seconds, 5)
        with ClockSampler(dev.index or 0) as clk:
            per, _ = timed_rounds(kern, rounds, stream)
        r = pk.quant(rows * cols * DUAL_B_PER_ELT, per[0])
        r.update({"rounds": rounds, "input_sets": sets, "clocks": clk.summary()})
        r["b2b"] = pk.quant(rows * cols * DUAL_B_PER_ELT, b2b_ms(kern[0][1], stream, min(seconds, 0.3)))
        out[f"quant_act_dual_1x128_128x1 X[{rows},{cols}]"] = r
        del xs, base
    if fb.fp8fg_last_device_status() != 0:
        raise SystemExit("dual quantizer: device status not clean")
    return out


def run_gpu(args):
    import torch
    import torch.distributed as dist

    from fp8_fine_grained_act_gb300 import binding as fb
    from fp8_fine_grained_act_gb300 import synth

    rank, world, local = dist_env()
    dev = _gpu_setup(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

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

    # soak: the same step for at least --soak seconds right before the timed
    # steps, so that the clock sampler sees the GPU under this load
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(5):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    soak_steps = int(max(1, math.ceil(args.soak * 1e3 / max(e0.elapsed_time(e1) / 5, 1e-3))))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        e0.record(stream)
        for _ in range(soak_steps):
            step()
        e1.record(stream)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(args.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        # the per-kernel breakdown: the same steps again with an event between
        # kernels, outside the timed region (an event pair around a launch
        # serialises it with its neighbours and costs a small kernel a few
        # microseconds, which the timed steps must not carry)
        for i in range(args.steps):
            step(evs[i])
        torch.cuda.synchronize()
    soak_ms = e0.elapsed_time(e1) / soak_steps
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

    # the activation quantizer fused into the GEMM (one launch): the same
    # step with fp8_gemm_quant_a in place of the 1x128 quantizer + GEMM
    flags = torch.empty((M // 128,), dtype=torch.int32, device=dev)
    fused_k = [("w", lambda i: fb.fp8_quant_w_128x128(w, q=qw, scales=sw, stream=stream)),
               ("fused", lambda i: fb.fp8_gemm_quant_a(x, qw, sw, out_dtype=fb.FP8FG_OUT_BF16, q_a=qx, s_a=sx,
                                                       d=y, band_flags=flags, stream=stream))]
    f_rounds = block_rounds(fused_k, stream, min(args.block_seconds, 1.0), 3)
    with ClockSampler(local) as clk_f:
        f_per, _ = timed_rounds(fused_k, f_rounds, stream)
    if fb.fp8fg_last_device_status() != 0:
        raise SystemExit("fused step: device status not clean")
    t_fused = max_over_ranks(f_per[1])
    t_fused_step = max_over_ranks(sum(f_per))

    ms_step = max_over_ranks(total_ms / args.steps)
    t_gemm = max_over_ranks(t_gemm)
    t_act = max_over_ranks(t_act)
    t_w = max_over_ranks(t_w)
    single = world == 1 and args.configs == "all"
    probe = probe_tensor_rate(fb, stream) if single else None
    pk = Peaks(probe)
    kernels = {"fprop": {"quant_act_1x128 X[4096,7168]": pk.quant(ACT_BYTES, t_act),
                         "quant_w_128x128 W[18432,7168]": pk.quant(W_BYTES, t_w),
                         "gemm_blockscaled fprop 4096x18432x7168 bf16": pk.gemm(FLOPS, t_gemm),
                         "step": {"ms": ms_step, "soak_ms_per_step": soak_ms, "soak_steps": soak_steps,
                                  "l2": "inputs larger than L2: each step reads X (58.7 MB) and W (528 MB)"},
                         "gemm_quant_a (1x128 quantizer fused into the GEMM, one launch)": pk.gemm(
                             FLOPS, t_fused, {"two_launches_us": (t_act + t_gemm) * 1e3,
                                              "step_with_fused_ms": t_fused_step, "rounds": f_rounds,
                                              "clocks": clk_f.summary()}),
                         "clocks": clk.summary()}}
    launches = 3 * args.steps
    if single:
        flush = L2Flush(dev)
        fk = [("a", lambda i: fb.fp8_quant_act_1x128(x, q=qx, scales=sx, stream=stream)),
              ("w", lambda i: fb.fp8_quant_w_128x128(w, q=qw, scales=sw, stream=stream)),
              ("g", lambda i: fb.fp8_gemm_blockscaled(qx, sx, qw, sw, out_dtype=fb.FP8FG_OUT_BF16, d=y,
                                                      stream=stream))]
        ta, tw, tg = isolated_times(fk, flush, stream, 0.5)
        f = kernels["fprop"]
        f["quant_act_1x128 X[4096,7168]"]["alone"] = pk.quant(ACT_BYTES, ta)
        f["quant_w_128x128 W[18432,7168]"]["alone"] = pk.quant(W_BYTES, tw)
        f["gemm_blockscaled fprop 4096x18432x7168 bf16"]["alone"] = pk.gemm(FLOPS, tg)
        # back to back: X rotated over more than twice the L2; W alone is larger than L2
        xsets = rotations(M * K * 2)
        xs = [x.clone() for _ in range(xsets)]
        f["quant_act_1x128 X[4096,7168]"]["b2b"] = pk.quant(ACT_BYTES, b2b_ms(
            lambda i: fb.fp8_quant_act_1x128(xs[i % xsets], q=qx, scales=sx, stream=stream), stream, 0.3))
        f["quant_w_128x128 W[18432,7168]"]["b2b"] = pk.quant(W_BYTES, b2b_ms(
            lambda i: fb.fp8_quant_w_128x128(w, q=qw, scales=sw, stream=stream), stream, 0.3))
        del xs
        del x_h, w_h, y_h, yhs
        torch.cuda.empty_cache()
        kernels.update(measure_dual(dev, stream, pk, args.block_seconds))
        for name in ("tiny", "dgrad", "wgrad", "grouped"):
            rec, _, _ = measure_config(name, dev, stream, pk, args.block_seconds, args.warmup, flush)
            kernels[name] = rec
            torch.cuda.empty_cache()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    gemm_tflops = FLOPS / (t_gemm * 1e-3) / 1e12
    roof = {"bound": "tensor", "achieved": gemm_tflops, "peak": pk.fp8, "unit": "TFLOP/s",
            "frac": gemm_tflops / pk.fp8, "traffic": profiled_traffic(),
            "kernel": "gemm_blockscaled_kernel<0>",
            "peak_source": f"{pk.src} bf16 burst {pk.bf16} TFLOP/s x {FP8_OVER_BF16} (FP8:BF16 nominal ratio)",
            "frac_nominal_fp8": gemm_tflops / NOMINAL_FP8_TFLOPS}
    if pk.fp8_sustained:
        roof["frac_sustained_fp8"] = gemm_tflops / pk.fp8_sustained
        roof["sustained_fp8_tflops"] = pk.fp8_sustained
    if probe:
        roof["frac_tensor_probe"] = gemm_tflops / probe["tflops"]
        roof["tensor_probe_tflops"] = probe["tflops"]
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
        "roofline": roof,
        "kernels": kernels,
        "peaks": pk.legend(),
        "e2e": {"value": world * FLOPS / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": M * K * 2 + N * K * 4,
                "d2h_bytes_per_step": M * N * 2, "ms_per_step": e2e_ms, "steps": e2e_steps,
                "how": "copies of step i+1 (H2D) and i-1 (D2H) overlap step i's kernels on separate streams",
                "serial_ms_per_step": e2e_serial_ms},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    if probe:
        line["tensor_probe"] = probe
    if not args.no_cpu_baseline:
        mb, nb = 1024, 4096
        v, cores, dt = cpu_baseline(mb, nb)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": f"first {mb} tokens x {nb} output channels of the workload: both "
                                          f"quantizers + {mb}x{nb}x{K} double GEMM, {dt:.1f} s",
                                "quantizers_1core": cpu_quantizers_1core(1024)}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_other(args):
    """One configuration alone (single GPU): a line of the same metric with
    its per-kernel breakdown."""
    import torch
    from fp8_fine_grained_act_gb300 import binding as fb
    dev = _gpu_setup(0)
    stream = torch.cuda.current_stream()
    pk = Peaks()
    rec, flops, ms = measure_config(args.workload, dev, stream, pk, args.block_seconds, args.warmup,
                                    L2Flush(dev) if args.alone else None)
    line = {"metric": METRIC, "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": rec["step"]["rounds"], "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": {"workload": rec["workload"], "M_N_K": rec["M_N_K"], "parallelism": "single GPU"},
            "kernels": {args.workload: rec}, "peaks": pk.legend(), "clocks": rec["clocks"],
            "gpu_launches": rec["gpu_launches"]}
    del fb
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["fprop", "tiny", "dgrad", "wgrad", "grouped"], default="fprop")
    ap.add_argument("--configs", choices=["all", "none"], default="all",
                    help="with the Fprop step, also measure the other configurations (N = 1 only)")
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of the Fprop step before the timed steps")
    ap.add_argument("--block-seconds", type=float, default=1.0, help="GPU seconds of each configuration's block")
    ap.add_argument("--alone", action="store_true",
                    help="with --workload: also time each kernel alone after an L2 flush")
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
