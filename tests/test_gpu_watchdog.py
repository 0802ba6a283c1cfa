"""Bounded device waits: a kernel whose mbarrier is never signalled gives up
after its limit, records FP8FG_ERR_TIMEOUT in the device status word and
returns; the context stays usable.  The GEMM's own waits, and those of the
fused quantizer + GEMM, are made to run out with a 1 ns limit.  No fault,
trap or hang is involved."""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_act_gb300 import binding as fb
from fp8_fine_grained_act_gb300 import synth
from gpu_util import dev, dev_bf16, host

pytestmark = pytest.mark.gpu


def test_wait_times_out_and_reports(gpu_device):
    fb.fp8fg_last_device_status()                            # clear
    t0 = time.perf_counter()
    assert fb.fp8fg_selftest_watchdog(2_000_000) == 0        # 2 ms limit
    assert fb.fp8fg_last_device_status() == fb.FP8FG_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert fb.fp8fg_last_device_status() == 0                # read clears it
    # the context still works
    x = synth.activations_random_outliers(np.random.default_rng(0), 4, 128)
    q, s = fb.fp8_quant_act_1x128(dev_bf16(x, gpu_device))
    torch.cuda.synchronize()
    assert host(s).shape == (1, 4)


@pytest.mark.parametrize("bscale", [fb.FP8FG_BSCALE_BLOCK128, fb.FP8FG_BSCALE_ROW])
def test_gemm_waits_run_out_and_the_kernel_ends(gpu_device, bscale):
    """With a 1 ns limit the GEMM's producer, operand-watcher and scale-ring
    waits give up almost at once: every CTA must still end (the watcher and
    the promotion warps keep their lock step with the MMA warp), report
    FP8FG_ERR_TIMEOUT, and leave a context in which the next call with the
    default limit is correct."""
    M, N, K = 512, 1024, 4096
    rng = np.random.default_rng(11)
    a = torch.from_numpy(rng.integers(0, 0x7E, (M, K), dtype=np.uint8)).to(gpu_device)
    b = torch.from_numpy(rng.integers(0, 0x7E, (N, K), dtype=np.uint8)).to(gpu_device)
    sa = torch.full((K // 128, M), 1.0 / 64, device=gpu_device)
    sb = (torch.full((N // 128, K // 128), 1.0 / 64, device=gpu_device) if bscale == fb.FP8FG_BSCALE_BLOCK128
          else torch.full((K // 128, N), 1.0 / 64, device=gpu_device))
    fb.fp8fg_last_device_status()                            # clear
    assert fb.fp8fg_set_wait_limit(1) == 0
    try:
        t0 = time.perf_counter()
        fb.fp8_gemm_blockscaled(a, sa, b, sb, bscale=bscale, out_dtype=fb.FP8FG_OUT_F32)
        st = fb.fp8fg_last_device_status()
        assert time.perf_counter() - t0 < 30.0
    finally:
        assert fb.fp8fg_set_wait_limit(0) == 0
    assert st == fb.FP8FG_ERR_TIMEOUT
    # the next call, with the default limit, is correct (sampled entries)
    d = fb.fp8_gemm_blockscaled(a, sa, b, sb, bscale=bscale, out_dtype=fb.FP8FG_OUT_F32)
    assert fb.fp8fg_last_device_status() == 0
    ii, jj = rng.integers(0, M, 64), rng.integers(0, N, 64)
    o, m = oracle.gemm_entries(host(a), host(sa), host(b), host(sb), ii, jj,
                               bscale=oracle.BSCALE_BLOCK128 if bscale == fb.FP8FG_BSCALE_BLOCK128 else oracle.BSCALE_ROW)
    assert np.all(np.abs(host(d)[ii, jj] - o) <= oracle.gemm_tolerance(o, m, "f32"))


def test_fused_quantizer_waits_run_out_and_the_kernel_ends(gpu_device):
    """fp8_gemm_quant_a with a 1 ns limit: the phase-1 ring's waits and the
    band waits (each lane of warp 0 polling its own band counters) give up,
    every CTA ends without computing, FP8FG_ERR_TIMEOUT is reported, and the
    next call with the default limit equals the two-launch path (quantizer,
    then GEMM) bit for bit."""
    d = synth.fprop_linear(seed=21, M=1024, N=512, K=1024)
    x = dev_bf16(d["x"], gpu_device)
    qw, sw = fb.fp8_quant_w_128x128(dev(d["w"], gpu_device))
    torch.cuda.synchronize()
    fb.fp8fg_last_device_status()                            # clear
    assert fb.fp8fg_set_wait_limit(1) == 0
    try:
        t0 = time.perf_counter()
        fb.fp8_gemm_quant_a(x, qw, sw, out_dtype=fb.FP8FG_OUT_F32)
        st = fb.fp8fg_last_device_status()
        assert time.perf_counter() - t0 < 30.0
    finally:
        assert fb.fp8fg_set_wait_limit(0) == 0
    assert st == fb.FP8FG_ERR_TIMEOUT
    y, q_a, s_a = fb.fp8_gemm_quant_a(x, qw, sw, out_dtype=fb.FP8FG_OUT_F32)
    qa_ref, sa_ref = fb.fp8_quant_act_1x128(x)
    y_ref = fb.fp8_gemm_blockscaled(qa_ref, sa_ref, qw, sw, out_dtype=fb.FP8FG_OUT_F32)
    torch.cuda.synchronize()
    assert fb.fp8fg_last_device_status() == 0
    assert torch.equal(q_a, qa_ref) and torch.equal(s_a, sa_ref)
    assert torch.equal(y.view(torch.int32), y_ref.view(torch.int32))
