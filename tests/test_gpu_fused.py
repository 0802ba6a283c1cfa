"""GPU parity of fp8_gemm_quant_a, the 1x128 activation quantizer fused into
the block-scaled GEMM (one cooperative launch), through the C ABI.

The fused call must write exactly what the two-call path writes:
fp8_quant_act_1x128 on the BF16 operand (codes and scales, bit for bit) and
fp8_gemm_blockscaled on those codes (the same GEMM arithmetic, so the output
is bit-identical too).  The oracle pins both: the codes and scales against
its quantizer, the output within |d - o| <= 2^-16 * sum|a~ b~| (+ one BF16
spacing for BF16 output).  Shapes: the tiny Fprop, medium shapes spanning
several tiles with a ragged N tile and more 128-row bands than CTAs of one
wave would hold, the Dgrad operand roles (transposed weight codes, block
scales read through swapped strides), the full Fprop layer on sampled
outputs; the workspace reused by consecutive calls (the call zeroes it), a
poisoned workspace, N = 0 (the quantizer alone) and K = 0.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_act_gb300 import binding as fb
from fp8_fine_grained_act_gb300 import synth
from gpu_util import assert_gemm_close, dev, dev_bf16, host

pytestmark = pytest.mark.gpu

BF16, F32 = fb.FP8FG_OUT_BF16, fb.FP8FG_OUT_F32
ODT = {BF16: "bf16", F32: "f32"}


def _same(a, b):
    a, b = host(a), host(b)
    return np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                          b.view(np.uint32) if b.dtype == np.float32 else b)


def _two_calls(x, qw, sw, out_dtype, sb_strides=None):
    qx, sx = fb.fp8_quant_act_1x128(x)
    y = fb.fp8_gemm_blockscaled(qx, sx, qw, sw, sb_strides=sb_strides, out_dtype=out_dtype)
    return y, qx, sx


@pytest.mark.parametrize("out_dtype", [F32, BF16])
def test_tiny_fprop_fused_equals_two_calls_and_oracle(gpu_device, out_dtype):
    d = synth.tiny_fprop(seed=0)
    x = dev_bf16(d["x"], gpu_device)
    qw, sw = fb.fp8_quant_w_128x128(dev(d["w"], gpu_device))
    y, qa, sa = fb.fp8_gemm_quant_a(x, qw, sw, out_dtype=out_dtype)
    y2, qx, sx = _two_calls(x, qw, sw, out_dtype)
    torch.cuda.synchronize()
    assert fb.fp8fg_last_device_status() == 0
    assert _same(qa, qx) and _same(sa, sx) and _same(y, y2)
    qxo, sxo = oracle.quant_act(d["x"])
    assert np.array_equal(host(qa), qxo) and np.array_equal(host(sa).view(np.uint32), sxo.view(np.uint32))
    o, m = oracle.gemm(qxo, sxo, host(qw), host(sw))
    assert_gemm_close(host(y), o, m, ODT[out_dtype], "fused tiny fprop")


@pytest.mark.parametrize("M,N,K", [(384, 640, 640), (128, 128, 128), (4096, 512, 256), (640, 2304, 1280)])
def test_medium_fused(gpu_device, M, N, K):
    d = synth.fprop_linear(seed=7, M=M, N=N, K=K)
    x = dev_bf16(d["x"], gpu_device)
    qw, sw = fb.fp8_quant_w_128x128(dev(d["w"], gpu_device))
    y, qa, sa = fb.fp8_gemm_quant_a(x, qw, sw, out_dtype=BF16)
    y2, qx, sx = _two_calls(x, qw, sw, BF16)
    torch.cuda.synchronize()
    assert fb.fp8fg_last_device_status() == 0
    assert _same(qa, qx) and _same(sa, sx) and _same(y, y2)
    qxo, sxo = oracle.quant_act(d["x"])
    assert np.array_equal(host(qa), qxo)
    o, m = oracle.gemm(qxo, sxo, host(qw), host(sw))
    assert_gemm_close(host(y), o, m, "bf16", f"fused {M}x{N}x{K}")


def test_dgrad_roles_fused(gpu_device):
    """dX = dY . W: the weight's transposed codes as B, its block scales read
    through swapped strides, dY quantized inside the GEMM."""
    d = synth.dgrad(seed=2, M=512, N=768, K=384)
    dy = dev_bf16(d["dy"], gpu_device)
    _, qwt, sw = fb.fp8_quant_w_128x128(dev(d["w"], gpu_device), transposed=True)
    nw = d["w"].shape[1] // 128
    dx, qa, sa = fb.fp8_gemm_quant_a(dy, qwt, sw, sb_strides=(1, nw), out_dtype=BF16)
    dx2, qd, sd = _two_calls(dy, qwt, sw, BF16, sb_strides=(1, nw))
    torch.cuda.synchronize()
    assert _same(qa, qd) and _same(sa, sd) and _same(dx, dx2)
    qdo, sdo = oracle.quant_act(d["dy"])
    o, m = oracle.gemm(qdo, sdo, host(qwt), host(sw), sb_strides=(1, nw))
    assert_gemm_close(host(dx), o, m, "bf16", "fused dgrad")


def test_full_fprop_sampled(gpu_device):
    """The Fprop layer X[4096,7168] . W[18432,7168]^T: codes and scales
    equal the standalone quantizer's, the output equals the two-call path's
    bit for bit, and sampled outputs are within the oracle's tolerance."""
    d = synth.fprop_linear(seed=1)
    x = dev_bf16(d["x"], gpu_device)
    qw, sw = fb.fp8_quant_w_128x128(dev(d["w"], gpu_device))
    y, qa, sa = fb.fp8_gemm_quant_a(x, qw, sw, out_dtype=BF16)
    y2, qx, sx = _two_calls(x, qw, sw, BF16)
    torch.cuda.synchronize()
    assert fb.fp8fg_last_device_status() == 0
    assert _same(qa, qx) and _same(sa, sx) and torch.equal(y.view(torch.int16), y2.view(torch.int16))
    rng = np.random.default_rng(3)
    ii, jj = rng.integers(0, 4096, 256), rng.integers(0, 18432, 256)
    qxo, sxo = oracle.quant_act(d["x"])
    assert np.array_equal(host(qa), qxo)
    o, m = oracle.gemm_entries(qxo, sxo, host(qw), host(sw), ii, jj)
    err = np.abs(host(y)[ii, jj].astype(np.float64) - o)
    assert np.all(err <= oracle.gemm_tolerance(o, m, "bf16"))


def test_workspace_reused_and_poisoned(gpu_device):
    """The call zeroes its band counters itself: two calls in a row on one
    workspace, and a workspace full of garbage, give the same result."""
    d = synth.fprop_linear(seed=5, M=512, N=512, K=512)
    x = dev_bf16(d["x"], gpu_device)
    qw, sw = fb.fp8_quant_w_128x128(dev(d["w"], gpu_device))
    flags = torch.full((4,), 123456, dtype=torch.int32, device=gpu_device)
    y0, _, _ = fb.fp8_gemm_quant_a(x, qw, sw, out_dtype=F32, band_flags=flags)
    y1, _, _ = fb.fp8_gemm_quant_a(x, qw, sw, out_dtype=F32, band_flags=flags)
    torch.cuda.synchronize()
    assert fb.fp8fg_last_device_status() == 0
    assert _same(y0, y1)
    y2, _, _ = _two_calls(x, qw, sw, F32)
    assert _same(y0, y2)


def test_degenerate_shapes(gpu_device):
    x = dev_bf16(synth.activations_random_outliers(np.random.default_rng(1), 256, 384), gpu_device)
    # N = 0: the quantizer alone
    b = torch.empty((0, 384), dtype=torch.uint8, device=gpu_device)
    sb = torch.empty((0, 3), dtype=torch.float32, device=gpu_device)
    y, qa, sa = fb.fp8_gemm_quant_a(x, b, sb, out_dtype=F32)
    qx, sx = fb.fp8_quant_act_1x128(x)
    torch.cuda.synchronize()
    assert y.shape == (256, 0) and _same(qa, qx) and _same(sa, sx)
    # K = 0: D = 0
    x0 = torch.empty((256, 0), dtype=torch.bfloat16, device=gpu_device)
    b0 = torch.empty((128, 0), dtype=torch.uint8, device=gpu_device)
    d0 = torch.full((256, 128), 5.0, dtype=torch.float32, device=gpu_device)
    fb.fp8_gemm_quant_a(x0, b0, torch.empty((1, 0), dtype=torch.float32, device=gpu_device), out_dtype=F32, d=d0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(d0).item() == 0
