"""fp8_gemm_quant_a_noalloc through the C ABI: the fused 1x128 quantizer +
block-scaled GEMM for callers that cannot allocate device memory (no
allocator of their own, or a steady state that must not allocate).  It keeps
its band counters in a fixed array in the library instead of a workspace the
caller passes, so its results must equal fp8_gemm_quant_a's bit for bit and
lie within the oracle's tolerance, call after call: the array keeps the last
call's counters, and each call must clear them itself.

This file is collected last, so that it runs both in a fresh process (where
its first call looks up the array's address) and after every other test.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_act_gb300 import binding as fb
from fp8_fine_grained_act_gb300 import synth
from gpu_util import assert_gemm_close, dev, dev_bf16, host

BF16, F32 = fb.FP8FG_OUT_BF16, fb.FP8FG_OUT_F32
ODT = {BF16: "bf16", F32: "f32"}
MAX_M = 4096 * 128


def _noalloc(x, qw, sw, out_dtype, sb_strides=None):
    """One call of the no-allocation entry point on fresh outputs."""
    M, K = x.shape
    N = qw.shape[0]
    sn, sk = sb_strides if sb_strides is not None else (K // 128, 1)
    q_a = torch.full((M, K), 0x7F, dtype=torch.uint8, device=x.device)
    s_a = torch.full((K // 128, M), -1.0, dtype=torch.float32, device=x.device)
    d = torch.full((M, N), 7.0, dtype=torch.float32 if out_dtype == F32 else torch.bfloat16, device=x.device)
    st = fb.load().fp8_gemm_quant_a_noalloc(x.data_ptr(), q_a.data_ptr(), s_a.data_ptr(), qw.data_ptr(),
                                            sw.data_ptr(), sn, sk, d.data_ptr(), out_dtype, M, N, K,
                                            torch.cuda.current_stream(x.device).cuda_stream)
    assert st == 0, fb.status_string(st)
    return d, q_a, s_a


def _bits(t):
    a = host(t) if t.dtype != torch.bfloat16 else t.view(torch.int16).cpu().numpy()
    return a.view(np.uint32) if a.dtype == np.float32 else a


def _check_pair(x_bits, x, qw, sw, out_dtype, sb_strides=None):
    """Two no-allocation calls in a row, each against fp8_gemm_quant_a (its
    own zeroed workspace) bit for bit and against the oracle."""
    ref_d, ref_q, ref_s = fb.fp8_gemm_quant_a(x, qw, sw, sb_strides=sb_strides, out_dtype=out_dtype)
    first = _noalloc(x, qw, sw, out_dtype, sb_strides)
    second = _noalloc(x, qw, sw, out_dtype, sb_strides)
    torch.cuda.synchronize()
    assert fb.fp8fg_last_device_status() == 0
    qxo, sxo = oracle.quant_act(x_bits)
    o, m = oracle.gemm(qxo, sxo, host(qw), host(sw), sb_strides=sb_strides)
    for i, (d, q, s) in enumerate((first, second)):
        assert np.array_equal(_bits(q), _bits(ref_q)) and np.array_equal(_bits(s), _bits(ref_s)), f"call {i}"
        assert np.array_equal(_bits(d), _bits(ref_d)), f"call {i}: output differs from fp8_gemm_quant_a"
        assert np.array_equal(host(q), qxo)
        assert_gemm_close(host(d), o, m, ODT[out_dtype], f"no-allocation call {i}")


@pytest.mark.gpu
@pytest.mark.parametrize("out_dtype", [BF16, F32])
def test_two_calls_match_fused_entry_point(gpu_device, out_dtype):
    """Fprop roles, several tiles with a ragged N tile."""
    d = synth.fprop_linear(seed=11, M=512, N=640, K=640)
    x = dev_bf16(d["x"], gpu_device)
    qw, sw = fb.fp8_quant_w_128x128(dev(d["w"], gpu_device))
    _check_pair(d["x"], x, qw, sw, out_dtype)


@pytest.mark.gpu
def test_larger_then_smaller_problem(gpu_device):
    """A call over more bands leaves more counters set; the next, smaller,
    call (Dgrad roles: transposed weight codes, swapped scale strides) must
    not see them."""
    big = synth.fprop_linear(seed=12, M=2048, N=512, K=1024)
    xb = dev_bf16(big["x"], gpu_device)
    qwb, swb = fb.fp8_quant_w_128x128(dev(big["w"], gpu_device))
    _check_pair(big["x"], xb, qwb, swb, BF16)
    small = synth.dgrad(seed=13, M=384, N=768, K=384)
    dy = dev_bf16(small["dy"], gpu_device)
    _, qwt, sw = fb.fp8_quant_w_128x128(dev(small["w"], gpu_device), transposed=True)
    _check_pair(small["dy"], dy, qwt, sw, BF16, sb_strides=(1, small["w"].shape[1] // 128))


@pytest.mark.gpu
def test_rejects_more_rows_than_the_array_covers(gpu_device):
    """M beyond 4096 bands of 128 rows is refused before anything runs."""
    lib = fb.load()
    st = lib.fp8_gemm_quant_a_noalloc(None, None, None, None, None, 1, 1, None, BF16, MAX_M + 128, 128, 128,
                                      torch.cuda.current_stream(gpu_device).cuda_stream)
    assert st == fb.FP8FG_ERR_TOO_LARGE
    assert "524288" in fb.status_string(st)
    assert fb.fp8fg_last_device_status() == 0
