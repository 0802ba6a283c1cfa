"""GPU parity of the GEMM around the persistent grid's wave boundaries.

The grid holds min(T, P) CTAs for T output tiles of 128 x 256 on P SMs, and
CTA b takes tiles b, b + P, b + 2P, ...; so around T = P and T = 2P the CTAs
differ in their tile counts, and the last tile column (N = 640: 2.5 tiles) is
half empty.  Tile counts are chosen from the device's SM count; block and
per-row B scales and both output types are covered; the whole output is
compared with the oracle on operands quantized by the GPU.
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

N_COLS = 640            # 3 tile columns, the last one holding 128 columns
N_TILE_COLS = 3
K_DEPTH = 384           # 3 chunks: every prefetched A scale is used


def _tiles_near(target: int) -> int:
    """The multiple of 3 (3 tile columns) nearest to target, at least 3."""
    return max(N_TILE_COLS, N_TILE_COLS * round(target / N_TILE_COLS))


CASES = [
    # (tile count relative to P, B scale mode, output)
    ("P-1", "block", "bf16"), ("P+1", "block", "f32"), ("P+1", "row", "bf16"),
    ("2P-1", "row", "f32"), ("2P+1", "block", "bf16"), ("P/2", "block", "f32"),
]


@pytest.mark.parametrize("where,bmode,odt", CASES)
def test_wave_boundaries(gpu_device, where, bmode, odt):
    sms = torch.cuda.get_device_properties(gpu_device).multi_processor_count
    target = {"P-1": sms - 1, "P+1": sms + 1, "2P-1": 2 * sms - 1, "2P+1": 2 * sms + 1, "P/2": sms // 2}[where]
    tiles = _tiles_near(target)
    M, N, K = 128 * (tiles // N_TILE_COLS), N_COLS, K_DEPTH
    out_dtype = fb.FP8FG_OUT_BF16 if odt == "bf16" else fb.FP8FG_OUT_F32
    rng = np.random.default_rng(700 + CASES.index((where, bmode, odt)))
    if bmode == "row":
        a_src = synth.gradients_token_outliers(rng, K, M)
        b_src = synth.activations_channel_outliers(rng, K, N)
        qa, sa = fb.fp8_quant_act_1x128(dev_bf16(a_src, gpu_device), axis=fb.FP8FG_AXIS_ROWS)
        qb, sb = fb.fp8_quant_act_1x128(dev_bf16(b_src, gpu_device), axis=fb.FP8FG_AXIS_ROWS)
        d = fb.fp8_gemm_blockscaled(qa, sa, qb, sb, bscale=fb.FP8FG_BSCALE_ROW, out_dtype=out_dtype)
        qa_o, sa_o = oracle.quant_act(a_src, axis=1)
        qb_o, sb_o = oracle.quant_act(b_src, axis=1)
        bscale = oracle.BSCALE_ROW
    else:
        a_src = synth.activations_random_outliers(rng, M, K)
        b_src = synth.master_weight(rng, N, K)
        qa, sa = fb.fp8_quant_act_1x128(dev_bf16(a_src, gpu_device))
        qb, sb = fb.fp8_quant_w_128x128(dev(b_src, gpu_device))
        d = fb.fp8_gemm_blockscaled(qa, sa, qb, sb, out_dtype=out_dtype)
        qa_o, sa_o = oracle.quant_act(a_src)
        qb_o, sb_o = oracle.quant_w(b_src)
        bscale = oracle.BSCALE_BLOCK128
    torch.cuda.synchronize()
    assert np.array_equal(host(qa), qa_o) and np.array_equal(host(qb), qb_o)
    assert np.array_equal(host(sa).view(np.uint32), sa_o.view(np.uint32))
    assert np.array_equal(host(sb).view(np.uint32), sb_o.view(np.uint32))
    o, m = oracle.gemm(qa_o, sa_o, qb_o, sb_o, bscale=bscale)
    assert_gemm_close(host(d), o, m, odt, f"{where} {bmode} {M}x{N}x{K}")
