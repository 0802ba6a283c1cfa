"""GPU parity of the three quantizers, through the C ABI: E4M3 bytes and FP32
scales must equal the oracle's bit for bit.

Shapes: the tiny and full workloads (Fprop X[4096,7168], Dgrad dY[8192,2048],
Wgrad X[8192,7168] transposed, W[2048,7168] with its transposed copy), ragged
row counts and channel counts, sampled blocks of the full-size weights
(W[18432,7168]; the 64 expert weights), and the edge cases: empty input,
all-zero groups, groups whose scale is subnormal or underflows, and a dense
sweep of (value, group maximum) BF16 pairs.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_act_gb300 import binding as fb
from fp8_fine_grained_act_gb300 import synth
from gpu_util import dev, dev_bf16, host

pytestmark = pytest.mark.gpu


def _act_parity(xb: np.ndarray, axis: int, device):
    q, s = fb.fp8_quant_act_1x128(dev_bf16(xb, device), axis=axis)
    torch.cuda.synchronize()
    qo, so = oracle.quant_act(xb, axis=axis)
    qg, sg = host(q), host(s)
    assert sg.shape == so.shape and qg.shape == qo.shape
    assert np.array_equal(sg.view(np.uint32), so.view(np.uint32)), "scales differ"
    nbad = int(np.count_nonzero(qg != qo))
    assert nbad == 0, f"{nbad} E4M3 codes differ"


@pytest.mark.parametrize("shape", [(256, 512), (1, 128), (37, 384), (300, 1024)])
def test_act_rows_small(gpu_device, shape):
    rng = np.random.default_rng(100 + shape[0])
    _act_parity(synth.activations_random_outliers(rng, *shape), 0, gpu_device)


@pytest.mark.parametrize("shape", [(128, 64), (256, 8), (384, 200), (512, 1000), (640, 384)])
def test_act_cols_small(gpu_device, shape):
    rng = np.random.default_rng(200 + shape[1])
    _act_parity(synth.gradients_token_outliers(rng, *shape), 1, gpu_device)


def test_act_rows_full_fprop_x(gpu_device):
    _act_parity(synth.fprop_linear(seed=1, N=128)["x"], 0, gpu_device)


def test_act_rows_full_dgrad_dy(gpu_device):
    _act_parity(synth.dgrad(seed=2, N=128)["dy"], 0, gpu_device)


def test_act_cols_full_wgrad(gpu_device):
    d = synth.wgrad(seed=3)
    _act_parity(d["dy"], 1, gpu_device)
    _act_parity(d["x"], 1, gpu_device)


def _w_parity(w: np.ndarray, device, transposed=True):
    out = fb.fp8_quant_w_128x128(dev(w, device), transposed=transposed)
    torch.cuda.synchronize()
    ref = oracle.quant_w(w, transposed=transposed)
    if transposed:
        (q, qt, s), (qo, so, qto) = out, ref
        assert np.array_equal(host(qt), qto), "transposed codes differ"
    else:
        (q, s), (qo, so) = out, ref
    assert np.array_equal(host(s).view(np.uint32), so.view(np.uint32)), "scales differ"
    assert np.array_equal(host(q), qo), "codes differ"


@pytest.mark.parametrize("shape", [(128, 128), (256, 512), (384, 1280)])
def test_weight_small(gpu_device, shape):
    _w_parity(synth.master_weight(np.random.default_rng(shape[1]), *shape), gpu_device)


def test_weight_full_dgrad(gpu_device):
    _w_parity(synth.dgrad(seed=2, M=128)["w"], gpu_device)


def _w_sampled(w: np.ndarray, device, n_blocks: int, seed: int):
    """Full-size weight through the kernel; the oracle re-quantizes a sample
    of 128x128 blocks one by one."""
    q, qt, s = fb.fp8_quant_w_128x128(dev(w, device), transposed=True)
    torch.cuda.synchronize()
    qg, qtg, sg = host(q), host(qt), host(s)
    R, C = w.shape
    rng = np.random.default_rng(seed)
    picks = [(0, 0), (R // 128 - 1, C // 128 - 1)] + [tuple(rng.integers(0, [R // 128, C // 128])) for _ in range(n_blocks)]
    for br, bc in picks:
        blk = np.ascontiguousarray(w[128 * br:128 * br + 128, 128 * bc:128 * bc + 128])
        qo, so = oracle.quant_w(blk)
        assert sg[br, bc].view(np.uint32) == so[0, 0].view(np.uint32)
        assert np.array_equal(qg[128 * br:128 * br + 128, 128 * bc:128 * bc + 128], qo)
        assert np.array_equal(qtg[128 * bc:128 * bc + 128, 128 * br:128 * br + 128], qo.T)


def test_weight_full_fprop_sampled(gpu_device):
    _w_sampled(synth.fprop_linear(seed=1, M=128)["w"], gpu_device, 200, 7)


def test_weight_moe_experts_sampled(gpu_device):
    rng = np.random.default_rng(4)
    synth.moe_group_sizes(rng)           # same draw order as the grouped workload
    w_all = np.concatenate([synth.master_weight(rng, 2048, 7168) for _ in range(4)])   # 4 of the 64 experts
    _w_sampled(w_all, gpu_device, 100, 8)


def test_empty_inputs_are_noops(gpu_device):
    x = torch.empty((0, 256), dtype=torch.bfloat16, device=gpu_device)
    q, s = fb.fp8_quant_act_1x128(x)
    assert q.shape == (0, 256) and s.shape == (2, 0)
    w = torch.empty((0, 128), dtype=torch.float32, device=gpu_device)
    q, s = fb.fp8_quant_w_128x128(w)
    assert q.numel() == 0 and s.numel() == 0


def test_zero_and_tiny_groups(gpu_device):
    x = np.zeros((4, 512), np.float32)
    x[1, 128:256] = -0.0
    x[2, 256:384] = np.float32(2.0 ** -133) * np.arange(128)          # BF16 subnormals: subnormal scale
    x[3, 384:512] = np.float32(1e-38) * (1 - 2 * (np.arange(128) % 2))
    x[0, 5] = -3.0
    _act_parity(synth.f32_to_bf16_bits(x), 0, gpu_device)
    w = np.zeros((128, 384), np.float32)
    w[3, 130] = 1e-44          # amax/448 underflows to zero
    w[4, 131] = -2e-45
    w[5, 300] = 1e-40          # subnormal scale
    w[6, 301] = -7e-41
    _w_parity(w, gpu_device)


def test_dense_sweep_value_and_group_max(gpu_device):
    """Every positive finite BF16 value x (2^15 patterns, both signs) under a
    sample of group maxima: each group is [amax, 127 values <= amax]."""
    mags = (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(np.float32)  # positive finite BF16
    amaxes = mags[::97]
    rows = []
    for amax in amaxes:
        vals = mags[mags <= amax]
        vals = np.concatenate([vals, -vals])
        n = len(vals)
        ng = (n + 126) // 127
        pad = np.resize(vals, ng * 127).reshape(ng, 127)
        grp = np.concatenate([np.full((ng, 1), amax, np.float32), pad], axis=1)
        rows.append(grp)
    x = np.concatenate(rows)
    # rows of 4 groups of 128
    n = (len(x) // 4) * 4
    x = x[:n].reshape(-1, 512)
    _act_parity(synth.f32_to_bf16_bits(x), 0, gpu_device)


def test_weight_quotients_at_rounding_midpoints(gpu_device):
    """FP32 weights placed on, and a few ulps around, every E4M3 rounding
    midpoint times the block scale, for scales with arbitrary mantissas and
    for scales below 2^-90 (the kernel's full-division path).  Any one-ulp
    error in the quotient x / s would flip a code here."""
    grid = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (grid[1:] + grid[:-1]) / 2                       # rounding midpoints in [2^-10, 464)
    rng = np.random.default_rng(77)
    blocks = []
    amaxes = [np.float32(rng.uniform(1, 2) * 2.0 ** e) for e in (-30, -3, 0, 5, 40)]
    amaxes += [np.float32(1.3e-28), np.float32(3.0e-29)]     # scale below 2^-90
    for amax in amaxes:
        s = np.float32(amax / np.float32(448))              # the block scale the kernel derives
        vals = []
        for m in mids:
            x = np.float32(m * np.float64(s))
            for k in range(-3, 4):
                y = x
                step = np.float32(np.inf) if k > 0 else np.float32(-np.inf)
                for _ in range(abs(k)):
                    y = np.nextafter(y, step)
                if abs(y) <= amax:
                    vals += [y, -y]
        vals = np.array(vals, np.float32)
        blk = np.resize(vals, 128 * 128).reshape(128, 128)
        blk[0, 0] = amax
        blocks.append(blk)
    w = np.concatenate(blocks, axis=1)                      # [128, 128 * n_blocks]
    _w_parity(np.ascontiguousarray(w), gpu_device)


def _dual_parity(xb: np.ndarray, device):
    q_row, s_row, q_col_t, s_col = fb.fp8_quant_act_dual(dev_bf16(xb, device))
    torch.cuda.synchronize()
    qo, so = oracle.quant_act(xb, axis=0)
    qto, sto = oracle.quant_act(xb, axis=1)
    assert np.array_equal(host(s_row).view(np.uint32), so.view(np.uint32)), "row scales differ"
    assert np.array_equal(host(q_row), qo), "row codes differ"
    assert np.array_equal(host(s_col).view(np.uint32), sto.view(np.uint32)), "column scales differ"
    assert np.array_equal(host(q_col_t), qto), "column codes differ"


@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (384, 1280)])
def test_dual_small(gpu_device, shape):
    rng = np.random.default_rng(300 + shape[1])
    _dual_parity(synth.activations_channel_outliers(rng, *shape), gpu_device)


def test_dual_zero_and_tiny_groups(gpu_device):
    x = np.zeros((256, 256), np.float32)
    x[5, 3] = -2.0
    x[130:140, 200] = np.float32(2.0 ** -133)    # a column group and row groups with subnormal scales
    x[200, 128:256] = -0.0
    _dual_parity(synth.f32_to_bf16_bits(x), gpu_device)


def test_dual_zero_and_tiny_groups_large(gpu_device):
    """The same special groups in a tensor large enough (3584 tiles) for the
    staged-tile kernel, spread over several tiles."""
    x = np.zeros((8192, 7168), np.float32)
    x[5, 3] = -2.0
    x[130:140, 200] = np.float32(2.0 ** -133)
    x[200, 128:256] = -0.0
    x[4000:4128, 5000] = np.float32(448.0)
    x[8191, 7040:7168] = np.float32(-(2.0 ** -140))
    _dual_parity(synth.f32_to_bf16_bits(x), gpu_device)


def test_dual_full_wgrad_x(gpu_device):
    """X[8192,7168] of the Wgrad workload: the fused kernel against the
    oracle on both axes, and against the two single-axis kernels."""
    xb = synth.wgrad(seed=3)["x"]
    _dual_parity(xb, gpu_device)
    x = dev_bf16(xb, gpu_device)
    q_row, s_row, q_col_t, s_col = fb.fp8_quant_act_dual(x)
    q0, s0 = fb.fp8_quant_act_1x128(x, axis=fb.FP8FG_AXIS_COLS)
    q1, s1 = fb.fp8_quant_act_1x128(x, axis=fb.FP8FG_AXIS_ROWS)
    torch.cuda.synchronize()
    assert torch.equal(q_row, q0) and torch.equal(s_row.view(torch.int32), s0.view(torch.int32))
    assert torch.equal(q_col_t, q1) and torch.equal(s_col.view(torch.int32), s1.view(torch.int32))


@pytest.mark.parametrize("seed", range(8))
def test_random_shapes_all_quantizers(gpu_device, seed):
    """Random shapes for every quantizer, bit for bit against the oracle:
    1x128 with any row count, 128x1 with channel counts that are and are not
    multiples of 128, the fused kernel, and 128x128 with its transposed copy."""
    rng = np.random.default_rng(500 + seed)
    rows_any = int(rng.integers(1, 700))
    t128, c128 = int(rng.integers(1, 6)) * 128, int(rng.integers(1, 9)) * 128
    c8 = int(rng.integers(1, 100)) * 8
    _act_parity(synth.activations_random_outliers(rng, rows_any, c128), 0, gpu_device)
    _act_parity(synth.gradients_token_outliers(rng, t128, c8), 1, gpu_device)
    _act_parity(synth.gradients_token_outliers(rng, t128, c128), 1, gpu_device)
    _dual_parity(synth.activations_channel_outliers(rng, t128, c128), gpu_device)
    _w_parity(synth.master_weight(rng, t128, c128), gpu_device, transposed=bool(seed % 2))
