"""GPU parity of the block-scaled FP8 GEMM, through the C ABI.

Every case runs the whole path on the GPU (quantizers -> GEMM) and compares
with the oracle run on the same seeded inputs (oracle quantizers -> double
GEMM).  The quantized operands are also compared byte for byte, so the GEMM
sees exactly the oracle's inputs.  Pass: |gpu - o| <= 2^-16 * sum|a~ b~|,
plus one BF16 spacing of o for BF16 output.

Cases: the tiny Fprop in FP32 and BF16; medium shapes spanning several
tiles with a ragged N tile (N = 640 is 2.5 tiles of 256); token counts
that are not a multiple of 128 (Fprop and Dgrad); Dgrad through the
transposed weight copy and swapped scale strides; Wgrad with per-row B
scales; an exact integer case (bit-exact); K = 0; the full-size Fprop,
Dgrad and Wgrad workloads on sampled outputs; and the accumulation probe
(the tensor core's precision inside one 128-wide chunk).
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


def _fprop(x_bits, w, device, out_dtype):
    qx, sx = fb.fp8_quant_act_1x128(dev_bf16(x_bits, device))
    qw, sw = fb.fp8_quant_w_128x128(dev(w, device))
    y = fb.fp8_gemm_blockscaled(qx, sx, qw, sw, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return y, (qx, sx, qw, sw)


def _check_operands(gpu_ops, oracle_ops):
    for g, o in zip(gpu_ops, oracle_ops):
        g = host(g)
        assert np.array_equal(g.view(np.uint8) if g.dtype == np.uint8 else g.view(np.uint32),
                              o.view(np.uint8) if o.dtype == np.uint8 else o.view(np.uint32))


@pytest.mark.parametrize("out_dtype", [F32, BF16])
def test_tiny_fprop(gpu_device, out_dtype):
    d = synth.tiny_fprop(seed=0)
    y, ops = _fprop(d["x"], d["w"], gpu_device, out_dtype)
    qx, sx = oracle.quant_act(d["x"])
    qw, sw = oracle.quant_w(d["w"])
    _check_operands(ops, (qx, sx, qw, sw))
    o, m = oracle.gemm(qx, sx, qw, sw)
    assert_gemm_close(host(y), o, m, ODT[out_dtype], "tiny fprop")


@pytest.mark.parametrize("M,N,K", [(384, 640, 640), (128, 128, 128), (256, 1152, 384), (640, 256, 1280)])
def test_fprop_medium(gpu_device, M, N, K):
    d = synth.fprop_linear(seed=M + N + K, M=M, N=N, K=K)
    for out_dtype in (F32, BF16):
        y, ops = _fprop(d["x"], d["w"], gpu_device, out_dtype)
        qx, sx = oracle.quant_act(d["x"])
        qw, sw = oracle.quant_w(d["w"])
        _check_operands(ops, (qx, sx, qw, sw))
        o, m = oracle.gemm(qx, sx, qw, sw)
        assert_gemm_close(host(y), o, m, ODT[out_dtype], f"fprop {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(1, 256, 128), (200, 384, 256), (1000, 640, 384), (290, 128, 640)])
def test_fprop_ragged_m(gpu_device, M, N, K):
    """Token counts that are not a multiple of 128: the last 128-row tile
    is partial (single token, one row past a tile, several tiles plus a
    tail, and a warp-sized remainder); the rows past M must stay untouched."""
    d = synth.fprop_linear(seed=7 * M + N + K, M=M, N=N, K=K)
    qx, sx = oracle.quant_act(d["x"])
    qw, sw = oracle.quant_w(d["w"])
    o, m = oracle.gemm(qx, sx, qw, sw)
    for out_dtype in (F32, BF16):
        gx, gsx = fb.fp8_quant_act_1x128(dev_bf16(d["x"], gpu_device))
        gw, gsw = fb.fp8_quant_w_128x128(dev(d["w"], gpu_device))
        _check_operands((gx, gsx, gw, gsw), (qx, sx, qw, sw))
        # the output is a view of a taller buffer whose extra rows hold a sentinel
        dt = torch.float32 if out_dtype == F32 else torch.bfloat16
        big = torch.full((M + 160, N), 7.0, dtype=dt, device=gpu_device)
        y = fb.fp8_gemm_blockscaled(gx, gsx, gw, gsw, out_dtype=out_dtype, d=big[:M])
        torch.cuda.synchronize()
        assert_gemm_close(host(y), o, m, ODT[out_dtype], f"fprop ragged {M}x{N}x{K}")
        assert bool((big[M:] == 7.0).all()), "rows past M were written"


def test_dgrad_ragged_m(gpu_device):
    d = synth.dgrad(seed=9, M=333, N=640, K=384)           # dY[333,384], W[384,640], dX[333,640]
    qdy, sdy = fb.fp8_quant_act_1x128(dev_bf16(d["dy"], gpu_device))
    qw, qwt, sw = fb.fp8_quant_w_128x128(dev(d["w"], gpu_device), transposed=True)
    nw = d["w"].shape[1] // 128
    dx = fb.fp8_gemm_blockscaled(qdy, sdy, qwt, sw, sb_strides=(1, nw), out_dtype=BF16)
    torch.cuda.synchronize()
    qdy_o, sdy_o = oracle.quant_act(d["dy"])
    qw_o, sw_o, qwt_o = oracle.quant_w(d["w"], transposed=True)
    o, m = oracle.gemm(qdy_o, sdy_o, qwt_o, sw_o, sb_strides=(1, nw))
    assert_gemm_close(host(dx), o, m, "bf16", "dgrad ragged")


def test_dgrad_medium(gpu_device):
    d = synth.dgrad(seed=5, M=512, N=640, K=384)           # dY[512,384], W[384,640], dX[512,640]
    qdy, sdy = fb.fp8_quant_act_1x128(dev_bf16(d["dy"], gpu_device))
    qw, qwt, sw = fb.fp8_quant_w_128x128(dev(d["w"], gpu_device), transposed=True)
    nw = d["w"].shape[1] // 128                             # block columns of W
    dx = fb.fp8_gemm_blockscaled(qdy, sdy, qwt, sw, sb_strides=(1, nw), out_dtype=BF16)
    torch.cuda.synchronize()
    qdy_o, sdy_o = oracle.quant_act(d["dy"])
    qw_o, sw_o, qwt_o = oracle.quant_w(d["w"], transposed=True)
    assert np.array_equal(host(qwt), qwt_o)
    o, m = oracle.gemm(qdy_o, sdy_o, qwt_o, sw_o, sb_strides=(1, nw))
    assert_gemm_close(host(dx), o, m, "bf16", "dgrad")


def test_wgrad_medium(gpu_device):
    d = synth.wgrad(seed=6, T=640, N_out=384, K_in=640)     # dW[384,640] = dY^T X over 640 tokens
    qdyt, sdy = fb.fp8_quant_act_1x128(dev_bf16(d["dy"], gpu_device), axis=fb.FP8FG_AXIS_ROWS)
    qxt, sx = fb.fp8_quant_act_1x128(dev_bf16(d["x"], gpu_device), axis=fb.FP8FG_AXIS_ROWS)
    dw = fb.fp8_gemm_blockscaled(qdyt, sdy, qxt, sx, bscale=fb.FP8FG_BSCALE_ROW, out_dtype=F32)
    torch.cuda.synchronize()
    qa, sa = oracle.quant_act(d["dy"], axis=1)
    qb, sb = oracle.quant_act(d["x"], axis=1)
    _check_operands((qdyt, sdy, qxt, sx), (qa, sa, qb, sb))
    o, m = oracle.gemm(qa, sa, qb, sb, bscale=oracle.BSCALE_ROW)
    assert_gemm_close(host(dw), o, m, "f32", "wgrad")


def test_integer_case_is_exact(gpu_device):
    rng = np.random.default_rng(9)
    M, N, K = 256, 512, 512
    ia = rng.integers(-16, 17, size=(M, K))
    ib = rng.integers(-16, 17, size=(N, K))
    qa = oracle.e4m3_encode(ia.astype(np.float32))
    qb = oracle.e4m3_encode(ib.astype(np.float32))
    sa = np.ones((K // 128, M), np.float32)
    sb = np.ones((N // 128, K // 128), np.float32)
    y = fb.fp8_gemm_blockscaled(dev(qa, gpu_device), dev(sa, gpu_device), dev(qb, gpu_device),
                                dev(sb, gpu_device), out_dtype=F32)
    torch.cuda.synchronize()
    want = (ia.astype(np.int64) @ ib.astype(np.int64).T).astype(np.float64)   # |sum| < 2^24: exact in FP32
    assert np.array_equal(host(y).astype(np.float64), want)


def test_k_zero_writes_zeros(gpu_device):
    a = torch.empty((128, 0), dtype=torch.uint8, device=gpu_device)
    b = torch.empty((256, 0), dtype=torch.uint8, device=gpu_device)
    s = torch.empty((0, 128), dtype=torch.float32, device=gpu_device)
    d = torch.full((128, 256), 7.0, dtype=torch.float32, device=gpu_device)
    fb.fp8_gemm_blockscaled(a, s, b, torch.empty((2, 0), dtype=torch.float32, device=gpu_device),
                            out_dtype=F32, d=d)
    torch.cuda.synchronize()
    assert torch.count_nonzero(d).item() == 0


def test_accumulation_within_a_chunk(gpu_device, record_property):
    """Accumulation precision of one 128-wide chunk on the tensor cores: one
    large product (448 * 448) plus 127 small ones (1 * 2^-j), the large term
    first (row 0) or last (row 1).  With full FP32 accumulation every small
    term survives while 2^-j is above about 2^-23 of the large one; an
    accumulator that keeps ~14 bits (what the pages measure on H800) would
    drop them and break the 2^-16 tolerance at j = 0.  The measured errors are
    recorded in the test report."""
    K = M = N = 128
    codes = {0: 0x38, 3: 0x20, 6: 0x08, 9: 0x01}          # 1, 2^-3, 2^-6, 2^-9
    qa = np.zeros((M, K), np.uint8)
    qb = np.zeros((N, K), np.uint8)
    qa[0, 0] = 0x7E
    qa[0, 1:] = 0x38
    qa[1, :127] = 0x38
    qa[1, 127] = 0x7E
    for v, (j, c) in enumerate(codes.items()):
        qb[v, 0] = 0x7E
        qb[v, 1:] = c
        qb[4 + v, :127] = c
        qb[4 + v, 127] = 0x7E
    sa = np.ones((1, M), np.float32)
    sb = np.ones((1, 1), np.float32)
    y = fb.fp8_gemm_blockscaled(dev(qa, gpu_device), dev(sa, gpu_device), dev(qb, gpu_device),
                                dev(sb, gpu_device), out_dtype=F32)
    torch.cuda.synchronize()
    y = host(y).astype(np.float64)
    report = {}
    for v, j in enumerate(codes):
        exact = 448.0 * 448.0 + 127 * 2.0 ** -j
        for row, col, where in ((0, v, "first"), (1, 4 + v, "last")):
            err = y[row, col] - exact
            report[f"j={j},large {where}"] = err
            assert abs(err) <= 2.0 ** -16 * exact, (j, where, err)
    record_property("chunk_accumulation_errors", repr(report))
    print("chunk accumulation errors:", report)


# ------------------------------------------------------- full-size cases ---
# The GPU runs the whole workload; the oracle quantizes only the 128-row
# blocks that hold the sampled outputs (quantizer groups are independent) and
# computes those outputs one by one.

def _sample_blocks(rng, n_blocks, k):
    picks = {0, n_blocks - 1} | set(int(v) for v in rng.choice(n_blocks, size=min(k, n_blocks), replace=False))
    return np.array(sorted(picks))


def _rows_of(blocks):
    return (blocks[:, None] * 128 + np.arange(128)[None, :]).reshape(-1)


def _entries(rng, n_i, n_j, per_pair=8, bi=128, bj=128):
    """per_pair random entries in every (row block, column block) pair of the
    sampled sub-matrix [n_i, n_j]."""
    ii, jj = [], []
    for a in range(n_i // bi):
        for b in range(n_j // bj):
            ii.append(a * bi + rng.integers(0, bi, per_pair))
            jj.append(b * bj + rng.integers(0, bj, per_pair))
    return np.concatenate(ii), np.concatenate(jj)


def test_fprop_full_sampled(gpu_device):
    d = synth.fprop_linear(seed=1)                          # X[4096,7168], W[18432,7168], Y bf16
    y, _ = _fprop(d["x"], d["w"], gpu_device, BF16)
    yh = host(y)
    rng = np.random.default_rng(11)
    ri = _rows_of(_sample_blocks(rng, 4096 // 128, 5))
    rj = _rows_of(_sample_blocks(rng, 18432 // 128, 6))
    qx, sx = oracle.quant_act(d["x"][ri])
    qw, sw = oracle.quant_w(d["w"][rj])
    ii, jj = _entries(rng, len(ri), len(rj))
    o, m = oracle.gemm_entries(qx, sx, qw, sw, ii, jj)
    assert_gemm_close(yh[ri[ii], rj[jj]], o, m, "bf16", "fprop full")


def test_dgrad_full_sampled(gpu_device):
    d = synth.dgrad(seed=2)                                 # dY[8192,2048], W[2048,7168], dX[8192,7168]
    qdy, sdy = fb.fp8_quant_act_1x128(dev_bf16(d["dy"], gpu_device))
    qw, qwt, sw = fb.fp8_quant_w_128x128(dev(d["w"], gpu_device), transposed=True)
    dx = fb.fp8_gemm_blockscaled(qdy, sdy, qwt, sw, sb_strides=(1, 7168 // 128), out_dtype=BF16)
    torch.cuda.synchronize()
    dxh = host(dx)
    rng = np.random.default_rng(12)
    ri = _rows_of(_sample_blocks(rng, 8192 // 128, 5))
    qa, sa = oracle.quant_act(d["dy"][ri])
    _, sw_o, qwt_o = oracle.quant_w(d["w"], transposed=True)
    ii, jj = _entries(rng, len(ri), 7168, per_pair=4)
    o, m = oracle.gemm_entries(qa, sa, qwt_o, sw_o, ii, jj, sb_strides=(1, 7168 // 128))
    assert_gemm_close(dxh[ri[ii], jj], o, m, "bf16", "dgrad full")


def test_wgrad_full_sampled(gpu_device):
    d = synth.wgrad(seed=3)                                 # dY[8192,2048], X[8192,7168], dW[2048,7168]
    qa_g, sa_g = fb.fp8_quant_act_1x128(dev_bf16(d["dy"], gpu_device), axis=fb.FP8FG_AXIS_ROWS)
    qb_g, sb_g = fb.fp8_quant_act_1x128(dev_bf16(d["x"], gpu_device), axis=fb.FP8FG_AXIS_ROWS)
    dw = fb.fp8_gemm_blockscaled(qa_g, sa_g, qb_g, sb_g, bscale=fb.FP8FG_BSCALE_ROW, out_dtype=F32)
    torch.cuda.synchronize()
    dwh = host(dw)
    rng = np.random.default_rng(13)
    ci = _rows_of(_sample_blocks(rng, 2048 // 128, 4))      # output rows = channels of dY
    cj = _rows_of(_sample_blocks(rng, 7168 // 128, 5))      # output columns = channels of X
    qa, sa = oracle.quant_act(np.ascontiguousarray(d["dy"][:, ci]), axis=1)
    qb, sb = oracle.quant_act(np.ascontiguousarray(d["x"][:, cj]), axis=1)
    ii, jj = _entries(rng, len(ci), len(cj))
    o, m = oracle.gemm_entries(qa, sa, qb, sb, ii, jj, bscale=oracle.BSCALE_ROW)
    assert_gemm_close(dwh[ci[ii], cj[jj]], o, m, "f32", "wgrad full")


def test_calls_on_a_side_stream(gpu_device):
    """Every entry point honours its stream argument: the Fprop chain issued
    on a non-default stream gives the default stream's results bit for bit."""
    d = synth.fprop_linear(seed=1, M=256, N=512, K=1024)
    x, w = dev_bf16(d["x"], gpu_device), dev(d["w"], gpu_device)
    qx0, sx0 = fb.fp8_quant_act_1x128(x)
    qw0, sw0 = fb.fp8_quant_w_128x128(w, transposed=False)
    y0 = fb.fp8_gemm_blockscaled(qx0, sx0, qw0, sw0, out_dtype=F32)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        qx1, sx1 = fb.fp8_quant_act_1x128(x, stream=side)
        qw1, sw1 = fb.fp8_quant_w_128x128(w, transposed=False, stream=side)
        y1 = fb.fp8_gemm_blockscaled(qx1, sx1, qw1, sw1, out_dtype=F32, stream=side)
    side.synchronize()
    assert torch.equal(qx0, qx1) and torch.equal(qw0, qw1)
    assert torch.equal(y0, y1)


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes_against_the_oracle(gpu_device, seed):
    """Random shapes (multiples of 128, ragged against the 128x256 tile),
    block or per-row B scales, BF16 or FP32 output: the whole output against
    the oracle, on operands quantized by the GPU and checked byte for byte."""
    rng = np.random.default_rng(1000 + seed)
    M, N, K = (int(rng.integers(1, 5)) * 128, int(rng.integers(1, 7)) * 128, int(rng.integers(1, 9)) * 128)
    row_b = bool(seed % 3 == 2)
    dgrad_like = bool(seed % 3 == 1)
    out_dtype = F32 if seed % 2 else BF16
    if dgrad_like:
        # Dgrad-like: B is the transposed copy of a weight W[K, N], its block
        # scales read through swapped strides
        a_src = synth.gradients_token_outliers(rng, M, K)
        w_src = synth.master_weight(rng, K, N)
        qa, sa = fb.fp8_quant_act_1x128(dev_bf16(a_src, gpu_device))
        _, qb, sb = fb.fp8_quant_w_128x128(dev(w_src, gpu_device), transposed=True)
        d = fb.fp8_gemm_blockscaled(qa, sa, qb, sb, sb_strides=(1, N // 128), out_dtype=out_dtype)
        qa_o, sa_o = oracle.quant_act(a_src)
        _, sb_o, qb_o = oracle.quant_w(w_src, transposed=True)
        torch.cuda.synchronize()
        assert np.array_equal(host(qa), qa_o) and np.array_equal(host(qb), qb_o)
        assert np.array_equal(host(sb).view(np.uint32), sb_o.view(np.uint32))
        o, m = oracle.gemm(qa_o, sa_o, qb_o, sb_o, sb_strides=(1, N // 128))
        assert_gemm_close(host(d), o, m, ODT[out_dtype], f"random dgrad-like {M}x{N}x{K}")
        return
    if row_b:
        # Wgrad-like: both operands from token-axis groups (K = tokens)
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
    assert_gemm_close(host(d), o, m, ODT[out_dtype], f"random {M}x{N}x{K} row_b={row_b}")
