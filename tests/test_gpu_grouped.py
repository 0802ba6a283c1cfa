"""GPU parity of the grouped MoE-expert GEMM through the C ABI: rows
[off[g], off[g+1]) of the token matrix multiply expert weight g.  Small
shapes are compared in full (including an empty expert and zero pad rows,
which must come out exactly zero); the full workload (64 experts, 32768
tokens, Dirichlet(1) counts padded to 128, N = 2048, K = 7168) on sampled
outputs; offsets that break the layout rules are reported through the device
status word with nothing written."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_act_gb300 import binding as fb
from fp8_fine_grained_act_gb300 import synth
from gpu_util import assert_gemm_close, dev, dev_bf16, host

pytestmark = pytest.mark.gpu


def _quant_experts_gpu(w_g, device):
    G, N, K = w_g.shape
    qb = torch.empty((G, N, K), dtype=torch.uint8, device=device)
    sb = torch.empty((G, N // 128, K // 128), dtype=torch.float32, device=device)
    for g in range(G):   # one call per expert, or one call on [G*N, K]: the blocks are the same
        fb.fp8_quant_w_128x128(dev(w_g[g], device), q=qb[g], scales=sb[g])
    return qb, sb


@pytest.mark.parametrize("out_dtype,counts", [
    (fb.FP8FG_OUT_BF16, [100, 0, 300, 128, 5]),
    (fb.FP8FG_OUT_F32, [100, 0, 300, 128, 5]),
    (fb.FP8FG_OUT_BF16, [0, 0, 256, 1, 0]),          # empty experts first and last
])
def test_grouped_small(gpu_device, out_dtype, counts):
    rng = np.random.default_rng(21)
    counts = np.array(counts)
    padded = ((counts + 127) // 128) * 128
    offsets = np.zeros(len(counts) + 1, np.int32)
    offsets[1:] = np.cumsum(padded)
    N, K = 384, 512
    x = synth.moe_tokens(rng, counts, padded, K)
    w = np.stack([synth.master_weight(rng, N, K) for _ in counts])
    qa, sa = fb.fp8_quant_act_1x128(dev_bf16(x, gpu_device))
    qb, sb = _quant_experts_gpu(w, gpu_device)
    y = fb.fp8_gemm_grouped(qa, sa, qb, sb, dev(offsets, gpu_device), out_dtype=out_dtype)
    torch.cuda.synchronize()
    qa_o, sa_o = oracle.quant_act(x)
    qs = [oracle.quant_w(w[g]) for g in range(len(counts))]
    qb_o = np.stack([q for q, _ in qs])
    sb_o = np.stack([s for _, s in qs])
    o, m = oracle.gemm_grouped(qa_o, sa_o, qb_o, sb_o, offsets)
    yh = host(y)
    assert_gemm_close(yh, o, m, "bf16" if out_dtype == fb.FP8FG_OUT_BF16 else "f32", "grouped small")
    # pad rows are zero inputs -> exactly zero outputs
    r = 0
    for c, p in zip(counts, padded):
        assert np.all(yh[r + c:r + p] == 0)
        r += p


def test_grouped_full_sampled(gpu_device):
    d = synth.grouped_moe(seed=4)
    off = d["offsets"]
    G, N, K = d["w"].shape
    qa, sa = fb.fp8_quant_act_1x128(dev_bf16(d["x"], gpu_device))
    qb, sb = _quant_experts_gpu(d["w"], gpu_device)
    y = fb.fp8_gemm_grouped(qa, sa, qb, sb, dev(off, gpu_device))
    torch.cuda.synchronize()
    yh = host(y)
    rng = np.random.default_rng(22)
    nonempty = [g for g in range(G) if off[g + 1] > off[g]]
    experts = sorted(set([nonempty[0], nonempty[-1]]) | set(rng.choice(nonempty, 6, replace=False).tolist()))
    for g in experts:
        r0, r1 = int(off[g]), int(off[g + 1])
        rows = np.arange(r0, r1)
        xb = d["x"][rows]
        qa_o, sa_o = oracle.quant_act(xb)
        qb_o, sb_o = oracle.quant_w(d["w"][g])
        ii = np.concatenate([rng.integers(0, r1 - r0, 64), [0, r1 - r0 - 1]])
        jj = np.concatenate([rng.integers(0, N, 64), [0, N - 1]])
        o, m = oracle.gemm_entries(qa_o, sa_o, qb_o, sb_o, ii, jj)
        assert_gemm_close(yh[rows[ii], jj], o, m, "bf16", f"grouped full, expert {g}")
    # zero pad rows
    for g in range(G):
        pad0 = int(off[g] + d["counts"][g])
        assert np.all(yh[pad0:int(off[g + 1])] == 0)


def test_grouped_bad_offsets_reported(gpu_device):
    assert fb.fp8fg_last_device_status() in (0,)            # clean start
    N, K = 256, 128
    qa = torch.zeros((256, K), dtype=torch.uint8, device=gpu_device)
    sa = torch.ones((1, 256), dtype=torch.float32, device=gpu_device)
    qb = torch.zeros((2, N, K), dtype=torch.uint8, device=gpu_device)
    sb = torch.ones((2, N // 128, 1), dtype=torch.float32, device=gpu_device)
    for bad in ([0, 100, 256], [0, 256, 128], [0, 128, 384], [128, 128, 256]):
        y = torch.full((256, N), 3.0, dtype=torch.float32, device=gpu_device)
        fb.fp8_gemm_grouped(qa, sa, qb, sb, torch.tensor(bad, dtype=torch.int32, device=gpu_device),
                            out_dtype=fb.FP8FG_OUT_F32, d=y)
        assert fb.fp8fg_last_device_status() == fb.FP8FG_ERR_INVALID_ARG
        assert torch.all(y == 3.0).item()
    # a good call afterwards works and reports nothing
    y = fb.fp8_gemm_grouped(qa, sa, qb, sb, torch.tensor([0, 128, 256], dtype=torch.int32, device=gpu_device),
                            out_dtype=fb.FP8FG_OUT_F32)
    assert fb.fp8fg_last_device_status() == 0
    assert torch.count_nonzero(y).item() == 0


@pytest.mark.parametrize("seed", range(6))
def test_grouped_random(gpu_device, seed):
    """Random expert counts (empty experts included), random N and K: the
    whole output against the oracle, pad rows exactly zero."""
    rng = np.random.default_rng(700 + seed)
    G = int(rng.integers(1, 13))
    counts = rng.integers(0, 400, G) * (rng.random(G) > 0.2)
    padded = ((counts + 127) // 128) * 128
    if padded.sum() == 0:
        counts[0], padded[0] = 1, 128
    offsets = np.zeros(G + 1, np.int32)
    offsets[1:] = np.cumsum(padded)
    N, K = int(rng.integers(1, 5)) * 128, int(rng.integers(1, 7)) * 128
    x = synth.moe_tokens(rng, counts, padded, K)
    w = np.stack([synth.master_weight(rng, N, K) for _ in range(G)])
    qa, sa = fb.fp8_quant_act_1x128(dev_bf16(x, gpu_device))
    qb, sb = _quant_experts_gpu(w, gpu_device)
    y = fb.fp8_gemm_grouped(qa, sa, qb, sb, dev(offsets, gpu_device), out_dtype=fb.FP8FG_OUT_F32)
    torch.cuda.synchronize()
    qa_o, sa_o = oracle.quant_act(x)
    qs = [oracle.quant_w(w[g]) for g in range(G)]
    o, m = oracle.gemm_grouped(qa_o, sa_o, np.stack([q for q, _ in qs]), np.stack([s for _, s in qs]), offsets)
    yh = host(y)
    assert_gemm_close(yh, o, m, "f32", f"grouped random G={G} N={N} K={K}")
    r = 0
    for c, p in zip(counts, padded):
        assert np.all(yh[r + c:r + p] == 0)
        r += p
