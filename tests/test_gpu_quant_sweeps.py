"""Exhaustive quantizer sweeps on the GPU against the oracle, bit for bit.

The per-group scale s = fl32(amax / 448) and the element code
enc(fl32(x / s)) depend only on the pair (x, amax) ("Unified E4M3 format in
DeepSeek-V3", Dynamic Scaling and Online Quantization: each group's scale
comes from its own maximum).  Two sweeps cover that dependence:

* BF16 activations: every positive finite BF16 value as a group maximum,
  each with every BF16 value of smaller or equal magnitude, both signs, as
  the other members of its groups (about 1.07e9 elements, in chunks);
* FP32 weights: every one of the 2^23 FP32 mantissas as an element of a
  128x128 block, at quotient binades across the E4M3 range (the top
  binade, where the block maximum's own quotient may round above 448 and
  saturate; normal; subnormal; the tie to zero), under block scales with random
  mantissas, all-ones mantissas and scales on both sides of 2^-90 (below
  which the kernel switches from the corrected reciprocal to a full
  division);
* the conversion alone: every finite FP32 value of magnitude at most 448,
  both signs, encoded under a block scale of exactly 1.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_act_gb300 import binding as fb
from gpu_util import dev, dev_bf16, host

pytestmark = pytest.mark.gpu

CHUNK = 1 << 25          # elements per GPU/oracle round


def _act_rows_parity(groups: list, device):
    """Groups of 128 BF16 patterns -> rows of 512 (4 groups, zero groups as
    padding) -> the 1x128 quantizer on the GPU and in the oracle."""
    g = np.concatenate(groups)
    pad = (-len(g)) % 4
    if pad:
        g = np.concatenate([g, np.zeros((pad, 128), np.uint16)])
    xb = np.ascontiguousarray(g.reshape(-1, 512))
    q, s = fb.fp8_quant_act_1x128(dev_bf16(xb, device))
    torch.cuda.synchronize()
    qo, so = oracle.quant_act(xb)
    qg, sg = host(q), host(s)
    bad = np.argwhere(qg != qo)
    assert len(bad) == 0, f"{len(bad)} codes differ, first at {bad[0]}: x=0x{xb[tuple(bad[0])]:04x} " \
                          f"gpu=0x{qg[tuple(bad[0])]:02x} oracle=0x{qo[tuple(bad[0])]:02x}"
    assert np.array_equal(sg.view(np.uint32), so.view(np.uint32))
    return len(g) * 128


def test_every_bf16_group_maximum_with_every_smaller_value(gpu_device):
    total = 0
    groups, n = [], 0
    for a in range(1, 0x7F80):                            # positive finite BF16 patterns, in numeric order
        vals = np.arange(1, a + 1, dtype=np.uint16)
        vals = np.concatenate([vals, vals | np.uint16(0x8000)])
        ng = (len(vals) + 126) // 127
        body = np.resize(vals, ng * 127).reshape(ng, 127)
        grp = np.concatenate([np.full((ng, 1), a, np.uint16), body], axis=1)
        grp[::2, 0] |= np.uint16(0x8000)                  # the maximum itself with either sign
        groups.append(grp)
        n += grp.size
        if n >= CHUNK:
            total += _act_rows_parity(groups, gpu_device)
            groups, n = [], 0
    if groups:
        total += _act_rows_parity(groups, gpu_device)
    assert total > 1_000_000_000


def _weight_parity(w: np.ndarray, device):
    q, s = fb.fp8_quant_w_128x128(dev(w, device))
    torch.cuda.synchronize()
    qo, so = oracle.quant_w(w)
    qg, sg = host(q), host(s)
    bad = np.argwhere(qg != qo)
    assert len(bad) == 0, f"{len(bad)} codes differ, first at {bad[0]}: w={w[tuple(bad[0])]!r} " \
                          f"gpu=0x{qg[tuple(bad[0])]:02x} oracle=0x{qo[tuple(bad[0])]:02x}"
    assert np.array_equal(sg.view(np.uint32), so.view(np.uint32))


def _f32(bits) -> np.float32:
    return np.array([bits], np.uint32).view(np.float32)[0]


@pytest.mark.parametrize("amax_bits", [
    0x3FDA3C91,        # 1.705: a random mantissa, s ~ 2^-8.0
    0x3FFFFFFF,        # 2 - 2^-23: all-ones mantissa, s ~ 2^-7.8
    0x42FFFFFF,        # 128 - 2^-17: all-ones mantissa, s ~ 2^-1.8
    0x1E2B17E3,        # 9.06e-21: a random mantissa, s ~ 2^-75.4
    0x16E00000,        # 448 * 2^-90: s = 2^-90 exactly (corrected reciprocal, at its bound)
    0x16DFFFFF,        # the FP32 value below: s just below 2^-90 (full division)
    0x15FFFFFF,        # all-ones mantissa, s ~ 2^-91.8 (full division)
    0x604321AB,        # 5.6e19: a random mantissa, s ~ 2^56.8
])
def test_weight_path_every_fp32_mantissa(gpu_device, amax_bits):
    amax = _f32(amax_bits)
    s = np.float32(amax / np.float32(448.0))
    e_s = int(np.floor(np.log2(np.float64(s))))
    m = np.arange(1 << 23, dtype=np.uint32)
    cols = []
    for k in (9, 8, 3, -2, -6, -8, -10):           # quotient binades: the top of the E4M3 range .. the tie to zero
        e = e_s + k
        if e < -126 or e > 127:
            continue
        x = ((np.uint32(e + 127) << np.uint32(23)) | m).view(np.float32)
        x = np.where(m & 1, -x, x).astype(np.float32)   # both signs
        x = x[np.abs(x) <= amax]                      # keep the block maximum at amax
        cols.append(x)
    vals = np.concatenate(cols)
    per_block = 128 * 128 - 1
    nb = (len(vals) + per_block - 1) // per_block
    body = np.zeros(nb * per_block, np.float32)
    body[:len(vals)] = vals
    blocks = np.concatenate([np.full((nb, 1), amax, np.float32), body.reshape(nb, per_block)], axis=1)
    w = np.ascontiguousarray(blocks.reshape(nb, 128, 128).transpose(1, 0, 2).reshape(128, nb * 128))
    for c0 in range(0, nb, 1024):                  # at most 1024 blocks (16.8M elements) per round
        _weight_parity(np.ascontiguousarray(w[:, c0 * 128:(c0 + 1024) * 128]), gpu_device)


def test_encoder_every_fp32_value_up_to_448(gpu_device):
    """The GPU's FP32 -> E4M3 conversion on every finite FP32 pattern of
    magnitude at most 448, both signs (2.28e9 values), against the oracle's
    encoder.  Each 128x128 block of the weight quantizer's input holds 448
    in its first element and test values elsewhere, so its scale is
    fl32(448 / 448) = 1 and every code is the encoding of fl32(x / 1) = x
    itself: the conversion is checked alone, with no scale in between."""
    top = np.uint32(0x43E00000)                  # 448.0f
    per_block = 128 * 128 - 1
    step = per_block * 2048                      # values per round (~2^25)
    total = 0
    for start in range(0, int(top) + 1, step):
        bits = np.arange(start, min(start + step, int(top) + 1), dtype=np.uint32)
        ref = oracle.e4m3_encode(bits.view(np.float32))
        nb = -(-len(bits) // per_block)
        for sign in (np.uint32(0), np.uint32(0x80000000)):
            vals = np.zeros(nb * per_block, np.uint32)
            vals[:len(bits)] = bits | sign
            w = np.empty((nb, per_block + 1), np.float32)
            w[:, 0] = 448.0
            w[:, 1:] = vals.reshape(nb, per_block).view(np.float32)
            q, s = fb.fp8_quant_w_128x128(dev(w.reshape(nb * 128, 128), gpu_device))
            torch.cuda.synchronize()
            assert np.all(host(s) == 1.0)
            qg = host(q).reshape(nb, per_block + 1)[:, 1:].reshape(-1)[:len(bits)]
            want = ref | np.uint8(0x80) if sign else ref
            bad = np.flatnonzero(qg != want)
            assert len(bad) == 0, f"{len(bad)} codes differ, first x=0x{int(bits[bad[0]] | sign):08x} " \
                                  f"gpu=0x{qg[bad[0]]:02x} oracle=0x{want[bad[0]]:02x}"
            total += len(bits)
    assert total == 2 * (int(top) + 1)
