"""Pins for the oracle's group quantizers (CPU only).

What fixes each expected value:
  * construction: a group built from known E4M3 codes times a power-of-two
    scale, with the code 0x7E (448) present, must come back as exactly those
    codes and exactly that scale (s = 448 * 2^k / 448 = 2^k is exact and
    every x / s is exact).  Each group gets its own exponent k and its own
    position of the maximum, so a wrong group geometry, axis, transpose or
    scale index changes some byte or some scale;
  * the quantize/dequantize error bound: |x - dec(q) s| is at most half an
    E4M3 spacing of fl(x/s), times s, plus the FP32 rounding of the quotient
    (|x/s - fl(x/s)| s);
  * invariants: the element with |x| = amax encodes to +-448 (the group's
    maximum is scaled to the FP8 maximum), signs are kept, scaling a group by
    a power of two keeps the codes and scales s by the same power;
  * special case: an all-zero group has s = 0 and signed-zero codes;
  * the 128x1 mode on X equals the 1x128 mode on X^T (the two layouts
    describe the same groups);
  * an independent implementation (numpy float32 division + ml_dtypes
    float8_e4m3fn encoding) where ml_dtypes is installed.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from fp8_fine_grained_act_gb300 import synth

G = 128


def _bits_of(f32: np.ndarray) -> np.ndarray:
    """BF16 bits of FP32 values that are exactly representable in BF16."""
    u = np.ascontiguousarray(f32, np.float32).view(np.uint32)
    assert np.all((u & 0xFFFF) == 0)
    return (u >> 16).astype(np.uint16)


def _random_codes(rng, shape):
    """Random finite E4M3 codes, at most 0x7D in magnitude (0x7E is placed
    separately), both signs."""
    mag = rng.integers(0, 0x7E, size=shape).astype(np.uint8)
    sign = (rng.integers(0, 2, size=shape).astype(np.uint8) << 7)
    return mag | sign


def _constructed_rows(rng, rows, cols):
    """x[i, 128c + t] = dec(code) * 2^k[i, c], with code 0x7E (or 0xFE) at a
    per-group position.  Returns (x_f32, codes, scales[c, i])."""
    ng = cols // G
    codes = _random_codes(rng, (rows, cols))
    k = rng.integers(-20, 10, size=(rows, ng))
    pos = rng.integers(0, G, size=(rows, ng))
    for i in range(rows):
        for c in range(ng):
            codes[i, c * G + pos[i, c]] = 0x7E | (rng.integers(0, 2) << 7)
    vals = oracle.e4m3_decode(codes)
    scale = np.exp2(k.astype(np.float64))
    x = vals * np.repeat(scale, G, axis=1)
    return x.astype(np.float32), codes, scale.T.astype(np.float32)


def test_constructed_groups_axis0():
    rng = np.random.default_rng(11)
    x, codes, s_want = _constructed_rows(rng, 37, 4 * G)   # ragged row count
    q, s = oracle.quant_act(_bits_of(x), axis=0)
    assert np.array_equal(s, s_want)
    assert np.array_equal(q, codes)


def test_constructed_groups_axis1():
    rng = np.random.default_rng(12)
    xt, codes, s_want = _constructed_rows(rng, 45, 3 * G)   # groups along rows of x = xt^T
    x = np.ascontiguousarray(xt.T)                          # [3G, 45]
    q, s = oracle.quant_act(_bits_of(x), axis=1)
    assert q.shape == (45, 3 * G) and s.shape == (3, 45)
    assert np.array_equal(s, s_want)
    assert np.array_equal(q, codes)


def test_constructed_blocks_weight():
    rng = np.random.default_rng(13)
    R, C = 3 * G, 2 * G
    codes = _random_codes(rng, (R, C))
    k = rng.integers(-30, 5, size=(R // G, C // G))
    for r in range(R // G):
        for c in range(C // G):
            i, j = rng.integers(0, G, size=2)
            codes[r * G + i, c * G + j] = 0xFE
    scale = np.exp2(k.astype(np.float64))
    w = (oracle.e4m3_decode(codes) * np.kron(scale, np.ones((G, G)))).astype(np.float32)
    q, s, qt = oracle.quant_w(w, transposed=True)
    assert np.array_equal(s, scale.astype(np.float32))
    assert np.array_equal(q, codes)
    assert np.array_equal(qt, codes.T)


def _half_spacing(v):
    """Half the E4M3 grid spacing at |v| (spacing 2^-9 below 2^-6, else
    2^(floor(log2|v|) - 3)); 448's spacing is taken as the one below it."""
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return np.where(a < 2.0 ** -6, 2.0 ** -10, np.exp2(e - 4))


@pytest.mark.parametrize("axis", [0, 1])
def test_error_bound_and_invariants_act(axis):
    rng = np.random.default_rng(21 + axis)
    xb = synth.activations_random_outliers(rng, 256, 384, frac=5e-3, factor=300.0)
    x = synth.bf16_bits_to_f32(xb).astype(np.float64)
    q, s = oracle.quant_act(xb, axis=axis)
    if axis == 1:   # view everything as row groups of x^T
        x = x.T
    xs = x.reshape(x.shape[0], -1, G)                           # [rows, ng, 128]
    sc = s.T[:, :, None].astype(np.float64)    # both layouts: [groups along the last dim]
    qq = q.reshape(x.shape[0], -1, G)
    deq = oracle.e4m3_decode(qq) * sc
    quot = (xs.astype(np.float32) / sc.astype(np.float32)).astype(np.float64)   # fl32(x/s)
    bound = _half_spacing(quot) * sc + np.abs(xs / sc - quot) * sc
    assert np.all(np.abs(xs - deq) <= bound * (1 + 1e-12))   # slack: this check's own double rounding
    # the maximum lands on +-448, the sign is kept, s = fl32(amax / 448)
    amax = np.abs(xs).max(axis=2)
    assert np.array_equal(sc[:, :, 0], (amax.astype(np.float32) / np.float32(448)).astype(np.float64))
    at_max = np.abs(xs) == amax[:, :, None]
    assert np.all((qq[at_max] & 0x7F) == 0x7E)
    nz = xs != 0
    assert np.array_equal(np.signbit(xs[nz]), (qq[nz] & 0x80) != 0)


def test_power_of_two_invariance_and_zero_group():
    rng = np.random.default_rng(31)
    x = synth.bf16_bits_to_f32(synth.activations_channel_outliers(rng, 64, 3 * G))
    x[5, G:2 * G] = 0.0
    x[9, :G] = -0.0
    q0, s0 = oracle.quant_act(synth.f32_to_bf16_bits(x), axis=0)
    q1, s1 = oracle.quant_act(synth.f32_to_bf16_bits(x * np.float32(2.0 ** -12)), axis=0)
    assert np.array_equal(q0, q1)
    assert np.array_equal(s1, s0 * np.float32(2.0 ** -12))
    assert s0[1, 5] == 0.0 and np.all(q0[5, G:2 * G] == 0x00)
    assert s0[0, 9] == 0.0 and np.all(q0[9, :G] == 0x80)


def test_weight_zero_and_underflowing_scale():
    w = np.zeros((G, 2 * G), np.float32)
    w[3, 200] = 1e-44          # amax/448 underflows to 0 in FP32
    w[7, 201] = -1e-45
    q, s = oracle.quant_w(w)
    assert s[0, 0] == 0.0 and s[0, 1] == 0.0
    assert np.all(q[:, :G] == 0) and q[3, 200] == 0x00 and q[7, 201] == 0x80


def test_weight_error_bound_and_transpose():
    rng = np.random.default_rng(41)
    w = synth.master_weight(rng, 2 * G, 3 * G)
    q, s, qt = oracle.quant_w(w, transposed=True)
    assert np.array_equal(qt, q.T)
    sc = np.kron(s.astype(np.float64), np.ones((G, G)))
    deq = oracle.e4m3_decode(q) * sc
    quot = (w / sc.astype(np.float32)).astype(np.float64)
    bound = _half_spacing(quot) * sc + np.abs(w / sc - quot) * sc
    assert np.all(np.abs(w - deq) <= bound * (1 + 1e-12))
    blocks = np.abs(w).reshape(2, G, 3, G).max(axis=(1, 3))
    assert np.array_equal(s, blocks / np.float32(448))


@pytest.mark.parametrize("axis", [0, 1])
def test_matches_independent_quantizer(axis):
    mld = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(51 + axis)
    xb = synth.gradients_token_outliers(rng, 256, 256)
    x = synth.bf16_bits_to_f32(xb)
    q, s = oracle.quant_act(xb, axis=axis)
    xv = x if axis == 0 else x.T
    grp = np.ascontiguousarray(xv).reshape(xv.shape[0], -1, G)
    s_ref = np.abs(grp).max(axis=2) / np.float32(448)
    q_ref = (grp / s_ref[:, :, None]).astype(mld.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(s, s_ref.T)
    assert np.array_equal(q, q_ref.reshape(xv.shape))


def test_rejects_partial_groups():
    with pytest.raises(ValueError):
        oracle.quant_act(np.zeros((4, 100), np.uint16), axis=0)
    with pytest.raises(ValueError):
        oracle.quant_act(np.zeros((100, 4), np.uint16), axis=1)
    with pytest.raises(ValueError):
        oracle.quant_w(np.zeros((G, 100), np.float32))
