"""Pins for the oracle's block-scaled GEMM and its tolerance (CPU only).

What fixes each expected value:
  * brute force in exact rational arithmetic (Python Fractions) on tiny
    inputs spanning two 128-wide K chunks: the double oracle must be within
    2^-48 * m of the exact sum, for 128x128 block scales, transposed block
    strides and per-row B scales;
  * special case that reduces to integer arithmetic: E4M3 codes whose values
    are integers with all scales 1 -- the result is an exact int64 matmul
    (numpy), and must match bit for bit;
  * scale indexing: A with one non-zero per row, placed in a chosen K chunk,
    with a distinct power-of-two scale for every (row, chunk) and every B
    block -- each output is one product of known scales, so a swapped
    index, stride or transposed operand gives a different power of two;
  * closed form for rank-1 operands: o[i, j] = u_i v_j * sum_k p_k r_k;
  * an independent path: numpy's float64 matmul of dequantized operands
    built with ml_dtypes decoding and scale expansion by np.repeat / np.kron;
  * the grouped variant: each expert has a constant weight, so every output
    row shows which expert it used;
  * tolerance helpers: BF16 spacing at chosen values.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest

import oracle
from fp8_fine_grained_act_gb300 import synth

G = 128


def _codes(rng, shape, max_mag=0x7E):
    mag = rng.integers(0, max_mag + 1, size=shape).astype(np.uint8)
    return mag | (rng.integers(0, 2, size=shape).astype(np.uint8) << 7)


def _scales(rng, shape):
    return np.exp2(rng.uniform(-8, 4, size=shape)).astype(np.float32)


def _exact(qa, sa, qb, sb_of):
    """Exact D = A.B^T in Fractions; sb_of(j, k) is the B scale."""
    M, K = qa.shape
    N = qb.shape[0]
    dec = [Fraction(float(v)) if not np.isnan(v) else None for v in oracle.e4m3_decode(np.arange(256, dtype=np.uint8))]
    out = np.empty((M, N), dtype=object)
    for i in range(M):
        for j in range(N):
            acc = Fraction(0)
            for k in range(K):
                a = dec[qa[i, k]] * Fraction(float(sa[k // G, i]))
                b = dec[qb[j, k]] * Fraction(float(sb_of(j, k)))
                acc += a * b
            out[i, j] = acc
    return out


@pytest.mark.parametrize("mode", ["block", "block_transposed", "row"])
def test_exact_rational_bruteforce(mode):
    rng = np.random.default_rng({"block": 1, "block_transposed": 2, "row": 3}[mode])
    # K spans two chunks; with block scales N spans two B blocks
    M, K = 3, 2 * G
    N = 2 * G if mode != "row" else 5
    qa = _codes(rng, (M, K))
    qb = _codes(rng, (N, K))
    sa = _scales(rng, (K // G, M))
    jj = np.array([0, 1, N - 1, (N // 2 + 3) % N])
    ii = np.array([0, 2, 1, 2])
    if mode == "block":
        sb = _scales(rng, (N // G, K // G))
        o, m = oracle.gemm_entries(qa, sa, qb, sb, ii, jj)
        sb_of = lambda j, k: sb[j // G, k // G]
    elif mode == "block_transposed":
        sbt = _scales(rng, (K // G, N // G))            # stored as [k_blk, n_blk]
        o, m = oracle.gemm_entries(qa, sa, qb, sbt, ii, jj, sb_strides=(1, N // G))
        sb_of = lambda j, k: sbt[k // G, j // G]
    else:
        sb = _scales(rng, (K // G, N))
        o, m = oracle.gemm_entries(qa, sa, qb, sb, ii, jj, bscale=oracle.BSCALE_ROW)
        sb_of = lambda j, k: sb[k // G, j]
    for e, (i, j) in enumerate(zip(ii, jj)):
        ex = _exact(qa[i:i + 1], sa[:, i:i + 1], qb[j:j + 1], lambda _j, k: sb_of(j, k))[0, 0]
        assert abs(Fraction(o[e]) - ex) <= Fraction(m[e]) * Fraction(1, 2 ** 48)
        assert m[e] >= abs(o[e])


def test_integer_special_case_exact():
    rng = np.random.default_rng(5)
    # codes with integer values: 0..15 in E4M3 are 0x00 (0), 0x38 (1), 0x40 (2), 0x44 (3), ...
    ints = np.arange(0, 17)
    enc = oracle.e4m3_encode(ints.astype(np.float32))
    assert np.array_equal(oracle.e4m3_decode(enc), ints)      # all exact
    M, N, K = 40, 3 * G, 4 * G
    ia = rng.integers(-16, 17, size=(M, K))
    ib = rng.integers(-16, 17, size=(N, K))
    qa = oracle.e4m3_encode(ia.astype(np.float32))
    qb = oracle.e4m3_encode(ib.astype(np.float32))
    o, m = oracle.gemm(qa, np.ones((K // G, M), np.float32), qb, np.ones((N // G, K // G), np.float32))
    want = ia.astype(np.int64) @ ib.astype(np.int64).T
    assert np.array_equal(o, want.astype(np.float64))
    assert np.array_equal(m, (np.abs(ia) @ np.abs(ib).T).astype(np.float64))


def test_scale_indexing_single_terms():
    M, N, K = 2 * G, 2 * G, 3 * G
    kb, nb = K // G, N // G
    # A row i has a single 1.0 at k = 128*c_i + (i % 128); its scale 2^(i%7 + 3c)
    c_of = np.arange(M) % kb
    qa = np.zeros((M, K), np.uint8)
    qa[np.arange(M), c_of * G + (np.arange(M) % G)] = 0x38
    sa = np.exp2((np.arange(M)[None, :] % 7) + 3 * np.arange(kb)[:, None]).astype(np.float32)
    # B: value 2.0 everywhere, block scale 2^-(5*nblk + kblk)
    qb = np.full((N, K), 0x40, np.uint8)
    sb = np.exp2(-(5 * np.arange(nb)[:, None] + np.arange(kb)[None, :])).astype(np.float32)
    o, m = oracle.gemm(qa, sa, qb, sb)
    i = np.arange(M)[:, None]
    j = np.arange(N)[None, :]
    want = 2.0 * np.exp2((i % 7) + 3 * c_of[:, None]) * np.exp2(-(5 * (j // G) + c_of[:, None]))
    assert np.array_equal(o, want)
    assert np.array_equal(m, want)
    # the same B scales stored transposed and read through swapped strides
    o2, _ = oracle.gemm(qa, sa, qb, np.ascontiguousarray(sb.T), sb_strides=(1, nb))
    assert np.array_equal(o2, want)
    # per-row B scales: 2^-(j % 9 + kblk)
    sbr = np.exp2(-((np.arange(N)[None, :] % 9) + np.arange(kb)[:, None])).astype(np.float32)
    o3, _ = oracle.gemm(qa, sa, qb, sbr, bscale=oracle.BSCALE_ROW)
    want3 = 2.0 * np.exp2((i % 7) + 3 * c_of[:, None]) * np.exp2(-((j % 9) + c_of[:, None]))
    assert np.array_equal(o3, want3)


def test_rank_one_closed_form():
    rng = np.random.default_rng(6)
    M, N, K = 16, G, 2 * G
    p = _codes(rng, (K,), 0x60)
    r = _codes(rng, (K,), 0x60)
    qa = np.tile(p, (M, 1))
    qb = np.tile(r, (N, 1))
    u = np.exp2(rng.integers(-5, 5, size=M)).astype(np.float32)
    v = np.exp2(rng.integers(-5, 5, size=N // G)).astype(np.float32)
    sa = np.tile(u, (K // G, 1))
    sb = np.tile(v[:, None], (1, K // G))
    o, _ = oracle.gemm(qa, sa, qb, sb)
    dot = float(np.sum(oracle.e4m3_decode(p) * oracle.e4m3_decode(r)))    # exact: small dyadics
    want = np.outer(u.astype(np.float64), np.repeat(v.astype(np.float64), G)) * dot
    assert np.array_equal(o, want)


def test_matches_numpy_matmul_on_dequantized():
    mld = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(8)
    M, N, K = 3 * G, 3 * G, 4 * G
    qa = _codes(rng, (M, K))
    qb = _codes(rng, (N, K))
    sa = _scales(rng, (K // G, M))
    sb = _scales(rng, (N // G, K // G))
    dec = lambda q: q.view(mld.float8_e4m3fn).astype(np.float64)
    a = dec(qa) * np.repeat(sa.T.astype(np.float64), G, axis=1)
    b = dec(qb) * np.kron(sb.astype(np.float64), np.ones((G, G)))
    o, m = oracle.gemm(qa, sa, qb, sb)
    ref = a @ b.T
    mref = np.abs(a) @ np.abs(b).T
    assert np.all(np.abs(o - ref) <= 2.0 ** -44 * mref)
    assert np.allclose(m, mref, rtol=2.0 ** -44, atol=0)
    sbr = _scales(rng, (K // G, N))
    br = dec(qb) * np.repeat(sbr.T.astype(np.float64), G, axis=1)
    o2, m2 = oracle.gemm(qa, sa, qb, sbr, bscale=oracle.BSCALE_ROW)
    assert np.all(np.abs(o2 - a @ br.T) <= 2.0 ** -44 * (np.abs(a) @ np.abs(br).T))
    # entries agree with the full product
    ii = rng.integers(0, M, 50)
    jj = rng.integers(0, N, 50)
    oe, me = oracle.gemm_entries(qa, sa, qb, sb, ii, jj)
    assert np.array_equal(oe, o[ii, jj]) and np.array_equal(me, m[ii, jj])


def test_grouped_uses_each_experts_weight():
    G_e, N, K = 4, G, G
    offsets = np.array([0, 128, 128, 384, 512], np.int32)   # expert 1 is empty
    Mt = int(offsets[-1])
    qa = np.full((Mt, K), 0x38, np.uint8)                    # all ones
    sa = np.ones((K // G, Mt), np.float32)
    qb = np.full((G_e, N, K), 0x38, np.uint8)
    sb = np.stack([np.full((N // G, K // G), 2.0 ** g, np.float32) for g in range(G_e)])
    o, m = oracle.gemm_grouped(qa, sa, qb, sb, offsets)
    g_of_row = np.searchsorted(offsets, np.arange(Mt), side="right") - 1
    assert np.array_equal(o, np.repeat((K * np.exp2(g_of_row))[:, None], N, axis=1))
    ii = np.array([0, 127, 128, 383, 384, 511])
    jj = np.array([0, 5, 9, 127, 64, 1])
    oe, _ = oracle.gemm_grouped_entries(qa, sa, qb, sb, offsets, ii, jj)
    assert np.array_equal(oe, o[ii, jj])


def test_tolerance_helpers():
    o = np.array([1.0, 1.5, -3.0, 2.0 ** -130, 0.0, 448.0])
    assert np.array_equal(oracle.bf16_ulp(o), [2.0 ** -7, 2.0 ** -7, 2.0 ** -6, 2.0 ** -133, 2.0 ** -133, 2.0 ** 1])
    t = oracle.gemm_tolerance(np.array([1.0]), np.array([2.0 ** 16]), "f32")
    assert t[0] == 1.0
    t = oracle.gemm_tolerance(np.array([1.0]), np.array([2.0 ** 16]), "bf16")
    assert t[0] == 1.0 + 2.0 ** -7


def test_synthetic_workload_recipes():
    # the grouped workload's group sizes (the same first draws as grouped_moe(seed=4))
    counts, padded, off = synth.moe_group_sizes(np.random.default_rng(4))
    assert off.dtype == np.int32 and off.shape == (65,)
    assert np.all(off % 128 == 0) and np.all(np.diff(off) >= 0)
    assert int(counts.sum()) == 32768
    assert int(off[-1]) == 37120                   # M_total of the seed-4 draw
    # the token rows: N(0,1) then zero pad rows, per expert (the full recipe on 16 channels)
    d = synth.grouped_moe(seed=4, K=16, with_weights=False)
    assert np.array_equal(d["offsets"], off)
    assert d["x"].shape == (int(off[-1]), 16)
    g = int(np.argmax(padded - counts))
    r = int(off[g] + counts[g])
    assert np.all(d["x"][r:int(off[g + 1])] == 0)
    assert np.all(d["x"][int(off[g]):r] != 0)
    t = synth.tiny_fprop(seed=0)
    x = synth.bf16_bits_to_f32(t["x"])
    assert x.shape == (256, 512) and t["w"].shape == (256, 512)
    assert np.sum(np.abs(x) > 8) >= 100            # the 131 x100 outliers dominate the tail
    a = synth.tiny_fprop(seed=0)
    assert np.array_equal(a["x"], t["x"]) and np.array_equal(a["w"], t["w"])
