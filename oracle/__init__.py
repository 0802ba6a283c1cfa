"""CPU oracle for fine-grained FP8 quantization and the block-scaled FP8 GEMM.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The CUDA
library in ``fp8_fine_grained_act_gb300`` never calls it and shares no code
with it.

The arithmetic lives in plain C (``fp8fg_oracle.c``, double precision for the
GEMM, IEEE single precision for the scale and the element quotient); this
module is argument marshalling over numpy arrays plus the grouped-expert
driver, which calls the dense oracle once per expert.

Sources of each step (page title and section):
  * E4M3, 4-bit exponent + 3-bit mantissa: "FP8 Mixed-Precision Training:
    Hardware Acceleration Beyond NVIDIA's Paradigm", section 1.1; the
    max-448 variant is the OCP 8-bit floating point E4M3 format.
  * Scale the group's maximum magnitude to the FP8 maximum, 1x128 tiles for
    activations and 128x128 blocks for weights: DeepSeek-V3 FP8 post
    (innerforce.co.kr), fine-grained quantization, Figure 7 (a).
  * Online scales from the current group: "Unified E4M3 format in
    DeepSeek-V3" (codingmall.com), Dynamic Scaling and Online Quantization.
  * Fprop / Dgrad / Wgrad operand roles and output dtypes: "DeepSeek FP8
    Training" (arcalunar.github.io), forward pipeline and the two backward
    pipelines.
  * Grouped MoE experts: contiguous token groups, one weight per expert,
    groups padded to 128 rows (DeepSeek-V3 FP8 post, MoE training
    paragraphs; the padding is this library's reading).

Every function is pinned by ``tests/test_oracle_*.py`` against values fixed
by the format definition, closed forms, brute force and an independent
library (see the header of each test file).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8fg_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")

GROUP = 128
E4M3_MAX = 448.0

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (no FMA contraction, no
    fast-math, IEEE single division)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(_LIB_DIR, exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-fexcess-precision=standard",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    i64, u8p, f32p, f64p, i64p = (ctypes.c_int64, ctypes.POINTER(ctypes.c_uint8),
                                  ctypes.POINTER(ctypes.c_float),
                                  ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_int64))
    lib.fo_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.fo_e4m3_decode.restype = ctypes.c_double
    lib.fo_e4m3_encode.argtypes = [ctypes.c_float]
    lib.fo_e4m3_encode.restype = ctypes.c_uint8
    lib.fo_e4m3_encode_array.argtypes = [f32p, i64, u8p]
    lib.fo_e4m3_decode_array.argtypes = [u8p, i64, f64p]
    lib.fo_quant_act.argtypes = [ctypes.POINTER(ctypes.c_uint16), i64, i64, ctypes.c_int, u8p, f32p]
    lib.fo_quant_act.restype = ctypes.c_int
    lib.fo_quant_w.argtypes = [f32p, i64, i64, u8p, u8p, f32p]
    lib.fo_quant_w.restype = ctypes.c_int
    lib.fo_gemm_entries.argtypes = [u8p, f32p, i64, u8p, f32p, ctypes.c_int, i64, i64, i64,
                                    i64, i64, i64p, i64p, f64p, f64p]
    lib.fo_gemm_full.argtypes = [u8p, f32p, i64, u8p, f32p, ctypes.c_int, i64, i64, i64,
                                 i64, f64p, f64p, f64p, f64p]
    lib.fo_num_threads.restype = ctypes.c_int
    lib.fo_set_num_threads.argtypes = [ctypes.c_int]
    _lib = lib
    return lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def num_threads() -> int:
    return int(_load().fo_num_threads())


def set_num_threads(n: int) -> None:
    _load().fo_set_num_threads(int(n))


# ------------------------------------------------------------------ E4M3 ---

def e4m3_decode(codes) -> np.ndarray:
    """Exact value (float64) of each E4M3 code; 0x7F/0xFF are NaN."""
    shape = np.shape(codes)
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8).reshape(-1))
    out = np.empty(c.shape, dtype=np.float64)
    _load().fo_e4m3_decode_array(_ptr(c.reshape(-1), ctypes.c_uint8), c.size,
                                 _ptr(out.reshape(-1), ctypes.c_double))
    return out.reshape(shape)


def e4m3_encode(values) -> np.ndarray:
    """E4M3 code of each FP32 value: RNE, saturating to +-448."""
    shape = np.shape(values)
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float32).reshape(-1))
    out = np.empty(v.shape, dtype=np.uint8)
    _load().fo_e4m3_encode_array(_ptr(v.reshape(-1), ctypes.c_float), v.size,
                                 _ptr(out.reshape(-1), ctypes.c_uint8))
    return out.reshape(shape)


# ------------------------------------------------------------- quantize ---

def _bf16_bits(x) -> np.ndarray:
    """BF16 payload as uint16.  Accepts uint16 bit arrays or a torch bfloat16
    tensor on the CPU."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16, "BF16 input must be given as uint16 bits"
        return np.ascontiguousarray(x)
    import torch  # torch is only used to reinterpret the bits
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def quant_act(x_bf16, axis: int = 0):
    """Quantize BF16 activations or gradients.

    axis 0: 1x128 groups along the columns (per token per 128 channels);
      returns q[rows, cols] uint8 and s[cols/128, rows] float32.
    axis 1: 128x1 groups along the rows (128 tokens of one channel); returns
      q transposed, q[cols, rows], and s[rows/128, cols].
    """
    xb = _bf16_bits(x_bf16)
    rows, cols = xb.shape
    if axis == 0:
        q = np.empty((rows, cols), np.uint8)
        s = np.empty((cols // GROUP, rows), np.float32)
    else:
        q = np.empty((cols, rows), np.uint8)
        s = np.empty((rows // GROUP, cols), np.float32)
    rc = _load().fo_quant_act(_ptr(xb, ctypes.c_uint16), rows, cols, int(axis),
                              _ptr(q, ctypes.c_uint8), _ptr(s, ctypes.c_float))
    if rc != 0:
        raise ValueError(f"shape {xb.shape} does not tile into 128-element groups on axis {axis}")
    return q, s


def quant_w(w_f32: np.ndarray, transposed: bool = False):
    """Quantize an FP32 master weight w[rows, cols] in 128x128 blocks.
    Returns q[rows, cols], s[rows/128, cols/128] and, if asked, q_t[cols, rows]."""
    w = np.ascontiguousarray(np.asarray(w_f32, dtype=np.float32))
    rows, cols = w.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows // GROUP, cols // GROUP), np.float32)
    qt = np.empty((cols, rows), np.uint8) if transposed else None
    rc = _load().fo_quant_w(_ptr(w, ctypes.c_float), rows, cols, _ptr(q, ctypes.c_uint8),
                            _ptr(qt, ctypes.c_uint8) if transposed else None,
                            _ptr(s, ctypes.c_float))
    if rc != 0:
        raise ValueError(f"shape {w.shape} does not tile into 128x128 blocks")
    return (q, s, qt) if transposed else (q, s)


# ------------------------------------------------------------------ GEMM ---

BSCALE_BLOCK128 = 0
BSCALE_ROW = 1


def _sb_strides(sb: np.ndarray, bscale: int, N: int, K: int, sb_strides):
    if bscale == BSCALE_BLOCK128:
        if sb_strides is None:
            return K // GROUP, 1
        return int(sb_strides[0]), int(sb_strides[1])
    return 0, 0


def gemm(qa, sa, qb, sb, bscale: int = BSCALE_BLOCK128, sb_strides=None):
    """Whole output of D = A.B^T in double: returns (o[M,N], m[M,N]).

    qa[M,K], sa[K/128,M]; qb[N,K]; sb as bscale says (block: element
    (j,k) scale sb.flat[(j/128)*stride_n + (k/128)*stride_k], default strides
    (K/128, 1); row: sb[K/128, N])."""
    qa = np.ascontiguousarray(qa, np.uint8)
    qb = np.ascontiguousarray(qb, np.uint8)
    sa = np.ascontiguousarray(sa, np.float32)
    sb = np.ascontiguousarray(sb, np.float32)
    M, K = qa.shape
    N = qb.shape[0]
    assert qb.shape[1] == K
    sn, sk = _sb_strides(sb, bscale, N, K, sb_strides)
    a_deq = np.empty((M, K), np.float64)
    b_deq = np.empty((N, K), np.float64)
    o = np.empty((M, N), np.float64)
    m = np.empty((M, N), np.float64)
    _load().fo_gemm_full(_ptr(qa, ctypes.c_uint8), _ptr(sa, ctypes.c_float), M,
                         _ptr(qb, ctypes.c_uint8), _ptr(sb, ctypes.c_float), int(bscale), sn, sk, N,
                         K, _ptr(a_deq, ctypes.c_double), _ptr(b_deq, ctypes.c_double),
                         _ptr(o, ctypes.c_double), _ptr(m, ctypes.c_double))
    return o, m


def gemm_entries(qa, sa, qb, sb, ii, jj, bscale: int = BSCALE_BLOCK128, sb_strides=None):
    """Selected entries (ii[e], jj[e]) of D = A.B^T: returns (o[e], m[e])."""
    qa = np.ascontiguousarray(qa, np.uint8)
    qb = np.ascontiguousarray(qb, np.uint8)
    sa = np.ascontiguousarray(sa, np.float32)
    sb = np.ascontiguousarray(sb, np.float32)
    ii = np.ascontiguousarray(ii, np.int64)
    jj = np.ascontiguousarray(jj, np.int64)
    M, K = qa.shape
    N = qb.shape[0]
    sn, sk = _sb_strides(sb, bscale, N, K, sb_strides)
    o = np.empty(ii.shape, np.float64)
    m = np.empty(ii.shape, np.float64)
    _load().fo_gemm_entries(_ptr(qa, ctypes.c_uint8), _ptr(sa, ctypes.c_float), M,
                            _ptr(qb, ctypes.c_uint8), _ptr(sb, ctypes.c_float), int(bscale), sn, sk, N,
                            K, ii.size, _ptr(ii, ctypes.c_int64), _ptr(jj, ctypes.c_int64),
                            _ptr(o, ctypes.c_double), _ptr(m, ctypes.c_double))
    return o, m


def gemm_grouped_entries(qa, sa, qb_g, sb_g, offsets, ii, jj):
    """Grouped MoE-expert GEMM, selected entries.  Rows [offsets[g],
    offsets[g+1]) of A multiply expert weight g: qb_g[G,N,K], sb_g[G,N/128,K/128].
    The entry (i, j) uses the expert whose row range holds i."""
    offsets = np.asarray(offsets, np.int64)
    ii = np.asarray(ii, np.int64)
    jj = np.asarray(jj, np.int64)
    o = np.empty(ii.shape, np.float64)
    m = np.empty(ii.shape, np.float64)
    g_of = np.searchsorted(offsets, ii, side="right") - 1
    for g in np.unique(g_of):
        sel = np.nonzero(g_of == g)[0]
        o[sel], m[sel] = gemm_entries(qa, sa, qb_g[g], sb_g[g], ii[sel], jj[sel])
    return o, m


def gemm_grouped(qa, sa, qb_g, sb_g, offsets):
    """Whole output of the grouped GEMM, expert by expert, in double."""
    offsets = np.asarray(offsets, np.int64)
    M, K = qa.shape
    G, N, _ = qb_g.shape
    o = np.zeros((M, N), np.float64)
    m = np.zeros((M, N), np.float64)
    for g in range(G):
        r0, r1 = int(offsets[g]), int(offsets[g + 1])
        if r1 == r0:
            continue
        # the expert's rows of A with their own slice of the [K/128, M] scales
        og, mg = gemm(qa[r0:r1], np.ascontiguousarray(sa[:, r0:r1]), qb_g[g], sb_g[g])
        o[r0:r1] = og
        m[r0:r1] = mg
    return o, m


# ------------------------------------------------------------- tolerance ---

def bf16_ulp(o: np.ndarray) -> np.ndarray:
    """Spacing of BF16 numbers at |o|: 2^(floor(log2|o|) - 7), floored at the
    BF16 subnormal spacing 2^-133."""
    a = np.abs(np.asarray(o, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    return np.where(a > 0, np.exp2(e - 7.0), np.exp2(-133.0))


def gemm_tolerance(o: np.ndarray, m: np.ndarray, out_dtype: str) -> np.ndarray:
    """Allowed |gpu - o|: 2^-16 * m for FP32 output; plus one BF16 ulp of o
    for BF16 output."""
    tol = np.ldexp(np.asarray(m, np.float64), -16)
    if out_dtype == "bf16":
        tol = tol + bf16_ulp(o)
    return tol


__all__ = [
    "GROUP", "E4M3_MAX", "BSCALE_BLOCK128", "BSCALE_ROW", "build", "e4m3_decode", "e4m3_encode",
    "quant_act", "quant_w", "gemm", "gemm_entries", "gemm_grouped", "gemm_grouped_entries",
    "bf16_ulp", "gemm_tolerance", "num_threads", "set_num_threads",
]

if __name__ == "__main__":  # pragma: no cover
    print(build(force=True), file=sys.stderr)
