"""Python binding of the C ABI in ``include/fp8fg.h`` (ctypes over
``lib/libfp8fg.so``).

Argument marshalling only: every step of the quantization and the GEMM runs
in the library's CUDA kernels.  PyTorch provides device memory and the
current stream.  There is no CPU or PyTorch fallback: if the library is
missing the first call raises.

The functions carry the C names.  They take CUDA torch tensors, allocate any
output that is not given, call the entry point on the current stream (or
``stream``) and raise ``Fp8fgError`` on a non-zero status.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

FP8FG_OK = 0
FP8FG_ERR_INVALID_ARG = 1
FP8FG_ERR_MISALIGNED = 2
FP8FG_ERR_UNSUPPORTED_DEVICE = 3
FP8FG_ERR_CUDA = 4
FP8FG_ERR_TIMEOUT = 5
FP8FG_ERR_TEARDOWN = 6
FP8FG_ERR_TOO_LARGE = 7

FP8FG_OUT_F32 = 0
FP8FG_OUT_BF16 = 1
FP8FG_AXIS_COLS = 0
FP8FG_AXIS_ROWS = 1
FP8FG_BSCALE_BLOCK128 = 0
FP8FG_BSCALE_ROW = 1

GROUP = 128

# every entry point the header declares: name -> (restype, argtypes)
_vp, _i64, _i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
SIGNATURES = {
    "fp8_quant_act_1x128": (_i32, [_vp, _i64, _i64, _i32, _vp, _vp, _vp]),
    "fp8_quant_w_128x128": (_i32, [_vp, _i64, _i64, _vp, _vp, _vp, _vp]),
    "fp8_quant_act_dual": (_i32, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp]),
    "fp8_gemm_blockscaled": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i64, _vp, _i32, _i64, _i64, _i64, _vp]),
    "fp8_gemm_grouped": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i64, _i64, _i64, _vp]),
    "fp8_gemm_quant_a": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _vp, _i32, _i64, _i64, _i64, _vp, _vp]),
    "fp8_gemm_quant_a_noalloc": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _vp, _i32, _i64, _i64, _i64, _vp]),
    "fp8fg_status_string": (ctypes.c_char_p, [_i32]),
    "fp8fg_check_compute_capability": (_i32, [_i32, _i32]),
    "fp8fg_last_device_status": (_i32, [_vp]),
    "fp8fg_selftest_watchdog": (_i32, [_i64, _vp]),
    "fp8fg_set_wait_limit": (_i32, [_i64]),
    "fp8fg_probe_mma_rate": (_i32, [_i64, ctypes.POINTER(ctypes.c_int), _vp]),
}


class Fp8fgError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libfp8fg.so (optionally building it first).  Raises if it is
    missing: there is no fallback implementation."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing and (not os.path.exists(path) or _build.is_stale()):
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is not built; run fp8_fine_grained_act_gb300.build.build() "
                           "(nvcc for sm_103a). There is no CPU fallback.")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().fp8fg_status_string(int(status)).decode()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(st: int, where: str) -> None:
    if st != FP8FG_OK:
        raise Fp8fgError(st, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, shape, name, device=None):
    if (not isinstance(t, torch.Tensor) or t.dtype != dtype or tuple(t.shape) != tuple(shape)
            or not t.is_contiguous() or not t.is_cuda):
        got = f"{t.dtype} {tuple(t.shape)} on {t.device}" if isinstance(t, torch.Tensor) else type(t).__name__
        raise ValueError(f"{name}: expected contiguous CUDA {dtype} {tuple(shape)}, got {got}")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, the other operands on {device}")


def _need_flat(t, dtype, min_numel, name, device):
    """A contiguous CUDA array of at least ``min_numel`` elements (any shape):
    the block scales of a GEMM read through strides."""
    if (not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_contiguous() or not t.is_cuda
            or t.numel() < min_numel):
        got = f"{t.dtype} {tuple(t.shape)} on {t.device}" if isinstance(t, torch.Tensor) else type(t).__name__
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} array of >= {min_numel} elements, got {got}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, the other operands on {device}")


# ------------------------------------------------------------ quantizers ---

def fp8_quant_act_1x128(x: torch.Tensor, axis: int = FP8FG_AXIS_COLS, q=None, scales=None, stream=None):
    """BF16 x[rows, cols] -> (q uint8, scales float32).  axis 0 (1x128 along
    columns): q[rows, cols], scales[cols/128, rows].  axis 1 (128x1 along
    rows, transposed output): q[cols, rows], scales[rows/128, cols]."""
    rows, cols = x.shape
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or not x.is_cuda:
        raise ValueError("x must be a contiguous CUDA bfloat16 tensor")
    if axis == FP8FG_AXIS_COLS:
        qshape, sshape = (rows, cols), (cols // GROUP, rows)
    else:
        qshape, sshape = (cols, rows), (rows // GROUP, cols)
    if q is None:
        q = torch.empty(qshape, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(sshape, dtype=torch.float32, device=x.device)
    _need(q, torch.uint8, qshape, "q", x.device)
    _need(scales, torch.float32, sshape, "scales", x.device)
    st = load().fp8_quant_act_1x128(_ptr(x), rows, cols, int(axis), _ptr(q), _ptr(scales), _stream(stream))
    _check(st, "fp8_quant_act_1x128")
    return q, scales


def fp8_quant_act_dual(x: torch.Tensor, q_row=None, s_row=None, q_col_t=None, s_col=None, stream=None):
    """BF16 x[rows, cols] -> (q_row, s_row, q_col_t, s_col) from one read of x:
    the outputs of fp8_quant_act_1x128 with axis 0 and with axis 1."""
    rows, cols = x.shape
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or not x.is_cuda:
        raise ValueError("x must be a contiguous CUDA bfloat16 tensor")
    shapes = {"q_row": ((rows, cols), torch.uint8), "s_row": ((cols // GROUP, rows), torch.float32),
              "q_col_t": ((cols, rows), torch.uint8), "s_col": ((rows // GROUP, cols), torch.float32)}
    given = {"q_row": q_row, "s_row": s_row, "q_col_t": q_col_t, "s_col": s_col}
    for name, (shape, dt) in shapes.items():
        if given[name] is None:
            given[name] = torch.empty(shape, dtype=dt, device=x.device)
        _need(given[name], dt, shape, name, x.device)
    q_row, s_row, q_col_t, s_col = given["q_row"], given["s_row"], given["q_col_t"], given["s_col"]
    st = load().fp8_quant_act_dual(_ptr(x), rows, cols, _ptr(q_row), _ptr(s_row), _ptr(q_col_t), _ptr(s_col),
                                   _stream(stream))
    _check(st, "fp8_quant_act_dual")
    return q_row, s_row, q_col_t, s_col


def fp8_quant_w_128x128(w: torch.Tensor, transposed: bool = False, q=None, q_t=None, scales=None, stream=None):
    """FP32 w[rows, cols] -> (q[rows, cols], scales[rows/128, cols/128]) or,
    with ``transposed``, (q, q_t[cols, rows], scales)."""
    rows, cols = w.shape
    if w.dtype != torch.float32 or not w.is_contiguous() or not w.is_cuda:
        raise ValueError("w must be a contiguous CUDA float32 tensor")
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=w.device)
    if transposed and q_t is None:
        q_t = torch.empty((cols, rows), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((rows // GROUP, cols // GROUP), dtype=torch.float32, device=w.device)
    _need(q, torch.uint8, (rows, cols), "q", w.device)
    _need(scales, torch.float32, (rows // GROUP, cols // GROUP), "scales", w.device)
    if q_t is not None:
        _need(q_t, torch.uint8, (cols, rows), "q_t", w.device)
    st = load().fp8_quant_w_128x128(_ptr(w), rows, cols, _ptr(q), _ptr(q_t), _ptr(scales), _stream(stream))
    _check(st, "fp8_quant_w_128x128")
    return (q, q_t, scales) if transposed else (q, scales)


# ----------------------------------------------------------------- GEMMs ---

def _out(d, M, N, out_dtype, device):
    dt = torch.float32 if out_dtype == FP8FG_OUT_F32 else torch.bfloat16
    if d is None:
        d = torch.empty((M, N), dtype=dt, device=device)
    _need(d, dt, (M, N), "d", device)
    return d


def fp8_gemm_blockscaled(a, sa, b, sb, bscale: int = FP8FG_BSCALE_BLOCK128, sb_strides=None,
                         out_dtype: int = FP8FG_OUT_BF16, d=None, stream=None):
    """D[M,N] = A[M,K] . B[N,K]^T with group scales (see include/fp8fg.h).
    Block mode: sb_strides = (stride_n, stride_k) in elements, default
    (K/128, 1) for a row-major [N/128, K/128] array."""
    if not isinstance(a, torch.Tensor) or a.dim() != 2 or not isinstance(b, torch.Tensor) or b.dim() != 2:
        raise ValueError("a and b must be 2-D tensors [M, K] and [N, K]")
    M, K = a.shape
    N = b.shape[0]
    if b.shape[1] != K:
        raise ValueError("a and b disagree on K")
    dev = a.device
    _need(a, torch.uint8, (M, K), "a", dev)
    _need(b, torch.uint8, (N, K), "b", dev)
    _need(sa, torch.float32, (K // GROUP, M), "sa", dev)
    if bscale == FP8FG_BSCALE_BLOCK128:
        sn, sk = sb_strides if sb_strides is not None else (K // GROUP, 1)
        if sn < 0 or sk < 0:
            raise ValueError("sb_strides must be non-negative")
        last = (max(N // GROUP - 1, 0) * sn + max(K // GROUP - 1, 0) * sk + 1) if N and K else 0
        _need_flat(sb, torch.float32, last, "sb", dev)
    elif bscale == FP8FG_BSCALE_ROW:
        sn, sk = 0, 0
        _need(sb, torch.float32, (K // GROUP, N), "sb", dev)
    else:
        raise ValueError(f"bscale {bscale}: expected FP8FG_BSCALE_BLOCK128 or FP8FG_BSCALE_ROW")
    d = _out(d, M, N, out_dtype, dev)
    st = load().fp8_gemm_blockscaled(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), int(bscale), int(sn), int(sk),
                                     _ptr(d), int(out_dtype), M, N, K, _stream(stream))
    _check(st, "fp8_gemm_blockscaled")
    return d


def fp8_gemm_quant_a(x, b, sb, sb_strides=None, out_dtype: int = FP8FG_OUT_BF16, q_a=None, s_a=None, d=None,
                     band_flags=None, stream=None):
    """The 1x128 quantizer fused into the block-scaled GEMM (one launch):
    BF16 x[M, K], B codes b[N, K] with 128x128 block scales sb ->
    (d[M, N], q_a[M, K], s_a[K/128, M]); q_a and s_a are what
    fp8_quant_act_1x128(x) returns.  band_flags: int32[M/128] device
    workspace (allocated when not given)."""
    if not isinstance(x, torch.Tensor) or x.dim() != 2 or not isinstance(b, torch.Tensor) or b.dim() != 2:
        raise ValueError("x must be [M, K] and b [N, K]")
    M, K = x.shape
    N = b.shape[0]
    if b.shape[1] != K:
        raise ValueError("x and b disagree on K")
    dev = x.device
    _need(x, torch.bfloat16, (M, K), "x", dev)
    _need(b, torch.uint8, (N, K), "b", dev)
    sn, sk = sb_strides if sb_strides is not None else (K // GROUP, 1)
    if sn < 0 or sk < 0:
        raise ValueError("sb_strides must be non-negative")
    last = (max(N // GROUP - 1, 0) * sn + max(K // GROUP - 1, 0) * sk + 1) if N and K else 0
    _need_flat(sb, torch.float32, last, "sb", dev)
    if q_a is None:
        q_a = torch.empty((M, K), dtype=torch.uint8, device=dev)
    if s_a is None:
        s_a = torch.empty((K // GROUP, M), dtype=torch.float32, device=dev)
    if band_flags is None:
        band_flags = torch.empty((max(M // GROUP, 1),), dtype=torch.int32, device=dev)
    _need(q_a, torch.uint8, (M, K), "q_a", dev)
    _need(s_a, torch.float32, (K // GROUP, M), "s_a", dev)
    if band_flags.dtype != torch.int32 or not band_flags.is_cuda or band_flags.numel() < M // GROUP \
            or not band_flags.is_contiguous() or band_flags.device != dev:
        raise ValueError(f"band_flags: a contiguous CUDA int32 tensor of >= {M // GROUP} elements on {dev}")
    d = _out(d, M, N, out_dtype, dev)
    st = load().fp8_gemm_quant_a(_ptr(x), _ptr(q_a), _ptr(s_a), _ptr(b), _ptr(sb), int(sn), int(sk), _ptr(d),
                                 int(out_dtype), M, N, K, _ptr(band_flags), _stream(stream))
    _check(st, "fp8_gemm_quant_a")
    return d, q_a, s_a


def fp8_gemm_grouped(a, sa, b, sb, group_offsets, out_dtype: int = FP8FG_OUT_BF16, d=None, stream=None):
    """Grouped MoE GEMM: a[M_total, K], b[G, N, K], sb[G, N/128, K/128],
    group_offsets int32[G+1] on the device."""
    if not isinstance(a, torch.Tensor) or a.dim() != 2 or not isinstance(b, torch.Tensor) or b.dim() != 3:
        raise ValueError("a must be [M_total, K] and b [G, N, K]")
    M, K = a.shape
    G, N, Kb = b.shape
    if Kb != K:
        raise ValueError("a and b disagree on K")
    dev = a.device
    _need(a, torch.uint8, (M, K), "a", dev)
    _need(b, torch.uint8, (G, N, K), "b", dev)
    _need(sa, torch.float32, (K // GROUP, M), "sa", dev)
    _need(sb, torch.float32, (G, N // GROUP, K // GROUP), "sb", dev)
    _need(group_offsets, torch.int32, (G + 1,), "group_offsets", dev)
    d = _out(d, M, N, out_dtype, dev)
    st = load().fp8_gemm_grouped(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(group_offsets), int(G), _ptr(d),
                                 int(out_dtype), M, N, K, _stream(stream))
    _check(st, "fp8_gemm_grouped")
    return d


def fp8fg_last_device_status(stream=None) -> int:
    return int(load().fp8fg_last_device_status(_stream(stream)))


def fp8fg_selftest_watchdog(timeout_ns: int, stream=None) -> int:
    return int(load().fp8fg_selftest_watchdog(int(timeout_ns), _stream(stream)))


def fp8fg_set_wait_limit(limit_ns: int) -> int:
    """Limit of the GEMM kernels' bounded waits (0: the 2 s default)."""
    return int(load().fp8fg_set_wait_limit(int(limit_ns)))


def fp8fg_status_string(status: int) -> str:
    return status_string(status)


def fp8fg_probe_mma_rate(chunks: int, stream=None) -> int:
    """Launch the tensor-rate probe (back-to-back FP8 MMAs, one CTA per SM)
    on the stream; returns the number of CTAs.  Its FLOPs are
    ctas * chunks * 2 * 128 * 256 * 128."""
    n = ctypes.c_int(0)
    _check(load().fp8fg_probe_mma_rate(int(chunks), ctypes.byref(n), _stream(stream)), "fp8fg_probe_mma_rate")
    return int(n.value)
