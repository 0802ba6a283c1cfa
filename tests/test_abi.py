"""The C ABI without a GPU: the library builds and loads, exports every entry
point include/fp8fg.h declares, and rejects bad arguments on the host before
touching a device.  No compute call is made here."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8fg.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n.startswith("fp8")))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ["fp8_quant_act_1x128", "fp8_quant_act_dual", "fp8_quant_w_128x128", "fp8_gemm_blockscaled", "fp8_gemm_grouped",
              "fp8fg_status_string", "fp8fg_last_device_status", "fp8fg_selftest_watchdog",
              "fp8fg_set_wait_limit", "fp8fg_check_compute_capability"]:
        assert n in names


def test_library_exports_every_declared_symbol(cuda_lib_path):
    lib = ctypes.CDLL(cuda_lib_path)
    for n in _declared_functions():
        assert hasattr(lib, n), f"{n} declared in fp8fg.h but not exported"
    from fp8_fine_grained_act_gb300 import binding
    assert set(binding.SIGNATURES) == set(_declared_functions())


def test_status_strings(cuda_lib_path):
    from fp8_fine_grained_act_gb300 import binding as b
    for code, word in [(0, "OK"), (1, "INVALID_ARG"), (2, "MISALIGNED"), (3, "UNSUPPORTED"), (4, "CUDA"),
                       (5, "TIMEOUT"), (6, "TEARDOWN"), (7, "TOO_LARGE")]:
        assert word in b.status_string(code)
    assert "unknown" in b.status_string(99)


def test_compute_capability_rule(cuda_lib_path):
    """The device rule every entry point applies before a launch: sm_103
    (10.3) only, with no fallback for any other architecture.  Checked on the
    rule itself, so no such device is needed."""
    from fp8_fine_grained_act_gb300 import binding as b
    lib = b.load()
    assert lib.fp8fg_check_compute_capability(10, 3) == b.FP8FG_OK
    for major, minor in [(10, 0), (10, 1), (10, 4), (9, 0), (8, 9), (11, 0), (12, 0), (12, 1), (0, 0), (-1, 3)]:
        assert lib.fp8fg_check_compute_capability(major, minor) == b.FP8FG_ERR_UNSUPPORTED_DEVICE


def test_noalloc_rejects_oversize_on_the_host(cuda_lib_path):
    """More rows than the fixed band-counter array covers is refused before
    any CUDA call (so this runs without a GPU)."""
    from fp8_fine_grained_act_gb300 import binding as b
    st = b.load().fp8_gemm_quant_a_noalloc(None, None, None, None, None, 1, 1, None, b.FP8FG_OUT_BF16,
                                           4096 * 128 + 128, 128, 128, None)
    assert st == b.FP8FG_ERR_TOO_LARGE


@pytest.fixture(scope="module")
def lib(cuda_lib_path):
    from fp8_fine_grained_act_gb300 import binding as b
    return b.load()


A16 = 0x10000          # a 16-byte aligned fake address: never dereferenced (rejected before any launch)


def _has_gpu() -> bool:
    import torch
    return torch.cuda.is_available()

MIS = 0x10008          # an 8-byte aligned fake address
MIS2 = 0x10002         # a 2-byte aligned fake address (bad even for a scale array)
NOPROBE = (3, 4)       # arguments accepted; the device probe then fails (no GPU here)


def test_quant_act_argument_checks(lib):
    f = lib.fp8_quant_act_1x128
    assert f(A16, 4, 100, 0, A16, A16, None) == 1          # cols not a multiple of 128
    assert f(A16, 100, 8, 1, A16, A16, None) == 1          # rows not a multiple of 128 for 128x1
    assert f(A16, 128, 12, 1, A16, A16, None) == 1         # cols not a multiple of 8 for 128x1
    assert f(A16, 4, 128, 2, A16, A16, None) == 1          # bad axis
    assert f(A16, -1, 128, 0, A16, A16, None) == 1
    assert f(None, 4, 128, 0, A16, A16, None) == 1         # null input
    assert f(A16, 4, 128, 0, None, A16, None) == 1
    assert f(A16, 4, 128, 0, A16, None, None) == 1
    assert f(MIS, 4, 128, 0, A16, A16, None) == 2          # misaligned
    assert f(A16, 4, 128, 0, MIS, A16, None) == 2
    assert f(A16, 4, 128, 0, A16, MIS2, None) == 2         # scales need 4-byte alignment
    if not _has_gpu():
        assert f(A16, 4, 128, 0, A16, MIS, None) in NOPROBE   # ... and no more
    assert f(None, 0, 128, 0, None, None, None) == 0       # empty: no-op, nothing touched
    assert f(None, 4, 0, 0, None, None, None) == 0


def test_quant_dual_argument_checks(lib):
    f = lib.fp8_quant_act_dual
    assert f(A16, 128, 100, A16, A16, A16, A16, None) == 1        # cols not a multiple of 128
    assert f(A16, 100, 128, A16, A16, A16, A16, None) == 1        # rows not a multiple of 128
    assert f(A16, 128, 128, A16, A16, None, A16, None) == 1       # null output
    assert f(A16, 128, 128, A16, A16, MIS, A16, None) == 2        # misaligned codes
    assert f(A16, 128, 128, A16, MIS2, A16, A16, None) == 2       # misaligned scales
    assert f(None, 0, 128, None, None, None, None, None) == 0     # empty: no-op


def test_quant_w_argument_checks(lib):
    f = lib.fp8_quant_w_128x128
    assert f(A16, 128, 100, A16, None, A16, None) == 1
    assert f(A16, 100, 128, A16, None, A16, None) == 1
    assert f(None, 128, 128, A16, None, A16, None) == 1
    assert f(A16, 128, 128, A16, MIS, A16, None) == 2      # misaligned transposed output
    assert f(A16, 128, 128, A16, None, MIS2, None) == 2
    assert f(A16, 0, 128, None, None, None, None) == 0


def test_gemm_argument_checks(lib):
    f = lib.fp8_gemm_blockscaled
    ok = dict(a=A16, sa=A16, b=A16, sb=A16, bscale=0, sn=1, sk=1, d=A16, od=1, M=128, N=128, K=128)

    def call(**kw):
        v = dict(ok, **kw)
        return f(v["a"], v["sa"], v["b"], v["sb"], v["bscale"], v["sn"], v["sk"], v["d"], v["od"],
                 v["M"], v["N"], v["K"], None)

    assert call(N=200) == 1 and call(K=130) == 1
    assert call(M=100, bscale=1) == 1                      # per-row B scales: whole row tiles only
    if not _has_gpu():
        assert call(M=100) in NOPROBE                      # block B scales take any M
    assert call(M=-128) == 1
    assert call(od=7) == 1 and call(bscale=3) == 1
    assert call(sn=-1) == 1
    assert call(a=None) == 1 and call(sb=None) == 1 and call(d=None) == 1
    assert call(a=MIS) == 2 and call(d=MIS) == 2 and call(sa=MIS2) == 2 and call(sb=MIS2) == 2
    assert call(bscale=1, sb=MIS) == 2                     # per-row B scales: 16-byte aligned scale arrays
    assert call(bscale=1, sa=MIS) == 2                     # ... both of them
    if not _has_gpu():
        assert call(sa=MIS) in NOPROBE and call(sb=MIS) in NOPROBE
    assert call(M=0, a=None, d=None) == 0                  # empty: no-op
    assert call(M=1 << 32) == 1                            # beyond the supported range
    g = lib.fp8_gemm_grouped
    assert g(A16, A16, A16, A16, A16, 0, A16, 1, 128, 128, 128, None) == 1       # G < 1
    assert g(A16, A16, A16, A16, None, 4, A16, 1, 128, 128, 128, None) == 1      # no offsets
    assert g(A16, A16, A16, A16, A16 + 2, 4, A16, 1, 128, 128, 128, None) == 2   # offsets not 4-aligned
    assert g(A16, A16, A16, A16, A16, 4, A16, 1, 100, 128, 128, None) == 1
    assert g(A16, A16, A16, A16, A16, 4097, A16, 1, 128, 128, 128, None) == 1    # G > 4096
    assert g(A16, A16, A16, A16, A16, 4, A16, 7, 128, 128, 128, None) == 1       # bad output type
    assert g(MIS, A16, A16, A16, A16, 4, A16, 1, 128, 128, 128, None) == 2       # misaligned codes
    assert g(A16, A16, A16, MIS2, A16, 4, A16, 1, 128, 128, 128, None) == 2      # misaligned scales
    assert g(A16, A16, A16, A16, A16, 4, MIS, 1, 128, 128, 128, None) == 2       # misaligned output
    assert g(None, None, None, None, A16, 4, None, 1, 0, 128, 128, None) == 0    # empty: no-op


def test_watchdog_argument_checks(lib):
    assert lib.fp8fg_selftest_watchdog(0, None) == 1
    assert lib.fp8fg_selftest_watchdog(2_000_000_000, None) == 1


def test_wait_limit_range(lib):
    assert lib.fp8fg_set_wait_limit(-1) == 1
    assert lib.fp8fg_set_wait_limit(10_000_000_001) == 1
    assert lib.fp8fg_set_wait_limit(10_000_000_000) == 0
    assert lib.fp8fg_set_wait_limit(1) == 0
    assert lib.fp8fg_set_wait_limit(0) == 0             # back to the default


def test_no_device_means_an_error_not_a_fallback(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid arguments reach the device probe, which fails: no CPU path exists
    st = lib.fp8_quant_act_1x128(A16, 4, 128, 0, A16, A16, None)
    assert st in (3, 4)


def test_binding_rejects_host_tensors_before_any_call(lib):
    """The Python binding only marshals: tensors that are not contiguous CUDA
    tensors of the right dtype are refused with ValueError, before the C ABI
    (and any device) is reached."""
    import torch
    from fp8_fine_grained_act_gb300 import binding as b
    x = torch.zeros((128, 128), dtype=torch.bfloat16)                # host tensor
    with pytest.raises(ValueError):
        b.fp8_quant_act_1x128(x)
    with pytest.raises(ValueError):
        b.fp8_quant_act_dual(x)
    with pytest.raises(ValueError):
        b.fp8_quant_act_1x128(torch.zeros((128, 128), dtype=torch.float32))
    with pytest.raises(ValueError):
        b._need(torch.zeros((4, 4)), torch.float32, (4, 4), "d")    # right dtype and shape, not on a GPU


def test_gemm_bindings_check_every_operand_before_any_call(lib):
    """Both GEMM bindings refuse host, mistyped, misshaped or non-contiguous
    operands and undersized scale arrays with ValueError before the C ABI is
    reached: a raw pointer to host memory or past the end of a scale array
    must never reach a TMA load or a scale read on the device."""
    import torch
    from fp8_fine_grained_act_gb300 import binding as b
    M, N, K = 128, 256, 256
    a = torch.zeros((M, K), dtype=torch.uint8)
    bb = torch.zeros((N, K), dtype=torch.uint8)
    sa = torch.zeros((K // 128, M), dtype=torch.float32)
    sb = torch.zeros((N // 128, K // 128), dtype=torch.float32)
    with pytest.raises(ValueError):                                   # host operands
        b.fp8_gemm_blockscaled(a, sa, bb, sb)
    with pytest.raises(ValueError):                                   # mistyped A
        b.fp8_gemm_blockscaled(a.float(), sa, bb, sb)
    with pytest.raises(ValueError):                                   # non-contiguous B
        b.fp8_gemm_blockscaled(a, sa, torch.zeros((K, N), dtype=torch.uint8).t(), sb)
    with pytest.raises(ValueError):                                   # bad bscale enum
        b.fp8_gemm_blockscaled(a, sa, bb, sb, bscale=5)
    with pytest.raises(ValueError):                                   # negative strides
        b.fp8_gemm_blockscaled(a, sa, bb, sb, sb_strides=(-1, 1))
    G = 2
    off = torch.tensor([0, 128, 128], dtype=torch.int32)
    with pytest.raises(ValueError):
        b.fp8_gemm_grouped(a, sa, torch.zeros((G, N, K), dtype=torch.uint8),
                           torch.zeros((G, N // 128, K // 128)), off)
    with pytest.raises(ValueError):                                   # B not [G, N, K]
        b.fp8_gemm_grouped(a, sa, bb, sb, off)
    # the size rule of a strided block-scale array: the last index read is
    # (N/128 - 1) * stride_n + (K/128 - 1) * stride_k
    with pytest.raises(ValueError):
        b._need_flat(torch.zeros(3), torch.float32, 4, "sb", torch.device("cpu"))


def test_fused_gemm_argument_checks(lib):
    f = lib.fp8_gemm_quant_a
    ok = dict(x=A16, qa=A16, sa=A16, b=A16, sb=A16, sn=1, sk=1, d=A16, od=1, M=128, N=128, K=128, fl=A16)

    def call(**kw):
        v = dict(ok, **kw)
        return f(v["x"], v["qa"], v["sa"], v["b"], v["sb"], v["sn"], v["sk"], v["d"], v["od"], v["M"], v["N"],
                 v["K"], v["fl"], None)

    assert call(M=100) == 1 and call(N=200) == 1 and call(K=130) == 1 and call(od=9) == 1
    assert call(sn=-1) == 1
    assert call(x=None) == 1 and call(qa=None) == 1 and call(sa=None) == 1 and call(fl=None) == 1
    assert call(b=None) == 1 and call(d=None) == 1
    assert call(x=MIS) == 2 and call(qa=MIS) == 2 and call(sa=MIS2) == 2 and call(fl=MIS2) == 2
    assert call(d=MIS) == 2 and call(b=MIS) == 2
    assert call(M=0, x=None, qa=None, sa=None, b=None, sb=None, d=None, fl=None) == 0    # empty: no-op
    if not _has_gpu():
        assert call() in NOPROBE
        # K == 0: only d is used, the empty input buffers may be null
        assert call(K=0, x=None, qa=None, sa=None, b=None, sb=None, fl=None) in NOPROBE
