"""Fine-grained FP8 (E4M3) quantization and block-scaled FP8 GEMM for GB300.

The compute lives in ``lib/libfp8fg.so`` (CUDA, sm_103a), whose C ABI is
declared in ``include/fp8fg.h``; ``binding`` exposes the same entry points
to Python over torch tensors.  ``synth`` holds the seeded synthetic input
generators; ``build`` compiles the library in-tree.
"""
from .binding import (  # noqa: F401
    FP8FG_AXIS_COLS, FP8FG_AXIS_ROWS, FP8FG_BSCALE_BLOCK128, FP8FG_BSCALE_ROW, FP8FG_ERR_CUDA,
    FP8FG_ERR_INVALID_ARG, FP8FG_ERR_MISALIGNED, FP8FG_ERR_TEARDOWN, FP8FG_ERR_TIMEOUT, FP8FG_ERR_TOO_LARGE,
    FP8FG_ERR_UNSUPPORTED_DEVICE, FP8FG_OK, FP8FG_OUT_BF16, FP8FG_OUT_F32, Fp8fgError, fp8_gemm_blockscaled,
    fp8_gemm_grouped, fp8_gemm_quant_a, fp8_quant_act_1x128, fp8_quant_act_dual, fp8_quant_w_128x128, fp8fg_last_device_status,
    fp8fg_selftest_watchdog, fp8fg_set_wait_limit, fp8fg_status_string,
)
