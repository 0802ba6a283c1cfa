"""Helpers shared by the GPU parity tests: moving the synthetic host arrays to
the device and comparing GEMM outputs with the oracle under the stated
tolerance."""
from __future__ import annotations

import numpy as np
import torch

import oracle


def dev_bf16(bits: np.ndarray, device) -> torch.Tensor:
    """BF16 device tensor with exactly these 16-bit patterns."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def dev(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.cpu().numpy()


def assert_gemm_close(gpu: np.ndarray, o: np.ndarray, m: np.ndarray, out_dtype: str, what: str = ""):
    """|gpu - o| <= 2^-16 m (+ one BF16 spacing of o for BF16 output)."""
    gpu = np.asarray(gpu, np.float64)
    tol = oracle.gemm_tolerance(o, m, out_dtype)
    err = np.abs(gpu - o)
    bad = ~(err <= tol)
    if np.any(bad):
        idx = np.argwhere(bad)[:5]
        detail = "; ".join(f"{tuple(i)}: gpu={gpu[tuple(i)]!r} oracle={o[tuple(i)]!r} tol={tol[tuple(i)]:.3g}"
                           for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; {detail}")
    return float(np.max(err / np.maximum(m, 1e-300)))
