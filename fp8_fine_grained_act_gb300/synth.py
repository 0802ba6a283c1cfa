"""Seeded synthetic inputs shaped like the workloads of fine-grained FP8
training.  Shared by the tests, the benchmark and the smoke check; holds no
quantization or GEMM arithmetic (only random draws and the BF16 rounding of
the drawn FP32 values, which is how a BF16 activation tensor is produced).

Distributions (the pages give the structure -- 4K-token sequences,
activation outliers, token-correlated gradient outliers, MoE routing --
but no parameters; the numbers below are this library's choice):
  * activations X ~ N(0, 1) with outliers, because fine-grained groups exist
    to contain activation outliers (DeepSeek-V3 FP8 post on innerforce.co.kr,
    fine-grained quantization paragraph): either a random 0.1 % of entries
    x100, or 8 fixed channels x50 for every token;
  * output gradients dY with token-correlated outliers ("DeepSeek FP8
    Training", arcalunar.github.io, closing paragraph on grouping sizes):
    row i is N(0, 1) * exp(N(0, 2)) with one factor per row;
  * FP32 master weights ~ N(0, 0.02^2);
  * MoE token counts: Dirichlet(1) expert probabilities, multinomial counts,
    each group padded with zero rows to a multiple of 128.

N(mu, v) names the variance, so N(0, 2) has standard deviation sqrt(2).
All draws use numpy's PCG64 ``default_rng(seed)``; a configuration's draw
order is part of its definition.
"""
from __future__ import annotations

import numpy as np

GROUP = 128


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round FP32 values to BF16 (nearest, ties to even) and return the 16-bit
    patterns as uint16.  Inputs are finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact FP32 value of BF16 bit patterns."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def activations_random_outliers(rng, rows: int, cols: int, frac: float = 1e-3,
                                factor: float = 100.0) -> np.ndarray:
    """N(0,1) with round(frac*rows*cols) entries, chosen uniformly without
    replacement, multiplied by ``factor``.  Returns BF16 bits [rows, cols]."""
    x = rng.standard_normal((rows, cols), dtype=np.float32)
    n_out = int(round(frac * rows * cols))
    if n_out:
        pos = rng.choice(rows * cols, size=n_out, replace=False)
        x.reshape(-1)[pos] *= np.float32(factor)
    return f32_to_bf16_bits(x)


def activations_channel_outliers(rng, rows: int, cols: int, n_channels: int = 8,
                                 factor: float = 50.0) -> np.ndarray:
    """N(0,1) with ``n_channels`` fixed channels (the same for every token)
    multiplied by ``factor``.  Returns BF16 bits [rows, cols]."""
    ch = rng.choice(cols, size=min(n_channels, cols), replace=False)
    x = rng.standard_normal((rows, cols), dtype=np.float32)
    x[:, ch] *= np.float32(factor)
    return f32_to_bf16_bits(x)


def gradients_token_outliers(rng, rows: int, cols: int, log_var: float = 2.0) -> np.ndarray:
    """Row i = N(0,1) * exp(N(0, log_var)), one factor per row (token).
    Returns BF16 bits [rows, cols]."""
    f = np.exp(rng.standard_normal(rows) * np.sqrt(log_var)).astype(np.float32)
    x = rng.standard_normal((rows, cols), dtype=np.float32)
    x *= f[:, None]
    return f32_to_bf16_bits(x)


def master_weight(rng, rows: int, cols: int, std: float = 0.02) -> np.ndarray:
    """FP32 master weight ~ N(0, std^2), [rows, cols]."""
    w = rng.standard_normal((rows, cols), dtype=np.float32)
    w *= np.float32(std)
    return w


def moe_group_sizes(rng, n_experts: int = 64, n_tokens: int = 32768, pad: int = GROUP):
    """Expert probabilities ~ Dirichlet(1), token counts ~ Multinomial, each
    padded up to a multiple of ``pad``.  Returns (counts, padded, offsets)
    with offsets int32[G+1], the prefix sums of the padded counts."""
    p = rng.dirichlet(np.ones(n_experts))
    counts = rng.multinomial(n_tokens, p)
    padded = ((counts + pad - 1) // pad) * pad
    offsets = np.zeros(n_experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(padded)
    return counts.astype(np.int64), padded.astype(np.int64), offsets


def moe_tokens(rng, counts, padded, cols: int) -> np.ndarray:
    """Concatenated expert inputs: expert g has counts[g] rows of N(0,1)
    followed by padded[g]-counts[g] zero rows.  Returns BF16 bits
    [sum(padded), cols]."""
    total = int(np.sum(padded))
    x = np.zeros((total, cols), dtype=np.float32)
    r = 0
    for c, p in zip(counts, padded):
        c, p = int(c), int(p)
        x[r:r + c] = rng.standard_normal((c, cols), dtype=np.float32)
        r += p
    return f32_to_bf16_bits(x)


# ----------------------------------------------------------- workloads ---
# Each returns a dict of host numpy arrays.  Shapes default to the full
# workload; the tests pass smaller shapes with the same recipe.

def tiny_fprop(seed: int = 0, M: int = 256, N: int = 256, K: int = 512):
    """Tiny Fprop: X[M,K] N(0,1) with 0.1 % of entries x100, W[N,K] ~ N(0, 0.02^2)."""
    rng = np.random.default_rng(seed)
    x = activations_random_outliers(rng, M, K)
    w = master_weight(rng, N, K)
    return {"x": x, "w": w}


def fprop_linear(seed: int = 1, M: int = 4096, N: int = 18432, K: int = 7168):
    """Fprop linear: X[M,K] N(0,1) with 8 fixed channels x50 (one 4K-token
    sequence at full size), W[N,K] ~ N(0, 0.02^2)."""
    rng = np.random.default_rng(seed)
    x = activations_channel_outliers(rng, M, K)
    w = master_weight(rng, N, K)
    return {"x": x, "w": w}


def dgrad(seed: int = 2, M: int = 8192, N: int = 7168, K: int = 2048):
    """Dgrad: dY[M,K] with token-correlated outliers, W[K,N] master (the
    layer maps N inputs to K outputs); dX = dY . W is [M, N]."""
    rng = np.random.default_rng(seed)
    dy = gradients_token_outliers(rng, M, K)
    w = master_weight(rng, K, N)
    return {"dy": dy, "w": w}


def wgrad(seed: int = 3, T: int = 8192, N_out: int = 2048, K_in: int = 7168):
    """Wgrad: dY[T, N_out] with token-correlated outliers and X[T, K_in] with
    8 fixed outlier channels; dW = dY^T . X is [N_out, K_in]."""
    rng = np.random.default_rng(seed)
    dy = gradients_token_outliers(rng, T, N_out)
    x = activations_channel_outliers(rng, T, K_in)
    return {"dy": dy, "x": x}


def grouped_moe(seed: int = 4, n_experts: int = 64, n_tokens: int = 32768,
                N: int = 2048, K: int = 7168, with_weights: bool = True):
    """Grouped MoE Fprop: Dirichlet(1)/multinomial token counts padded to 128,
    X_all[M_total, K] N(0,1) with zero pad rows, W_g[G, N, K] ~ N(0, 0.02^2)."""
    rng = np.random.default_rng(seed)
    counts, padded, offsets = moe_group_sizes(rng, n_experts, n_tokens)
    x = moe_tokens(rng, counts, padded, K)
    out = {"x": x, "counts": counts, "padded": padded, "offsets": offsets}
    if with_weights:
        w = np.empty((n_experts, N, K), dtype=np.float32)
        for g in range(n_experts):
            w[g] = master_weight(rng, N, K)
        out["w"] = w
    return out


__all__ = [
    "f32_to_bf16_bits", "bf16_bits_to_f32", "activations_random_outliers",
    "activations_channel_outliers", "gradients_token_outliers", "master_weight",
    "moe_group_sizes", "moe_tokens", "tiny_fprop", "fprop_linear", "dgrad", "wgrad",
    "grouped_moe",
]
