"""Decode linear layer y = x W^T (oracle).

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only the tests, the smoke check
and the benchmark's CPU-baseline leg may import or call this module. It shares
no code with the CUDA library and imports nothing from it.

"ninfer" issue 80 (Proposal: opt-in fixed decode width): every GEMM-class
decode op computes, for each token row t of the activations, y[t, n] =
sum_k x[t, k] W[n, k]; running it at a fixed padded width only changes which
kernel computes it, never the value it stands for, and rows never mix. The
oracle is that definition in float64, bf16 inputs widened exactly (raw uint16
bit patterns, the upper half of an IEEE binary32).
"""
from __future__ import annotations

import numpy as np


def widen_bf16(bits) -> np.ndarray:
    b = np.asarray(bits)
    if b.dtype != np.uint16:
        raise TypeError("bf16 data must be carried as uint16 bit patterns")
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def linear(x_bits, w_bits) -> np.ndarray:
    """float64 [T, N]: y[t, n] = sum_k x[t, k] w[n, k] for x [T, K], w [N, K]."""
    x = widen_bf16(x_bits)
    w = widen_bf16(w_bits)
    if x.shape[1] != w.shape[1]:
        raise ValueError("x [T, K] and w [N, K] must share K")
    return x @ w.T


def abs_sum(x_bits, w_bits) -> np.ndarray:
    """float64 [T, N]: sum_k |x[t, k] w[n, k]| (for rounding-error bounds)."""
    return np.abs(widen_bf16(x_bits)) @ np.abs(widen_bf16(w_bits)).T
