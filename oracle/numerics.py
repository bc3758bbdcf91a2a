"""Scalar helpers of the oracle: activations, their derivatives, bf16 rounding.

Test infrastructure only (see the package docstring).
"""
from __future__ import annotations

import numpy as np

SQRT_2_OVER_PI = np.sqrt(2.0 / np.pi)
GELU_C = 0.044715


def gelu_tanh(x):
    """tanh-form GeLU, ``0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))``.

    The TP/SP page, section "MLP:先 column,再 row", applies "GeLU" elementwise to
    each shard's columns; the tanh form is the one the toy MLP workload names.
    """
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(SQRT_2_OVER_PI * (x + GELU_C * x ** 3)))


def gelu_tanh_grad(x):
    """d/dx of :func:`gelu_tanh`, by the product and chain rules."""
    x = np.asarray(x, dtype=np.float64)
    u = SQRT_2_OVER_PI * (x + GELU_C * x ** 3)
    th = np.tanh(u)
    du = SQRT_2_OVER_PI * (1.0 + 3.0 * GELU_C * x ** 2)
    return 0.5 * (1.0 + th) + 0.5 * x * (1.0 - th * th) * du


def sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-x))


def silu(x):
    """``x * sigmoid(x)``; SwiGLU's gate nonlinearity (TP/SP page, "MLP:先 column,再 row",
    the Qwen3 SwiGLU bullet: gate and up are both column-split, multiplied elementwise)."""
    x = np.asarray(x, dtype=np.float64)
    return x * sigmoid(x)


def silu_grad(x):
    """d/dx of :func:`silu` = ``s (1 + x (1 - s))`` with ``s = sigmoid(x)``."""
    x = np.asarray(x, dtype=np.float64)
    s = sigmoid(x)
    return s * (1.0 + x * (1.0 - s))


def round_to_bf16(x) -> np.ndarray:
    """Round float32 values to the nearest bfloat16, ties to even, returned as float32.

    bfloat16 keeps the top 16 bits of an IEEE binary32.  Round-to-nearest-even on
    the 16 dropped bits: add ``0x7FFF`` plus the lowest kept bit, then truncate.
    NaN stays NaN (quiet); infinities and overflow to infinity follow from the
    same integer arithmetic.
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = ((bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    out = (rounded & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)
    nan = np.isnan(f)
    if nan.any():
        out = out.copy()
        out[nan] = np.float32(np.nan)
    return out

