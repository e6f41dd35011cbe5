"""Floating-point formats used by the cache: bfloat16 rows, float16 scales.

Oracle module (test infrastructure only).  The pages store BF16 windows and
staging rows ([OSCAR] section 4 "KV Cache Layout"; [WUSH] "方法步骤详情") and
16-bit scale factors ([OScaR] "内存布局"); rounding is to nearest, ties to even.
"""

from __future__ import annotations

import numpy as np

BF16_MAX = float(np.float32(3.3895313892515355e38))  # 0x7F7F


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 values that are exactly representable in bfloat16 -> bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return (u >> 16).astype(np.uint16)


def round_f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bfloat16 in ONE rounding step (nearest, ties to even).

    Returned as float32 (every bfloat16 value is a float32).  |x| = m 2^e with
    m in [0.5, 1); a bfloat16 keeps 8 significant bits, so the spacing is
    2^(e-8) for normal values and 2^-133 below the smallest normal 2^-126.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    _, e = np.frexp(ax)
    e = np.maximum(e, -125)
    q = np.rint(np.ldexp(ax, 8 - e))          # exact scaling, then integer rounding (half-even)
    y = np.ldexp(q, e - 8)
    y = np.where(y > BF16_MAX, np.inf, y)
    y = np.where(np.isnan(x), np.nan, y)
    return np.copysign(y, x).astype(np.float32)


def round_f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    return f32_to_bf16_bits(round_f64_to_bf16(x))


def to_f16(x: np.ndarray) -> np.ndarray:
    """Round float32 or float64 values to float16 (numpy converts in one step, nearest-even)."""
    return np.asarray(x).astype(np.float16)
