"""Per-head transforms applied on write (keys, values) and on read (queries).

Oracle module (test infrastructure only).

* Keys are transformed online, k' = T_K k, after RoPE; queries are compensated
  so that the logits are unchanged ([WUSH] "核心方法" and "方法步骤详情";
  [OSCAR] section 3 "Online Deployment").  For any invertible T the
  compensation is q' = T^{-T} q, because (T^{-T} q)^T (T k) = q^T T^{-1} T k
  = q^T k; for orthogonal T, T^{-T} = T ([OScaR] "Hadamard 变换简介",
  inner-product preservation).  The caller supplies T^{-T}.
* Values get T_V (or nothing, when T_V is folded into the projection weights,
  [OScaR] "步骤一" fusion note; [WUSH] value-side folding).
* The Hadamard path uses the normalised Walsh-Hadamard matrix, entries
  +-1/sqrt(d), H H^T = I ([OScaR] "Hadamard 变换简介" and "步骤一：Canalized
  Rotation"; [OSCAR] appendix A.1).

Every transformed row is the exact product rounded once to bfloat16 (the cache
stores BF16 rows).  Products of a float32 matrix entry and a bfloat16 input are
exact in float64 and the float64 sum of d = 128 of them is accurate to about
2^-46 relative, so one final rounding gives the correctly rounded row except
when the exact value lies within that distance of a rounding midpoint.
"""

from __future__ import annotations

import numpy as np

from .fp import bf16_to_f32, round_f64_to_bf16


def hadamard(d: int) -> np.ndarray:
    """Normalised Sylvester-Hadamard matrix, float64 [d, d] (d a power of two)."""
    if d < 1 or d & (d - 1):
        raise ValueError("Hadamard size must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h / np.sqrt(d)


def fwht(x: np.ndarray) -> np.ndarray:
    """Fast Walsh-Hadamard transform along the last axis in float64, normalised by 1/sqrt(d).

    O(d log d) butterflies (a + b, a - b) at strides 1, 2, 4, ..., d/2.
    """
    y = np.array(x, dtype=np.float64, copy=True)
    d = y.shape[-1]
    if d & (d - 1):
        raise ValueError("Hadamard size must be a power of two")
    h = 1
    while h < d:
        y = y.reshape(*y.shape[:-1], d // (2 * h), 2, h)
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        y = y.reshape(*y.shape[:-3], d)
        h *= 2
    return y / np.sqrt(d)


def apply_f64(t: np.ndarray, x: np.ndarray) -> np.ndarray:
    """x' = T x for every row of x (x [..., d] real values, T [d, d]); float64 result."""
    return np.asarray(x, np.float64) @ np.asarray(t, np.float64).T


def rotate_rows(t: np.ndarray | None, x_bits: np.ndarray, kind: str = "dense") -> np.ndarray:
    """Transformed rows rounded once to bfloat16 (returned as float32 values).

    kind "dense": T x with T float32 [d, d] (T None means identity: rows pass unchanged).
    kind "hadamard": H x with the normalised Walsh-Hadamard matrix.
    """
    x = bf16_to_f32(x_bits).astype(np.float64)
    if kind == "hadamard":
        y = apply_f64(hadamard(x.shape[-1]), x)
    elif t is None:
        y = x
    else:
        y = apply_f64(t, x)
    return round_f64_to_bf16(y)
