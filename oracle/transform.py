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
stores BF16 rows).  The float64 product (y = T x, or the +-1 Walsh-Hadamard sum S
times 1/sqrt(d)) comes with the standard error bound of a d-term dot product,
gamma_d sum |T_ij x_j|; wherever that interval does not lie inside one bfloat16
rounding cell -- a value near a rounding midpoint, or an exact cancellation, where
the float64 noise is not even of the right sign -- the element is recomputed in
exact rational arithmetic (fractions.Fraction) and rounded from there.  An exact
zero is +0.
"""

from __future__ import annotations

from fractions import Fraction

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


def _gamma(n: int) -> float:
    """gamma_n = n u / (1 - n u), u = 2^-53: |fl(sum of n products) - exact| <= gamma_n sum |products|
    for float64 dot products in any summation order (products of these inputs are exact)."""
    u = 2.0 ** -53
    return n * u / (1.0 - n * u)


def _bf16_cell(b: np.ndarray):
    """(lo, hi): the midpoints between each bfloat16 value b (float64 array) and its neighbours;
    values strictly inside (lo, hi) round to b."""
    mag = np.abs(b).astype(np.float32).view(np.uint32).astype(np.int64)
    up = ((mag + 0x10000) << 0).astype(np.uint32).view(np.float32).astype(np.float64)
    dn = np.where(mag > 0, np.maximum(mag - 0x10000, 0), 0x10000).astype(np.uint32).view(np.float32).astype(np.float64)
    dn = np.where(mag > 0, dn, -dn)                       # below +0: the negative smallest value
    lo_nb = np.where(b >= 0, dn, -up)
    hi_nb = np.where(b >= 0, up, np.where(mag > 0, -dn, -lo_nb))
    return (lo_nb + b) / 2.0, (b + hi_nb) / 2.0


def _bf16_candidates(est: float):
    """bfloat16 values around a float64 estimate (the nearest and its two neighbours), ascending."""
    b0 = float(round_f64_to_bf16(np.array([est]))[0])
    lo, hi = _bf16_cell(np.array([b0]))
    return [2.0 * float(lo[0]) - b0, b0, 2.0 * float(hi[0]) - b0]


def _even_bf16(v: float) -> bool:
    return (int(np.array([v], np.float32).view(np.uint32)[0] >> 16) & 1) == 0


def _round_exact_dyadic(S: Fraction) -> float:
    """Nearest bfloat16 (ties to even) of an exact rational S; +0 for S = 0."""
    if S == 0:
        return 0.0
    best = None
    for c in _bf16_candidates(float(S)):
        dist = abs(S - Fraction(c))
        if best is None or dist < best[0] or (dist == best[0] and _even_bf16(c)):
            best = (dist, c)
    return best[1]


def _round_exact_over_sqrt(S: Fraction, d: int) -> float:
    """Nearest bfloat16 of S / sqrt(d) (d not a square: the value is irrational unless S = 0,
    so there are no ties); compared through squares of exact rationals."""
    if S == 0:
        return 0.0
    mag2 = S * S / d                                      # |y|^2, exact
    cands = [abs(c) for c in _bf16_candidates(abs(float(S)) / np.sqrt(d))]
    cands = sorted(set(cands))
    pick = cands[0]
    for a, b in zip(cands, cands[1:]):
        m = (Fraction(a) + Fraction(b)) / 2
        if mag2 > m * m:
            pick = b
    return pick if S > 0 else -pick


def rotate_rows(t: np.ndarray | None, x_bits: np.ndarray, kind: str = "dense") -> np.ndarray:
    """Transformed rows rounded once to bfloat16 (returned as float32 values).

    kind "dense": T x with T float32 [d, d] (T None means identity: rows pass unchanged).
    kind "hadamard": H x with the normalised Walsh-Hadamard matrix.
    """
    x = bf16_to_f32(x_bits).astype(np.float64)
    if kind != "hadamard" and t is None:
        return round_f64_to_bf16(x)
    d = x.shape[-1]
    if kind == "hadamard":
        hint = np.rint(hadamard(d) * np.sqrt(d))          # the +-1 Sylvester matrix (exact)
        S = x @ hint.T
        a = np.abs(x).sum(axis=-1, keepdims=True) * np.ones_like(S)
        c = 1.0 / np.sqrt(d)
        y = S * c
        # S within gamma_d a; c and the product each one float64 rounding
        err = (_gamma(d) * a * c + np.abs(y) * 2.0 ** -51) * (1 + 2.0 ** -40)
    else:
        t64 = np.asarray(t, np.float64)
        y = x @ t64.T
        err = _gamma(d) * (np.abs(x) @ np.abs(t64).T) * (1 + 2.0 ** -40)
    out = round_f64_to_bf16(y)
    lo, hi = _bf16_cell(out.astype(np.float64))
    undecided = ~((y - err > lo) & (y + err < hi))
    if np.any(undecided):
        x2 = x.reshape(-1, d)
        flat_out = out.reshape(-1, d)
        for r, i in zip(*np.nonzero(undecided.reshape(-1, d))):
            xs = [Fraction(float(v)) for v in x2[r]]
            if kind == "hadamard":
                S_ex = sum(xs[j] if hint[i, j] > 0 else -xs[j] for j in range(d))
                flat_out[r, i] = _round_exact_over_sqrt(S_ex, d)
            else:
                S_ex = sum(Fraction(float(t64[i, j])) * xs[j] for j in range(d) if t64[i, j] != 0)
                flat_out[r, i] = _round_exact_dyadic(S_ex)
        out = flat_out.reshape(out.shape)
    return np.where(out == 0, np.float32(0.0), out)    # an exact zero is +0
