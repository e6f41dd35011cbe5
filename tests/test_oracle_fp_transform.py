"""Pins of the oracle's rounding helpers and transforms (CPU only).

Each check is pinned to something other than the oracle itself: exact
rational arithmetic, scipy's Hadamard matrix, and the algebraic invariants
the pages state for the key/query transform.
"""

import math
from fractions import Fraction

import numpy as np
import pytest
import scipy.linalg

import synth
from oracle import fp, transform


# ---- rounding: brute force "nearest representable value, ties to even" -----------------
def _nearest_by_enumeration(xq, fmt: str) -> float:
    """Nearest bfloat16 / float16 to the exact value xq (float or Fraction), found by
    enumerating the bit patterns around it and comparing exact distances."""
    x = float(xq)
    if fmt == "bf16":
        t = np.float32(x).view(np.uint32) >> 16
        cands = [int(t) + k for k in (-2, -1, 0, 1, 2)]
        vals = [float((np.uint32(c & 0xFFFF) << np.uint32(16)).view(np.float32)) for c in cands if 0 <= c <= 0xFFFF]
        pats = [c & 0xFFFF for c in cands if 0 <= c <= 0xFFFF]
    else:
        t = int(np.float16(x).view(np.uint16))
        pats = [t + k for k in (-2, -1, 0, 1, 2) if 0 <= t + k <= 0xFFFF]
        vals = [float(np.uint16(p).view(np.float16)) for p in pats]
    best = None
    fx = Fraction(xq)
    for v, p in zip(vals, pats):
        if not math.isfinite(v):
            continue
        dist = abs(Fraction(v) - fx)
        key = (dist, p & 1)  # ties: even mantissa LSB wins
        if best is None or key < best[0]:
            best = (key, v)
    return best[1]


def test_bf16_rounding_matches_enumeration():
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000),
        rng.standard_normal(300) * 1e-39,                       # bf16 subnormal range
    ])
    # exact midpoints between adjacent bfloat16 values (ties)
    base = fp.bf16_to_f32(rng.integers(0x0080, 0x7F00, 500).astype(np.uint16)).astype(np.float64)
    nxt = fp.bf16_to_f32((fp.f32_to_bf16_bits(base.astype(np.float32)) + 1).astype(np.uint16)).astype(np.float64)
    x = np.concatenate([x, (base + nxt) / 2, -(base + nxt) / 2])
    got = fp.round_f64_to_bf16(x).astype(np.float64)
    for xi, gi in zip(x, got):
        assert gi == _nearest_by_enumeration(float(xi), "bf16"), xi


def test_bf16_overflow_and_zero():
    assert np.isinf(fp.round_f64_to_bf16(np.array([3.4e38]))[0])
    assert fp.round_f64_to_bf16(np.array([0.0]))[0] == 0.0
    assert np.signbit(fp.round_f64_to_bf16(np.array([-0.0]))[0])


def test_f16_conversion_matches_enumeration():
    rng = np.random.default_rng(12)
    x = rng.standard_normal(3000) * 10.0 ** rng.integers(-8, 5, 3000)
    got64 = fp.to_f16(x).astype(np.float64)
    for xi, gi in zip(x, got64):
        if abs(xi) < 65504:
            assert gi == _nearest_by_enumeration(float(xi), "f16"), xi


# ---- transforms ------------------------------------------------------------------------
@pytest.mark.parametrize("d", [4, 32, 128])
def test_hadamard_is_scipy_sylvester(d):
    h = transform.hadamard(d)
    ref = scipy.linalg.hadamard(d) / math.sqrt(d)
    assert np.array_equal(h, ref)
    assert np.allclose(h @ h.T, np.eye(d), atol=1e-14)
    assert np.all(np.isclose(np.abs(h), 1 / math.sqrt(d)))


def test_fast_hadamard_equals_dense():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((50, 128))
    ref = x @ (scipy.linalg.hadamard(128) / math.sqrt(128)).T
    assert np.allclose(transform.fwht(x), ref, atol=1e-12)


def _qk_invariant_error(t, t_q, rng, n=64):
    d = t.shape[0]
    q = rng.standard_normal((n, d))
    k = rng.standard_normal((n, d))
    lhs = np.sum(transform.apply_f64(t_q, q) * transform.apply_f64(t, k), axis=1)
    rhs = np.sum(q * k, axis=1)
    return np.max(np.abs(lhs - rhs) / (np.linalg.norm(q, axis=1) * np.linalg.norm(k, axis=1)))


def test_orthogonal_transform_preserves_logits():
    rng = np.random.default_rng(4)
    t = synth.random_orthogonal(128, rng)
    assert _qk_invariant_error(t, t, rng) < 1e-12
    h = transform.hadamard(128)
    assert _qk_invariant_error(h, h, rng) < 1e-12


def test_invertible_transform_compensation():
    rng = np.random.default_rng(5)
    t = synth.spd_invertible(128, rng, 100.0)
    tit = np.linalg.inv(t).T
    # T^T T^{-T} = I
    assert np.max(np.abs(t.T @ tit - np.eye(128))) < 1e-10
    assert _qk_invariant_error(t, tit, rng) < 1e-10
    # planted mistake: compensating queries with T itself (right only for orthogonal T) is caught
    assert _qk_invariant_error(t, t, rng) > 1e-3


def test_rotate_rows_is_exact_product_rounded_once():
    rng = np.random.default_rng(6)
    d = 16
    t = rng.standard_normal((d, d)).astype(np.float32)
    x_bits = synth.f32_to_bf16_bits(rng.standard_normal((8, d)).astype(np.float32))
    got = transform.rotate_rows(t, x_bits)
    x = fp.bf16_to_f32(x_bits)
    for r in range(8):
        for i in range(d):
            exact = sum(Fraction(float(t[i, j])) * Fraction(float(x[r, j])) for j in range(d))
            assert float(got[r, i]) == _nearest_by_enumeration(exact, "bf16")


def test_rotate_identity_is_exact():
    rng = np.random.default_rng(7)
    x_bits = synth.f32_to_bf16_bits(rng.standard_normal((10, 128)).astype(np.float32))
    assert np.array_equal(fp.f32_to_bf16_bits(transform.rotate_rows(None, x_bits)), x_bits)
    eye = np.eye(128, dtype=np.float32)
    assert np.array_equal(fp.f32_to_bf16_bits(transform.rotate_rows(eye, x_bits)), x_bits)


def test_generator_transforms_inverse_transpose():
    w = synth.WUSH_CHUNK_B16
    tk, tkit, tv = synth.transforms(w)
    for h in range(2):
        e = tk[h].astype(np.float64).T @ tkit[h].astype(np.float64) - np.eye(128)
        assert np.max(np.abs(e)) < 1e-5          # float32-rounded T^{-T} of the float32 T


def _nearest_bf16_decimal(y) -> float:
    """Nearest bfloat16 to a high-precision Decimal y (no ties occur for irrational values),
    by enumerating the bit patterns around it."""
    import decimal
    t = int(np.float32(float(y)).view(np.uint32) >> 16)
    best = None
    for c in (t - 2, t - 1, t, t + 1, t + 2):
        if not 0 <= c <= 0xFFFF:
            continue
        v = float((np.uint32(c) << np.uint32(16)).view(np.float32))
        if not math.isfinite(v):
            continue
        dist = abs(decimal.Decimal(v) - y)
        if best is None or dist < best[0]:
            best = (dist, v)
    return best[1]


def test_hadamard_rows_exact_cancellation_and_rounding():
    """Rows whose Walsh-Hadamard sums cancel exactly (a constant row; small-integer rows) give
    +0 there -- float64 summation noise must not survive as a tiny bfloat16 -- and every other
    output is the nearest bfloat16 of S / sqrt(128), checked with 60-digit decimals."""
    import decimal
    decimal.getcontext().prec = 60
    rng = np.random.default_rng(11)
    rows = [np.full(128, 1.25)]
    rows += [rng.choice([-2.0, -1.0, 1.0, 2.0], 128) for _ in range(3)]
    rows += [rng.standard_normal(128) * 2.0 ** rng.integers(-30, 10) for _ in range(2)]
    x_bits = synth.f32_to_bf16_bits(np.array(rows, np.float32))
    got = transform.rotate_rows(None, x_bits, "hadamard")
    x = fp.bf16_to_f32(x_bits).astype(np.float64)
    sign = scipy.linalg.hadamard(128)
    root = decimal.Decimal(128).sqrt()
    zeros = 0
    for r in range(len(rows)):
        for i in range(128):
            S = sum(decimal.Decimal(float(x[r, j])) * int(sign[i, j]) for j in range(128))
            if S == 0:
                zeros += 1
                assert fp.f32_to_bf16_bits(got[r:r + 1, i:i + 1])[0, 0] == 0, (r, i)
            else:
                assert float(got[r, i]) == _nearest_bf16_decimal(S / root), (r, i)
    assert zeros > 127          # the constant row alone contributes 127


def test_dense_rows_exact_cancellation():
    """A dense row that cancels exactly (T_i = (x_1, -x_0, 0, ...)) gives +0, also when the row
    shares the batch with large rows (float64 blocking must not leak noise into it)."""
    rng = np.random.default_rng(12)
    x_bits = synth.f32_to_bf16_bits(rng.standard_normal((5, 128)).astype(np.float32) * 100)
    x = fp.bf16_to_f32(x_bits)
    t = rng.standard_normal((128, 128)).astype(np.float32)
    t[7] = 0.0
    t[7, 0], t[7, 1] = x[2, 1], -x[2, 0]
    got = transform.rotate_rows(t, x_bits)
    assert fp.f32_to_bf16_bits(got[2:3, 7:8])[0, 0] == 0
    for i in (0, 7, 100):
        exact = sum(Fraction(float(t[i, j])) * Fraction(float(x[2, j])) for j in range(128))
        assert float(got[2, i]) == _nearest_by_enumeration(exact, "bf16")
