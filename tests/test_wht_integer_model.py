"""Host model of the decode-size Walsh-Hadamard rotation's integer path (CPU only).

The kernel takes a row through int64 butterflies when every nonzero element is a normal bf16
of biased exponent E >= 9 and the row spans fewer than 32 binades: x_j = I_j 2^(emin - 134)
with I_j = +-M_j << (E_j - emin), M_j the 8-bit significand.  This checks the arithmetic
facts that path rests on, with exact rationals: the integers represent the row exactly, every
partial sum of the seven butterfly stages stays below 2^46 (so int64 never overflows and the
sums are exact), the pair (RN_f32(S), S - RN_f32(S)) holds S exactly, and the scale
2^(emin - 134) is a normal float32 -- so the product with 1/sqrt(128) and the rounding decision
start from S itself, as in the double-float path for rows where that one is exact.
"""

from fractions import Fraction

import numpy as np

import synth


def _row_ints(bits):
    """(I_j list, emin) of a row of bf16 bit patterns, or None when the integer path is not taken."""
    e = [(int(b) >> 7) & 0xFF for b in bits]
    nz = [(int(b) & 0x7FFF) != 0 for b in bits]
    es = [max(x, 1) for x, z in zip(e, nz) if z]
    if not es:
        return [0] * len(bits), 255
    emax, emin = max(es), min(es)
    if not (emax < emin + 32 and emin >= 9 and emax < 255):     # 255: Inf / NaN
        return None
    ints = []
    for b, E, z in zip(bits, e, nz):
        if not z:
            ints.append(0)
            continue
        mag = ((int(b) & 0x7F) | 0x80) << (E - emin)
        ints.append(-mag if int(b) & 0x8000 else mag)
    return ints, emin


def _butterflies(v):
    """Sylvester-order Walsh-Hadamard sums, recording the largest partial-sum magnitude."""
    v = list(v)
    n = len(v)
    top = max(abs(x) for x in v)
    h = 1
    while h < n:
        for i in range(0, n, 2 * h):
            for j in range(i, i + h):
                a, b = v[j], v[j + h]
                v[j], v[j + h] = a + b, a - b
                top = max(top, abs(a + b), abs(a - b))
        h *= 2
    return v, top


def _rows(rng, n):
    out = []
    for k in range(n):
        span = int(rng.integers(0, 32))
        base = int(rng.integers(-110, 95))
        x = rng.standard_normal(128) * np.exp2(base + rng.uniform(0, span, 128))
        x[rng.random(128) < 0.1] = 0.0
        if k % 7 == 0:                                  # the widest span the path accepts
            x[0], x[1] = 2.0 ** base, 1.99 * 2.0 ** (base + 31)
        out.append(synth.f32_to_bf16_bits(x.astype(np.float32)))
    return out


def test_integer_path_is_exact():
    rng = np.random.default_rng(77)
    taken = 0
    for bits in _rows(rng, 60):
        r = _row_ints(bits)
        if r is None:
            continue
        taken += 1
        ints, emin = r
        vals = synth.bf16_bits_to_f32(bits).astype(np.float64)
        scale = Fraction(2) ** (emin - 134)
        assert all(Fraction(i) * scale == Fraction(float(v)) for i, v in zip(ints, vals))
        assert max(abs(i) for i in ints) < 2 ** 39
        sums, top = _butterflies(ints)
        assert top < 2 ** 46
        for s in sums:
            hi = np.float32(s)                           # round to nearest
            lo = np.float32(s - int(hi))
            assert Fraction(int(hi)) + Fraction(float(lo)) == s
        assert -126 <= emin - 134 <= 127                 # 2^(emin - 134) is a normal float32
    assert taken >= 40


def test_rows_outside_the_path_are_refused():
    # a subnormal-range element (E < 9) or a span of 32 binades sends the row to the bounded path
    small = synth.f32_to_bf16_bits(np.array([2.0 ** -120] + [1.0] * 127, np.float32))
    wide = synth.f32_to_bf16_bits(np.array([1.0, 2.0 ** 32] + [0.0] * 126, np.float32))
    inf = synth.f32_to_bf16_bits(np.array([np.inf, 2.0 ** 120] + [0.0] * 126, np.float32))
    assert _row_ints(small) is None and _row_ints(wide) is None and _row_ints(inf) is None
    zero = np.zeros(128, np.uint16)
    assert _row_ints(zero) == ([0] * 128, 255)
