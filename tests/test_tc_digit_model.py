"""A host model of the arithmetic the tensor-core rotation uses (fixed-point digits, exact
integer level sums, the fp32 combination, the bound and the one-midpoint decision), checked
against exact rationals on random and adversarial rows.  It pins the bound's derivation --
what the kernel decides must be the correctly rounded result -- on far more inputs than the
device tests can, with the inputs the bound is most likely to miss: extreme digits, rows
spanning many binades, heavy cancellation, subnormal entries.

The model follows the kernel step for step in IEEE fp32: the digit steps and the combination
of the level sums are exact in float64 before their one rounding to fp32, so numpy reproduces
the kernel's fused operations there bit for bit (the bound's own fused multiply-add may differ
in its last bit).  It shares no code with the oracle and is compared with it."""

from fractions import Fraction

import numpy as np
import pytest

import synth
from oracle import transform

F32 = np.float32
BOUND_CONST = float(np.float32(float.fromhex("0x1.9p-10")))
REL = float(np.float32(float.fromhex("0x1.81p-23")))


def _f32(x) -> np.ndarray:
    return np.asarray(x, np.float64).astype(F32)


def _exp_field(a: np.ndarray) -> np.ndarray:
    """Largest exponent field (at least 1) of each row of float32 values."""
    e = (a.view(np.uint32) >> 23) & 0xFF
    return np.maximum(e.max(axis=-1), 1).astype(np.int64)


def _digits(x: np.ndarray, k: np.ndarray, n: int):
    """x * 2^k (rounded to fp32 like the kernel's power-of-two scaling) split into n balanced
    base-256 digits by round-to-nearest steps: returns the digits, the rest after them (scaled
    by 2^(8n)) and the scaled values."""
    scaled = _f32(x.astype(np.float64) * np.exp2(k.astype(np.float64))[..., None])
    r = scaled
    out = []
    for _ in range(n):
        d = np.rint(r)                             # float32 rint (ties to even)
        out.append(d.astype(np.float64))
        r = _f32((r.astype(np.float64) - d) * 256.0)
    return out, r.astype(np.float64), scaled


def model_rotate(t: np.ndarray, x_bits: np.ndarray):
    """(bits, decided) of y = T x per the tensor-core path for rows x (bf16 bits [R, 128])."""
    t = np.asarray(t, F32)
    x = (x_bits.astype(np.uint32) << 16).view(F32)
    e = _exp_field(t)                               # per output i
    f = _exp_field(x)                               # per row r
    td, _, t_units = _digits(t, 133 - e, 4)
    xd, xrest, x_units = _digits(x, 133 - f, 3)
    lossy = ((xrest != 0) | ((x_units == 0) & (x != 0))).any(axis=-1)
    # 2^-16 sum_j |T_ij| / U_i (X's truncation bound for lossy rows)
    st16 = _f32(_f32(np.abs(t_units.astype(np.float64)).sum(axis=-1)) * float.fromhex("0x1.01p-16"))
    # exact integer level sums D_L[r, i] = sum_{a+b=L} sum_j x_a[r, j] t_b[i, j]
    levels = np.zeros((4,) + (x.shape[0], t.shape[0]))
    for a in range(3):
        for b in range(4):
            if a + b <= 3:
                prod = xd[a] @ td[b].T
                assert np.abs(prod).max() < 2.0 ** 22
                levels[a + b] += prod
    assert np.abs(levels).max() < 2.0 ** 23
    # fp32 combination: each fused step is exact in float64 before its one rounding
    v = _f32(levels[0] + levels[1] * 2.0 ** -8)
    v = _f32(v.astype(np.float64) + levels[2] * 2.0 ** -16)
    v = _f32(v.astype(np.float64) + levels[3] * 2.0 ** -24)
    c = np.where(lossy[:, None], _f32(BOUND_CONST + st16[None, :].astype(np.float64)), F32(BOUND_CONST))
    bnd = _f32(np.abs(v.astype(np.float64)) * REL + c.astype(np.float64))
    vb = v.view(np.uint32)
    mid = ((vb & 0xFFFF0000) | 0x8000).astype(np.uint32).view(F32)
    decided = (np.abs(v.astype(np.float64) - mid.astype(np.float64)) > bnd) & \
              (bnd.astype(np.float64) * 1024.0 < np.abs(v.astype(np.float64)))
    # RN bf16 of v, then the exponent shift by S = e_i + f_r - 266
    bu = ((vb + 0x7FFF + ((vb >> 16) & 1)) >> 16).astype(np.int64)
    eu = (bu >> 7) & 0xFF
    s = e[None, :] + f[:, None] - 266
    ey = eu + s
    ok = decided & (eu > 0) & (ey >= 1) & (ey <= 254)
    bits = np.where(ok, bu + s * 128, -1)
    return bits, ok, v, bnd, levels, (e, f)


def _exact_units(t, x_bits, e, f, r, i):
    """y[r, i] / (U_i V_r) exactly."""
    x = (x_bits.astype(np.uint32) << 16).view(F32)
    s = sum(Fraction(float(t[i, j])) * Fraction(float(x[r, j])) for j in range(t.shape[1]))
    return s * Fraction(2) ** int(266 - e[i] - f[r])


def _check(t, x_bits, n_exact=300, seed=0):
    bits, ok, v, bnd, _, (e, f) = model_rotate(t, x_bits)
    ref = synth.f32_to_bf16_bits(transform.rotate_rows(t, x_bits))
    got = bits.astype(np.int64)
    # every decided output is the correctly rounded one
    assert np.array_equal(got[ok], ref.astype(np.int64)[ok])
    # the bound holds on a sample (exact rationals)
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, v.size, size=min(n_exact, v.size))
    for flat in idx:
        r, i = divmod(int(flat), v.shape[1])
        if not np.isfinite(v[r, i]):
            continue
        err = abs(_exact_units(t, x_bits, e, f, r, i) - Fraction(float(v[r, i])))
        assert err <= Fraction(float(bnd[r, i])), (r, i, float(err), float(bnd[r, i]))
    return ok.mean()


def _rows(rng, n, wide=False, outliers=False):
    x = rng.standard_normal((n, 128))
    if outliers:
        x[:, [3, 77]] *= 15.0
    if wide:
        x = x * np.exp2(rng.integers(-40, 41, size=(n, 1))) * np.exp2(rng.integers(-12, 13, size=(n, 128)))
    return synth.f32_to_bf16_bits(x.astype(np.float32))


def test_wush_invertible_matrix_key_rows():
    w = synth.WUSH_CHUNK_B16
    tk, _, _ = synth.transforms(w)
    rng = np.random.default_rng(1)
    frac = _check(tk[0], _rows(rng, 96, outliers=True))
    assert frac > 0.99


def test_orthogonal_matrix_wide_rows():
    tk, _, _ = synth.transforms(synth.QWEN3_8B_32K)
    rng = np.random.default_rng(2)
    _check(tk[3], _rows(rng, 96, wide=True), seed=2)


@pytest.mark.parametrize("signs", ["random", "aligned"])
def test_extreme_digits(signs):
    """Entries at the top of their binade (1.9921875 = 127.5 units: digits 128 and -128): the
    level sums reach their magnitude limit when every sign agrees."""
    rng = np.random.default_rng(3)
    v = np.float32(1.9921875)
    if signs == "random":
        t = (v * np.where(rng.random((128, 128)) < 0.5, -1, 1)).astype(np.float32)
        x = (v * np.where(rng.random((64, 128)) < 0.5, -1, 1)).astype(np.float32)
    else:
        t = np.full((128, 128), v, np.float32)
        x = np.full((64, 128), v, np.float32)
    xb = synth.f32_to_bf16_bits(x)
    _, _, _, _, levels, _ = model_rotate(t, xb)
    assert np.abs(levels).max() < 2.0 ** 23
    if signs == "aligned":
        assert np.abs(levels).max() >= 2.0 ** 22      # the extreme case is reached
    _check(t, xb, seed=3)


def test_cancellation_and_small_results():
    """Rows built so that y nearly cancels: the bound then exceeds the bf16 spacing and the
    output must be left undecided rather than decided wrongly."""
    rng = np.random.default_rng(4)
    t = rng.standard_normal((128, 128)).astype(np.float32)
    x = rng.standard_normal((64, 128))
    # make x nearly orthogonal to the first 16 rows of T
    q, _ = np.linalg.qr(t[:16].astype(np.float64).T)
    x = x - (x @ q) @ q.T
    xb = synth.f32_to_bf16_bits(x.astype(np.float32))
    frac = _check(t, xb, seed=4)
    assert frac < 1.0                               # some outputs go to the exact path


def test_subnormal_and_tiny_entries():
    rng = np.random.default_rng(5)
    t = (rng.standard_normal((128, 128)) * 0.1).astype(np.float32)
    t[5, 7] = np.float32(1e-39)
    t[9] *= np.float32(2.0 ** -100)
    x = rng.standard_normal((32, 128))
    x[:, ::5] *= 2.0 ** -30                         # rows with elements far below their maximum
    _check(t, synth.f32_to_bf16_bits(x.astype(np.float32)), seed=5)
