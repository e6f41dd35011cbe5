"""Pins of the oracle's quantizer (CPU only).

Pinned to: the worked example of the OScaR note (TNI section), the uniform
quantizer's definition and error bound ("整数量化基础"), KIVI's zero point,
numpy.quantile, brute force over all code vectors, the MSE-optimal clip of a
4-level uniform quantizer for a unit Gaussian (numerical integration), and
||y|| = 1 for l2-scaled keys.  The last tests plant plausible mistakes in the
oracle and check that a pin catches each one.
"""

import json
import math
import os

import numpy as np
import pytest
import scipy.integrate
import scipy.optimize
import scipy.stats

import synth
from oracle import quant

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))
F32 = np.float32


def _bits(x):
    return synth.f32_to_bf16_bits(np.asarray(x, np.float32))


def _q(x, group, **kw):
    return quant.quantize_rows(_bits(x), group, **kw)


def test_tni_worked_example():
    g = GOLD["tni_worked_example"]
    row = np.zeros((1, 4), np.float32)
    row[0] = [g["max"], g["min"], g["low_norm_value"], 0.0]
    q = _q(row, 4, kappa=1.0)
    assert float(q["delta16"][0, 0]) == g["delta"]
    xh = quant.dequantize(q)
    x = synth.bf16_bits_to_f32(_bits(row)).astype(np.float64)
    assert np.max(np.abs(x - xh)) <= g["error_bound"]
    # the low-norm value is reconstructed with an error close to the whole bound
    assert abs(x[0, 2] - xh[0, 2]) > 0.8


def test_hand_made_group_and_half_even_tie():
    g = GOLD["kivi_zero_point"]
    q = _q([[-1.0, 0.0, 0.5, 2.0]], 4, kappa=1.0)
    assert float(q["delta16"][0, 0]) == g["delta"]
    assert float(q["zero16"][0, 0]) == g["zero_point"]
    assert q["codes"].tolist() == [[0, 1, 2, 3]]          # 0.5 -> u = 1.5 -> 2 (half-even)
    q = _q([[-1.0, 1.5, 0.0, 2.0]], 4, kappa=1.0)
    assert q["codes"].tolist() == [[0, 2, 1, 3]]          # 1.5 -> u = 2.5 -> 2 (half-even)


@pytest.mark.parametrize("group", [32, 64, 128])
def test_error_bound_unclipped(group):
    rng = np.random.default_rng(group)
    x = rng.standard_normal((4000, 128)).astype(np.float32) * np.exp(rng.standard_normal((4000, 1))).astype(np.float32)
    q = _q(x, group, kappa=1.0)
    xh = quant.dequantize(q)
    xb = synth.bf16_bits_to_f32(_bits(x)).astype(np.float64)
    half = np.repeat(q["delta16"].astype(np.float64), group, axis=1) / 2
    assert np.all(np.abs(xb - xh) <= half * (1 + 1e-6))
    assert q["codes"].max() <= 3


def test_clipping_kappa():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((2000, 128)).astype(np.float32)
    xb = synth.bf16_bits_to_f32(_bits(x))
    q = _q(x, 128, kappa=0.99)
    lo, hi = quant.group_range(xb.reshape(2000, 1, 128), 0.99)
    xh = quant.dequantize(q)
    inside = (xb >= lo) & (xb <= hi)
    half = q["delta16"].astype(np.float64) / 2
    err = np.abs(xb - xh)
    # values inside [lo, hi] obey the bound; values outside land on an end level
    assert np.all(err[inside] <= np.broadcast_to(half, err.shape)[inside] * (1 + 1e-3) + 1e-6)
    outside_hi = xb > hi
    assert np.all(q["codes"][outside_hi] >= 2)


@pytest.mark.parametrize("kappa", [1.0, 0.999, 0.995, 0.99, 0.96, 0.92, 0.75])
@pytest.mark.parametrize("group", [32, 64, 128])
def test_quantile_matches_numpy(kappa, group):
    rng = np.random.default_rng(int(kappa * 1000) + group)
    y = rng.standard_normal((500, group)).astype(np.float32)
    lo, hi = quant.group_range(y, kappa)
    ref_hi = np.quantile(y.astype(np.float64), kappa, axis=-1, method="linear")
    ref_lo = np.quantile(y.astype(np.float64), 1 - kappa, axis=-1, method="linear")
    tol = 4 * np.spacing(np.abs(ref_hi).astype(np.float32)) + 1e-7
    assert np.all(np.abs(hi - ref_hi) <= tol)
    tol = 4 * np.spacing(np.abs(ref_lo).astype(np.float32)) + 1e-7
    assert np.all(np.abs(lo - ref_lo) <= tol)
    if kappa == 1.0:
        assert np.array_equal(hi, y.max(-1)) and np.array_equal(lo, y.min(-1))


def test_codes_are_nearest_level_brute_force():
    """G = 4, kappa = 1: the chosen code vector minimises the squared error over all 4^4."""
    rng = np.random.default_rng(9)
    allc = np.array(np.meshgrid(*[np.arange(4)] * 4, indexing="ij")).reshape(4, -1).T  # [256, 4]
    for _ in range(300):
        x = rng.standard_normal((1, 4)).astype(np.float32) * F32(rng.uniform(0.01, 10))
        q = _q(x, 4, kappa=1.0)
        xb = synth.bf16_bits_to_f32(_bits(x)).astype(np.float64)[0]
        dd = float(q["delta16"][0, 0]); zz = float(q["zero16"][0, 0])
        errs = np.sum((xb[None, :] - dd * (allc - zz)) ** 2, axis=1)
        best = errs.min()
        mine = np.sum((xb - dd * (q["codes"][0] - zz)) ** 2)
        assert mine <= best * (1 + 1e-9) + 1e-30


def _gauss_mse(alpha):
    """E[(x - Q(x))^2] for x ~ N(0,1), mid-rise 4-level grid +-alpha/3, +-alpha."""
    step = 2 * alpha / 3
    levels = step * (np.arange(4) - 1.5)
    edges = [-np.inf, -step, 0.0, step, np.inf]
    tot = 0.0
    for i in range(4):
        f = lambda t, c=levels[i]: (t - c) ** 2 * scipy.stats.norm.pdf(t)
        tot += scipy.integrate.quad(f, edges[i], edges[i + 1])[0]
    return tot


def test_quest_alpha_default_is_mse_optimal():
    res = scipy.optimize.minimize_scalar(_gauss_mse, bounds=(0.5, 3.0), method="bounded",
                                         options={"xatol": 1e-7})
    assert abs(res.x - synth.Workload.__dataclass_fields__["quest_alpha"].default) < 1e-4


def test_quest_grid_and_delta():
    rng = np.random.default_rng(10)
    x = rng.standard_normal((300, 128)).astype(np.float32)
    alpha = 1.4935705
    q = _q(x, 32, quantizer="quest", alpha=alpha)
    xb = synth.bf16_bits_to_f32(_bits(x)).astype(np.float64).reshape(300, 4, 32)
    delta = 2 * alpha * np.linalg.norm(xb, axis=-1) / (math.sqrt(32) * 3)   # Delta = 2 alpha ||x|| / (sqrt(G)(2^b-1))
    assert np.allclose(q["delta16"].astype(np.float64), delta, rtol=2 ** -10)
    assert np.all(q["zero16"] == 1.5)
    # nearest of the four levels, clipped to the outer ones
    dd = q["delta16"].astype(np.float64)[..., None]
    levels = dd * (np.arange(4) - 1.5)
    best = np.argmin(np.abs(xb[..., None] - levels[..., None, :]), axis=-1)
    c = q["codes"].reshape(300, 4, 32)
    ties = np.isclose(np.abs(xb / dd + 1.5 - np.round(xb / dd + 1.5)), 0.5)
    assert np.all((c == best) | ties)


def test_l2_scaling():
    rng = np.random.default_rng(13)
    x = rng.standard_normal((400, 128)).astype(np.float32) * np.exp(2 * rng.standard_normal((400, 1))).astype(np.float32)
    x[0] = 0
    xb = synth.bf16_bits_to_f32(_bits(x))
    y, s16 = quant.l2_scale(xb)
    n = np.linalg.norm(y[1:].astype(np.float64), axis=1)
    assert np.all(np.abs(n - 1) < 2 ** -10)      # s is stored as float16
    assert s16[0] == 0 and np.all(y[0] == 0)
    assert np.allclose(s16[1:].astype(np.float64), np.linalg.norm(xb[1:].astype(np.float64), axis=1), rtol=2 ** -11)
    q = _q(x, 32, kappa=1.0, l2=True)
    xh = quant.dequantize(q)
    half = np.repeat(q["delta16"].astype(np.float64), 32, axis=1) / 2 * q["norm16"].astype(np.float64)[:, None]
    # bound in the scaled domain, carried back by s16 (y = x / s16 exactly up to one float32 rounding)
    assert np.all(np.abs(xb - xh) <= half * (1 + 1e-5) + np.abs(xb) * 2 ** -23)
    assert np.all(xh[0] == 0)


def test_constant_group_and_nonfinite_flag():
    q = _q(np.full((1, 32), 2.5), 32, kappa=1.0)
    assert float(q["delta16"][0, 0]) == 1.0 and float(q["zero16"][0, 0]) == -2.5
    assert np.allclose(quant.dequantize(q), 2.5)
    big = np.zeros((1, 32), np.float32)
    big[0, 0] = 3e5; big[0, 1] = -3e5
    assert _q(big, 32, kappa=1.0)["nonfinite"][0]


def test_pack_layout_lsb_first():
    g = GOLD["codes_per_byte"]
    c = np.zeros((1, 128), np.uint8)
    c[0, :4] = [1, 2, 3, 0]
    words = quant.pack_lsb(c)
    assert words.shape == (1, 8)                       # 128 codes -> 32 bytes per row
    assert words.view(np.uint8).shape[1] == GOLD["code_bytes_per_token"]["code_bytes"]
    assert int(words.view(np.uint8)[0, 0]) == 1 | 2 << 2 | 3 << 4      # four codes per byte, LSB first
    assert g["codes_per_byte"] == 4
    rng = np.random.default_rng(14)
    c = rng.integers(0, 4, (50, 128)).astype(np.uint8)
    assert np.array_equal(quant.unpack_lsb(quant.pack_lsb(c)), c)


# ---- planted mistakes: each must be caught by one of the pins above ---------------------
def test_planted_zero_point_sign_is_caught(monkeypatch):
    orig = quant.affine_params

    def bad(lo, hi):
        d16, z16 = orig(lo, hi)
        return d16, (-z16.astype(np.float32)).astype(np.float16)     # mistake: z = +min/Delta
    monkeypatch.setattr(quant, "affine_params", bad)
    with pytest.raises(AssertionError):
        test_hand_made_group_and_half_even_tie()


def test_planted_quantile_index_is_caught(monkeypatch):
    def bad_pos(g, kappa):
        pos = g * float(kappa)               # mistake: G instead of G - 1
        i = int(math.floor(pos))
        return min(i, g - 1), F32(pos - i)
    monkeypatch.setattr(quant, "kappa_position", bad_pos)
    with pytest.raises(AssertionError):
        test_quantile_matches_numpy(0.99, 128)


def test_planted_dropped_rounding_is_caught(monkeypatch):
    def bad_codes(y, d16, z16):
        u = y.astype(F32) / d16.astype(F32)[..., None] + z16.astype(F32)[..., None]
        return np.clip(np.floor(u), 0, 3).astype(np.uint8)     # mistake: floor instead of round
    monkeypatch.setattr(quant, "codes_from_params", bad_codes)
    with pytest.raises(AssertionError):
        test_error_bound_unclipped(128)


def _quest_mse(alpha, group, seed=21, rows=4000):
    """Mean squared error of the oracle's QuEST grid on Gaussian rows, in units of each group's
    mean square."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, 128)).astype(np.float32)
    bits = synth.f32_to_bf16_bits(x)
    q = quant.quantize_rows(bits, group, quantizer="quest", alpha=alpha)
    xb = synth.bf16_bits_to_f32(bits).astype(np.float64)
    err = (xb - quant.dequantize(q)).reshape(rows, 128 // group, group)
    ms = (xb.reshape(rows, 128 // group, group) ** 2).mean(-1, keepdims=True)
    return float((err ** 2 / ms).mean())


def test_quest_delta_against_the_gaussian_integral():
    """The grid's scale is pinned by what it is for: on Gaussian groups the oracle's error (in
    units of the group's mean square) equals the integral of the 4-level clipped grid at alpha
    over N(0, 1) -- up to the group's own RMS estimate (1.3% at G = 128).  A grid scaled by the
    norm over sqrt(d) instead of sqrt(G), or by alpha / 2, lands far from it."""
    alpha = 1.4935705
    ref = _gauss_mse(alpha)
    assert abs(_quest_mse(alpha, 128) / ref - 1) < 0.03
    assert 0.9 < _quest_mse(alpha, 32) / ref < 1.0           # finite-G: RMS from 32 values
    # the same error with the grid misplaced: both far outside those bands
    assert _quest_mse(alpha / 2, 128) / ref > 1.5
    assert _quest_mse(alpha * 2, 128) / ref > 1.5
