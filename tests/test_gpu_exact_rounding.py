"""Transformed rows whose exact value lies on, or extremely close to, a bf16 rounding midpoint:
the rotation must still return the exact product rounded once (nearest-even), bit for bit
against the oracle's exact-rational rounding.

The rows are built so that every fast decision fails and the last resort must be exact:
* dense rows (T fp32, x bf16): four terms in the order tiny, +2^30, midpoint, -2^30 (scaled by
  2^s), so that the value is a midpoint m exactly (a tie: to even) or m +- 2^-46 m or
  m + 2^-70 m, and a double-float accumulation loses the tiny term on the way; at decode size
  (CUDA-core path) and at the size that takes the tensor-core path;
* Walsh-Hadamard rows whose first output S / sqrt(128) lies within about 2^-60 (relative) of a
  midpoint, S spread over eight bf16 pieces spanning 64 bits.
"""

from fractions import Fraction
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import synth
from oracle import transform
from tests import harness

TC_MIN_PAIRS = 128 * 152
HKV = 8
# column of the four-term pattern per kv head (some split across lanes) and its order
OFFSETS = [0, 4, 60, 124, 2, 33, 97, 125]
ORDERS = [(0, 1, 2, 3), (1, 0, 2, 3), (0, 2, 1, 3), (3, 1, 0, 2), (0, 1, 3, 2), (2, 0, 1, 3), (0, 3, 2, 1),
          (1, 2, 0, 3)]


def _pattern(h):
    off = min(OFFSETS[h], 124)
    return [off + k for k in ORDERS[h]]            # columns of (tiny, big, mid, -big)


def _matrices():
    """[HKV, 128, 128] float32: output i of head h has the value m_i + delta_i x_tiny / scale."""
    t = np.zeros((HKV, 128, 128), np.float32)
    for h in range(HKV):
        c_tiny, c_big, c_mid, c_neg = _pattern(h)
        for i in range(128):
            m = 1.0 + (2 * i + 1) * 2.0 ** -8           # the midpoints of bf16 in [1, 2)
            sgn = -1.0 if (i // 4) % 2 else 1.0
            delta = [0.0, 2.0 ** -6, -(2.0 ** -6), 2.0 ** -30][i % 4]
            t[h, i, c_tiny] = sgn * delta
            t[h, i, c_big] = 2.0 ** 10
            t[h, i, c_mid] = sgn * m
            t[h, i, c_neg] = -(2.0 ** 10)
    return t


def _rows(n, hq, rng, every=1):
    """[n, hq, 128] bf16 bits: the pattern (tiny 2^-40, big 2^20, 1, big 2^20) times 2^s on every
    `every`-th row (the oracle's exact rounding of each such output is slow), ordinary Gaussian
    rows elsewhere and on every fifth pattern slot."""
    g = hq // HKV
    x = np.zeros((n, hq, 128), np.float32)
    for r in range(n):
        s = [0, -30, 10, 40][(r // every) % 4]
        for hh in range(hq):
            if r % every or (r // every) % 5 == 4:
                x[r, hh] = rng.standard_normal(128)
                continue
            c_tiny, c_big, c_mid, c_neg = _pattern(hh // g)
            x[r, hh, c_tiny] = 2.0 ** (-40 + s)
            x[r, hh, c_big] = 2.0 ** (20 + s)
            x[r, hh, c_mid] = 2.0 ** s
            x[r, hh, c_neg] = 2.0 ** (20 + s)
    return synth.f32_to_bf16_bits(x)


def _run_queries(x_bits, tkit, hadamard=False):
    import bit_rotated_kv_gb300 as kvq
    n, hq, d = x_bits.shape
    w = synth.TINY_GQA4.replace(n_q_heads=hq, n_kv_heads=HKV, batch=1)
    dev = torch.device("cuda")
    cfg, _ = harness.kv_config(w, [512])
    t = None if hadamard else torch.from_numpy(np.ascontiguousarray(tkit, np.float32)).to(dev)
    kind = kvq.KVQ_TRANSFORM_HADAMARD if hadamard else kvq.KVQ_TRANSFORM_DENSE
    tr = kvq.Transform(kind, t, t, None)
    cache = kvq.KVCache(cfg, dev)
    q = harness._bf16_dev(x_bits, dev)
    q_out = torch.full_like(q, float("nan"))
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    kvq.kv_rotate_qk(cfg, tr, q, q_out, None, None, None, None, cache, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return harness.bits(q_out)


def _oracle(x_bits, tkit, hadamard=False):
    n, hq, d = x_bits.shape
    g = hq // HKV
    out = np.zeros_like(x_bits)
    for h in range(hq):
        if hadamard:
            out[:, h] = synth.f32_to_bf16_bits(transform.rotate_rows(None, x_bits[:, h], "hadamard"))
        else:
            out[:, h] = synth.f32_to_bf16_bits(transform.rotate_rows(tkit[h // g], x_bits[:, h]))
    return out


def _compare(got, ref):
    bad = np.argwhere(got != ref)
    assert bad.size == 0, (len(bad), bad[:5], hex(int(got[tuple(bad[0])])), hex(int(ref[tuple(bad[0])])))


def test_oracle_sees_ties_and_near_midpoints():
    """The constructed values really are ties / near-ties (CPU, on the oracle's side)."""
    tkit = _matrices()
    x = _rows(4, HKV, np.random.default_rng(0))
    ref = _oracle(x, tkit)
    # output i of pattern row 0 (scale 1): a tie rounds to even, +delta up, -delta down
    for i in range(0, 16):
        m = Fraction(1) + Fraction(2 * i + 1, 256)
        sgn = -1 if (i // 4) % 2 else 1
        lo_b = synth.f32_to_bf16_bits(np.array([float(m - Fraction(1, 256))], np.float32))[0]
        hi_b = synth.f32_to_bf16_bits(np.array([float(m + Fraction(1, 256))], np.float32))[0]
        want = {0: lo_b if (lo_b & 1) == 0 else hi_b, 1: hi_b, 2: lo_b, 3: hi_b}[i % 4]
        if sgn < 0:
            want |= 0x8000
        assert ref[0, 0, i] == want, (i, hex(int(ref[0, 0, i])), hex(int(want)))


@pytest.mark.gpu
def test_dense_near_midpoint_decode_size():
    tkit = _matrices()
    x = _rows(6, 32, np.random.default_rng(1))
    assert x.shape[0] * x.shape[1] < TC_MIN_PAIRS
    _compare(_run_queries(x, tkit), _oracle(x, tkit))


@pytest.mark.gpu
def test_dense_near_midpoint_tensor_core_size():
    tkit = _matrices()
    n = TC_MIN_PAIRS // 32 + 37
    x = _rows(n, 32, np.random.default_rng(2), every=24)
    assert x.shape[0] * x.shape[1] >= TC_MIN_PAIRS
    _compare(_run_queries(x, tkit), _oracle(x, tkit))


def _hadamard_rows(n, chunks=8):
    """Rows whose output 0, S / sqrt(128) with S = sum of the row, lies within ~2^-(8 chunks + 4)
    of a midpoint m: S = K 2^-(8 chunks) with K the integer nearest m sqrt(128) 2^(8 chunks),
    split into 8-bit chunks (each an exact bf16).  8 chunks span 56 binades (the double-float
    path with its bound); 4 span fewer than 32 (the integer path)."""
    getcontext().prec = 60
    sqrt128 = Decimal(128).sqrt()
    nb = 8 * chunks
    x = np.zeros((n, HKV, 128), np.float64)
    for r in range(n):
        for h in range(HKV):
            k = (r * HKV + h) % 128
            m = Decimal(1) + Decimal(2 * k + 1) / Decimal(256)
            K = int((m * sqrt128 * (Decimal(2) ** nb)).to_integral_value())
            s = [0, -50, 30][(r + h) % 3]
            sign = -1.0 if (r + h) % 2 else 1.0
            for c in range(chunks):
                chunk = (K >> (8 * c)) & 0xFF
                x[r, h, 3 + 7 * c] = sign * chunk * 2.0 ** (8 * c - nb + s)
    return synth.f32_to_bf16_bits(x.astype(np.float32))


@pytest.mark.gpu
@pytest.mark.parametrize("chunks", [8, 4])
def test_hadamard_near_midpoint(chunks):
    x = _hadamard_rows(12, chunks)
    # the chunks are exact bf16 values (8-bit integers times powers of two)
    assert np.array_equal(synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(x)), x)
    _compare(_run_queries(x, None, hadamard=True), _oracle(x, None, hadamard=True))
