"""Pins of the oracle's per-channel key quantizer (CPU only).

Pinned to: the OScaR note's block example of per-channel quantization (TNI analysis: a
channel spanning +3 .. -3 over the block gives Delta = 2 and error bound 1, which a
low-norm token's value of 0.1 fills almost entirely), the uniform quantizer's bound and
nearest-level property (brute force over the four levels), and two invariances that only
the per-channel direction has: scaling one channel by a power of two scales its Delta
exactly and changes no code anywhere, and permuting the tokens of a block permutes its
codes and leaves every scale as it was.  A planted mistake (statistics taken along a
token's channels instead of along a channel's tokens) is caught by those invariances.
"""

import json
import os

import numpy as np

import synth
from oracle import quant

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))
BLOCK = 16


def _bits(x):
    return synth.f32_to_bf16_bits(np.asarray(x, np.float32))


def _vals(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def test_tni_block_example():
    g = GOLD["tni_worked_example"]
    rng = np.random.default_rng(11)
    x = rng.uniform(-2.5, 2.5, size=(BLOCK, 128)).astype(np.float32)
    j = 5
    x[3, j] = g["max"]                  # the high-norm token
    x[9, j] = g["min"]
    x[0, j] = g["low_norm_value"]       # the low-norm (sink) token
    q = quant.quantize_keys_per_channel(_bits(x), BLOCK, kappa=1.0)
    assert float(q["delta16"][0, j]) == g["delta"]
    err = np.abs(_vals(_bits(x)) - quant.dequantize(q))
    assert err[:, j].max() <= g["error_bound"]
    assert err[0, j] > 0.8              # the low-norm token loses almost everything


def _check_bound_and_nearest(qfun, x):
    q = qfun(_bits(x), BLOCK, kappa=1.0)
    y = _vals(_bits(x))
    n, d = y.shape
    dd = np.repeat(q["delta16"].astype(np.float64), BLOCK, axis=0)
    zz = np.repeat(q["zero16"].astype(np.float64), BLOCK, axis=0)
    xh = quant.dequantize(q)
    assert np.all(np.abs(y - xh) <= dd / 2 * (1 + 2.0 ** -9) + 1e-30)
    levels = dd[..., None] * (np.arange(4)[None, None, :] - zz[..., None])
    best = np.abs(y[..., None] - levels).min(-1)
    assert np.all(np.abs(y - xh) <= best + dd * 2.0 ** -9)


def test_bound_and_nearest_level():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((4 * BLOCK, 128)) * np.exp2(rng.integers(-3, 4, size=(1, 128)))).astype(np.float32)
    _check_bound_and_nearest(quant.quantize_keys_per_channel, x)


def _invariances(qfun):
    """(channel scaling invariant holds, token permutation invariant holds) for a quantizer."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((2 * BLOCK, 128)).astype(np.float32)
    q0 = qfun(_bits(x), BLOCK, kappa=1.0)
    j, k = 17, 3
    xs = x.copy()
    xs[:, j] *= np.float32(2.0 ** k)
    q1 = qfun(_bits(xs), BLOCK, kappa=1.0)
    others = np.arange(128) != j
    scaling_ok = (np.array_equal(q1["codes"], q0["codes"])
                  and np.array_equal(q1["delta16"][:, others], q0["delta16"][:, others])
                  and np.array_equal(q1["delta16"][:, j].astype(np.float64),
                                     q0["delta16"][:, j].astype(np.float64) * 2.0 ** k)
                  and np.array_equal(q1["zero16"], q0["zero16"]))
    perm = rng.permutation(BLOCK)
    xp = x.copy()
    xp[:BLOCK] = x[:BLOCK][perm]
    q2 = qfun(_bits(xp), BLOCK, kappa=1.0)
    perm_ok = (np.array_equal(q2["codes"][:BLOCK], q0["codes"][:BLOCK][perm])
               and np.array_equal(q2["codes"][BLOCK:], q0["codes"][BLOCK:])
               and np.array_equal(q2["delta16"], q0["delta16"]) and np.array_equal(q2["zero16"], q0["zero16"]))
    return scaling_ok, perm_ok


def test_per_channel_invariances():
    assert _invariances(quant.quantize_keys_per_channel) == (True, True)


def test_l2_scaled_blocks():
    """Keys scaled per token first (OScaR's omni-token scaling), then quantized per channel:
    each token's reconstruction is s16 times a vector within Delta/2 of the scaled key."""
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((BLOCK, 128)) * np.exp(rng.normal(0, 1.5, size=(BLOCK, 1)))).astype(np.float32)
    q = quant.quantize_keys_per_channel(_bits(x), BLOCK, kappa=1.0, l2=True)
    s = q["norm16"].astype(np.float64)
    xv = _vals(_bits(x))
    assert np.allclose(s, np.linalg.norm(xv, axis=1), rtol=2.0 ** -10)
    y = xv / s[:, None]
    dd = q["delta16"].astype(np.float64)
    yh = quant.dequantize(q) / s[:, None]
    assert np.all(np.abs(y - yh) <= dd / 2 * (1 + 2.0 ** -8))


def test_planted_token_direction_is_caught():
    """Statistics along a token's channels (groups of 16 channels) instead of along a
    channel's 16 tokens: both invariances break."""
    def wrong(x_bits, block, kappa=1.0, l2=False):
        q = quant.quantize_rows(x_bits, block, kappa)
        n, d = q["codes"].shape
        return {"codes": q["codes"], "delta16": q["delta16"].reshape(n // block, -1)[:, :d],
                "zero16": q["zero16"].reshape(n // block, -1)[:, :d]}
    assert _invariances(wrong) != (True, True)


def test_pipeline_wiring_per_channel_keys():
    """A per-channel workload's INT2 region is whole 16-token blocks from S_sink on, keys go
    through the per-channel quantizer and values stay per token."""
    from oracle import pipeline
    w = synth.QWEN3_32B_128K.replace(batch=1, ctx_lo=300, ctx_hi=300, n_new=1, key_axis="channel",
                                     transform="orthogonal")
    tk, tkit, tv = synth.transforms(w)
    ui = synth.unit_inputs(w, 0, 0, synth.context_lengths(w))
    r = pipeline.run_unit(w, ui, tk, tkit, tv)
    u = r["unit"]
    assert u["qk"].get("axis") == "channel" and u["qv"].get("axis") is None
    n = u["s_quant"] - u["s_sink"]
    assert n > 0 and n % BLOCK == 0 and u["qk"]["delta16"].shape == (n // BLOCK, 128)
    q = quant.quantize_keys_per_channel(r["k_rot"][u["s_sink"]:u["s_quant"]], BLOCK, w.kappa_k, w.key_l2norm)
    assert np.array_equal(q["codes"], u["qk"]["codes"])
