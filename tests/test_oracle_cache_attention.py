"""Pins of the oracle's flush schedule, mixed cache and attention (CPU only).

Pinned to: the closed form of eager flushing and its invariants, torch's
scaled_dot_product_attention in float64 (an independent library routine),
special cases with known answers, and the all-BF16 case.
"""

import math

import numpy as np
import pytest
import torch

import synth
from oracle import attention, cache, pipeline
from oracle.fp import bf16_to_f32


@pytest.mark.parametrize("s_sink,s_keep,s_flush", [(64, 256, 8), (16, 128, 16), (0, 0, 128), (64, 256, 1), (4, 0, 1)])
def test_flush_schedule_closed_form(s_sink, s_keep, s_flush):
    rng = np.random.default_rng(s_flush + s_keep)
    L, sq = 0, s_sink
    for _ in range(400):
        L += int(rng.integers(0, 40))
        sq = cache.flush(L, sq, s_keep, s_flush)
        closed = s_sink + s_flush * max(0, (L - s_sink - s_keep) // s_flush)
        assert sq == closed
        assert (sq - s_sink) % s_flush == 0
        assert L - sq < s_keep + s_flush or L < s_sink
        if L >= s_sink + s_keep:
            assert sq <= L - s_keep


def test_cache_states_of_the_workloads():
    # tiny-gqa4-ctx512: INT2 [16, 384) = 23 pages, BF16 16 + 128
    w = synth.TINY_GQA4
    assert pipeline.s_quant_schedule(w, 504) == (376, 384)
    # qwen3-8b-ctx32k-b1: s_quant = 32768 - 264 before, one span of 8 flushed by the step
    w = synth.QWEN3_8B_32K
    assert pipeline.s_quant_schedule(w, 32760) == (32504, 32512)
    # wush-qwen3-8b-b16-chunk2048-on-16k: INT2 [64, 16128) before, +2048 after
    w = synth.WUSH_CHUNK_B16
    assert pipeline.s_quant_schedule(w, 16384) == (16128, 18176)
    # qwen3-32b-ctx128k-b4-oscar: everything INT2, one new BF16 token
    w = synth.QWEN3_32B_128K
    assert pipeline.s_quant_schedule(w, 131072) == (131072, 131072)


def _sdpa(q, k, v, scale):
    qt = torch.tensor(q, dtype=torch.float64)[None, :, None, :]
    kt = torch.tensor(k, dtype=torch.float64)[None, None].expand(1, q.shape[0], *k.shape)
    vt = torch.tensor(v, dtype=torch.float64)[None, None].expand(1, q.shape[0], *v.shape)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o[0, :, 0, :].numpy()


@pytest.mark.parametrize("L", [1, 2, 7, 300])
def test_attention_matches_torch_sdpa(L):
    rng = np.random.default_rng(L)
    q = rng.standard_normal((4, 128)) * 2
    k = rng.standard_normal((L, 128))
    v = rng.standard_normal((L, 128))
    s = 1 / math.sqrt(128)
    assert np.allclose(attention.decode(q, k, v, s), _sdpa(q, k, v, s), rtol=1e-12, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((3, 16))
    v = rng.standard_normal((5, 16))
    # one token -> its value row
    assert np.allclose(attention.decode(q, rng.standard_normal((1, 16)), v[:1], 0.25), np.repeat(v[:1], 3, 0))
    # equal keys -> mean of values
    k = np.repeat(rng.standard_normal((1, 16)), 5, 0)
    assert np.allclose(attention.decode(q, k, v, 0.25), np.repeat(v.mean(0, keepdims=True), 3, 0))
    # empty context -> zeros
    assert np.all(attention.decode(q, np.zeros((0, 16)), np.zeros((0, 16)), 0.25) == 0)
    # shift invariance of the logits (max subtraction) on huge scores
    kk = rng.standard_normal((5, 16))
    assert np.allclose(attention.decode(q * 1e3, kk, v, 1.0), _sdpa(q * 1e3, kk, v, 1.0))


def test_gqa_one_reduces_to_mha():
    w = synth.TINY_GQA4.replace(n_q_heads=1, n_kv_heads=1, ctx_lo=40, ctx_hi=40, s_sink=4, s_keep=8)
    tk, tkit, tv = synth.transforms(w)
    ui = synth.unit_inputs(w, 0, 0)
    r = pipeline.run_unit(w, ui, tk, tkit, tv)
    k, v = cache.dequantized_kv(r["unit"])
    q = bf16_to_f32(r["q_rot"]).astype(np.float64)
    assert r["out"].shape == (1, 128)
    assert np.allclose(r["out"], _sdpa(q, k, v, 1 / math.sqrt(128)), rtol=1e-12, atol=1e-12)


def test_all_bf16_when_context_fits_windows():
    # context <= S_sink + S_keep: nothing is quantized, attention is plain BF16 attention
    w = synth.TINY_GQA4.replace(ctx_lo=100, ctx_hi=100)
    tk, tkit, tv = synth.transforms(w)
    ui = synth.unit_inputs(w, 0, 0)
    r = pipeline.run_unit(w, ui, tk, tkit, tv)
    assert r["s_quant"] == w.s_sink
    k = bf16_to_f32(r["k_rot"]).astype(np.float64)
    v = bf16_to_f32(r["v_rot"]).astype(np.float64)
    q = bf16_to_f32(r["q_rot"]).astype(np.float64)
    assert np.allclose(r["out"], _sdpa(q, k, v, 1 / math.sqrt(128)), rtol=1e-12, atol=1e-12)


def test_tiny_workload_end_to_end_shapes_and_accuracy():
    """The tiny GQA-4 workload (512 tokens) through the oracle.  The accuracy of INT2 attention against
    unquantized attention is reported, not pinned (the pages' accuracy claims
    need trained models)."""
    w = synth.TINY_GQA4
    tk, tkit, tv = synth.transforms(w)
    ui = synth.unit_inputs(w, 0, 0)
    r = pipeline.run_unit(w, ui, tk, tkit, tv)
    u = r["unit"]
    assert u["qk"]["codes"].shape == (384 - 16, 128)
    k = bf16_to_f32(r["k_rot"]).astype(np.float64)
    v = bf16_to_f32(r["v_rot"]).astype(np.float64)
    q = bf16_to_f32(r["q_rot"]).astype(np.float64)
    ref = attention.decode(q, k, v, 1 / math.sqrt(128))
    rel = np.abs(r["out"] - ref).max() / np.abs(ref).max()
    # random synthetic rows have no attention structure, so INT2 noise is large relative to the
    # averaged output; only sanity is asserted here
    assert np.isfinite(rel) and rel < 2.0
