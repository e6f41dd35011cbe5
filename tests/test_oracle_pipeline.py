"""Pins of the oracle's end-to-end wiring (CPU only): which matrix compensates the
queries, and which tokens the cache quantizes.

Pinned to:
* the logit invariant q'^T k' = q^T k of the pages' query compensation ([WUSH]
  "核心方法": keys take T, queries T^{-T}, so that (T^{-T} q)^T (T k) = q^T k),
  checked on the pipeline's own BF16 outputs for a general invertible T (for
  which T and T^{-T} differ), within the rounding bound of the two BF16 rows;
* the region rule of the mixed cache ([WUSH] "方法步骤详情": tokens [0, S_sink)
  and [S_quant, L) stay BF16, [S_sink, S_quant) is quantized; S_quant from the
  closed form of eager flushing), checked row by row: every row inside the
  region is its own per-token quantization, every row outside is its BF16 row.

The last tests plant plausible mistakes in the oracle's wiring (T instead of
T^{-T} for queries, the quantized region shifted by one token) and check that
the pins catch each one.
"""

import numpy as np
import pytest

import synth
from oracle import attention, cache, pipeline, quant
from oracle.fp import bf16_to_f32

U_BF16 = 2.0 ** -8          # unit roundoff of bfloat16 (8-bit significand)


def _short_invertible():
    # general invertible T_K (condition number 100), everything inside the BF16 windows
    return synth.WUSH_CHUNK_B16.replace(batch=1, ctx_lo=40, ctx_hi=40, n_new=8)


def _logit_excess(q_raw, k_raw, q_rot, k_rot):
    """max over (query, token) of |q'.k' - q.k| / bound, bound = the BF16 rounding of q' and k'
    (2u + u^2 times sum |q'_j k'_j|) plus 1e-4 |q| |k| for T^{-T} being a float32 matrix."""
    q = bf16_to_f32(q_raw).astype(np.float64)
    k = bf16_to_f32(k_raw).astype(np.float64)
    qr = bf16_to_f32(q_rot).astype(np.float64)
    kr = bf16_to_f32(k_rot).astype(np.float64)
    lhs = qr @ kr.T
    rhs = q @ k.T
    bound = (2 * U_BF16 + U_BF16 ** 2) / (1 - U_BF16) ** 2 * (np.abs(qr) @ np.abs(kr).T)
    bound += 1e-4 * np.outer(np.linalg.norm(q, axis=1), np.linalg.norm(k, axis=1))
    return float(np.max(np.abs(lhs - rhs) / bound))


def test_pipeline_queries_keep_logits_invertible_t():
    w = _short_invertible()
    tk, tkit, tv = synth.transforms(w)
    for h in range(w.n_kv_heads):
        ui = synth.unit_inputs(w, 0, h)
        r = pipeline.run_unit(w, ui, tk, tkit, tv, attend=False)
        assert _logit_excess(ui.q, ui.k, r["q_rot"], r["k_rot"]) <= 1.0


def test_chunk_queries_keep_logits_invertible_t():
    w = _short_invertible()
    tk, tkit, tv = synth.transforms(w)
    for h in (0, 5):
        ui = synth.unit_inputs(w, 0, h)
        r = pipeline.run_unit(w, ui, tk, tkit, tv, attend=False)
        qc = synth.chunk_query_rows(w, 0, h)[:6]                 # [n, g, d]
        qc_rot = pipeline.rotate_chunk_queries(w, h, qc, tkit)
        assert qc_rot.shape == qc.shape
        assert _logit_excess(qc.reshape(-1, w.head_dim), ui.k, qc_rot.reshape(-1, w.head_dim), r["k_rot"]) <= 1.0


def _region_rows_hold(w, b=0, h=0):
    """The quantized region is [S_sink, closed-form S_quant); rows inside are their own per-row
    quantization (dequantized), rows outside their BF16 rows, element for element."""
    tk, tkit, tv = synth.transforms(w)
    ui = synth.unit_inputs(w, b, h)
    r = pipeline.run_unit(w, ui, tk, tkit, tv, attend=False)
    L = ui.ctx + w.n_new
    closed = w.s_sink + w.s_flush * max(0, (L - w.s_sink - w.s_keep) // w.s_flush)
    u = r["unit"]
    assert (u["s_sink"], u["s_quant"]) == (w.s_sink, closed)
    kh, vh = cache.dequantized_kv(u)
    k_bf = bf16_to_f32(r["k_rot"]).astype(np.float64)
    v_bf = bf16_to_f32(r["v_rot"]).astype(np.float64)
    inside = np.zeros(L, bool)
    inside[w.s_sink:closed] = True
    for t in range(L):
        if inside[t]:
            kq = quant.quantize_rows(r["k_rot"][t:t + 1], w.group_size, w.kappa_k, w.quantizer,
                                     w.quest_alpha, w.key_l2norm)
            vq = quant.quantize_rows(r["v_rot"][t:t + 1], w.group_size, w.kappa_v, w.quantizer,
                                     w.quest_alpha, False)
            assert np.array_equal(kh[t], quant.dequantize(kq)[0])
            assert np.array_equal(vh[t], quant.dequantize(vq)[0])
        else:
            assert np.array_equal(kh[t], k_bf[t]) and np.array_equal(vh[t], v_bf[t])
    # the two kinds of row really differ here (INT2 noise on random rows), so a region shifted
    # by one token changes at least one row on each edge
    assert not np.array_equal(kh[w.s_sink], k_bf[w.s_sink])
    assert not np.array_equal(kh[closed - 1], k_bf[closed - 1])


def test_quantized_region_row_by_row():
    _region_rows_hold(synth.TINY_GQA4.replace(ctx_lo=300, ctx_hi=300))
    _region_rows_hold(synth.TINY_GQA4.replace(ctx_lo=300, ctx_hi=300, s_flush=1, s_keep=16))


# ---- planted mistakes: each must be caught by one of the pins above ---------------------
def test_planted_query_matrix_swap_is_caught(monkeypatch):
    orig = pipeline.rotate_unit

    def bad(w, ui, tk, tkit, tv):
        return orig(w, ui, tk, tk, tv)           # mistake: queries compensated with T_K itself
    monkeypatch.setattr(pipeline, "rotate_unit", bad)
    with pytest.raises(AssertionError):
        test_pipeline_queries_keep_logits_invertible_t()


def test_planted_chunk_query_matrix_swap_is_caught(monkeypatch):
    orig = pipeline.rotate_chunk_queries
    tk, _, _ = synth.transforms(_short_invertible())

    def bad(w, h, q_bits, tkit):
        return orig(w, h, q_bits, tk)            # mistake: T_K instead of T_K^{-T}
    monkeypatch.setattr(pipeline, "rotate_chunk_queries", bad)
    with pytest.raises(AssertionError):
        test_chunk_queries_keep_logits_invertible_t()


def test_planted_region_shift_is_caught(monkeypatch):
    orig = cache.build_unit

    def bad(k, v, L, s_quant, *, s_sink, **kw):
        return orig(k, v, L, s_quant + 1, s_sink=s_sink + 1, **kw)   # mistake: region one token late
    monkeypatch.setattr(cache, "build_unit", bad)
    with pytest.raises(AssertionError):
        test_quantized_region_row_by_row()


def test_planted_region_shift_same_bounds_is_caught(monkeypatch):
    # the region's rows shifted while its reported bounds stay right: caught row by row
    orig = cache.build_unit

    def bad(k, v, L, s_quant, *, s_sink, **kw):
        u = orig(np.roll(k, -1, axis=0), np.roll(v, -1, axis=0), L, s_quant, s_sink=s_sink, **kw)
        u["k_rot"], u["v_rot"] = k[:L], v[:L]
        return u
    monkeypatch.setattr(cache, "build_unit", bad)
    with pytest.raises(AssertionError):
        test_quantized_region_row_by_row()


# ---- chunk attention (causal queries of an appended chunk over the mixed cache) ---------------

def _brute_prefix(q, pos, k, v, scale):
    """Softmax attention written out with loops: q [n, g, d], query i sees k[0..pos[i]]."""
    n, g, d = q.shape
    out = np.zeros((n, g, d))
    for i in range(n):
        for hh in range(g):
            s = np.array([sum(q[i, hh, c] * k[t, c] for c in range(d)) * scale for t in range(int(pos[i]) + 1)])
            e = np.exp(s - s.max())
            out[i, hh] = (e[:, None] * v[:int(pos[i]) + 1]).sum(0) / e.sum()
    return out


def test_chunk_attention_brute_force_causal():
    rng = np.random.default_rng(21)
    q = rng.standard_normal((5, 2, 6))
    k = rng.standard_normal((7, 6))
    v = rng.standard_normal((7, 6))
    pos = np.arange(2, 7)
    got = attention.chunk(q, pos, k, v, 0.4)
    assert np.allclose(got, _brute_prefix(q, pos, k, v, 0.4), rtol=1e-12, atol=1e-12)
    # an off-by-one prefix (tokens [0, p) instead of [0, p]) differs
    assert not np.allclose(attention.chunk(q, pos - 1, k, v, 0.4), got)


def test_chunk_attention_last_query_is_the_decode_query():
    """The chunk query at the last position with the decode query's values gives the decode
    output; a chunk inside the BF16 sink is causal attention over the rotated BF16 rows."""
    w = synth.TINY_GQA4.replace(ctx_lo=200, ctx_hi=200, n_new=40, s_sink=16, s_keep=64, s_flush=8)
    tk, tkit, tv = synth.transforms(w)
    ui = synth.unit_inputs(w, 0, 0, synth.context_lengths(w))
    qc = synth.chunk_query_rows(w, 0, 0)
    qc[-1] = ui.q
    r = pipeline.run_unit_chunk_attention(w, ui, tk, tkit, tv, qc)
    d = pipeline.run_unit(w, ui, tk, tkit, tv)
    assert np.allclose(r["out_chunk"][-1], d["out"], rtol=1e-12, atol=1e-14)
    w2 = w.replace(ctx_lo=5, ctx_hi=5, n_new=6, s_sink=16)
    ui2 = synth.unit_inputs(w2, 0, 0, synth.context_lengths(w2))
    r2 = pipeline.run_unit_chunk_attention(w2, ui2, tk, tkit, tv, synth.chunk_query_rows(w2, 0, 0))
    k = bf16_to_f32(r2["k_rot"]).astype(np.float64)
    v = bf16_to_f32(r2["v_rot"]).astype(np.float64)
    q = bf16_to_f32(r2["q_chunk_rot"]).astype(np.float64)
    want = _brute_prefix(q, 5 + np.arange(6), k, v, 1 / np.sqrt(128))
    assert np.allclose(r2["out_chunk"], want, rtol=1e-10, atol=1e-12)
