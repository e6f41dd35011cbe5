"""One (sequence, kv head) of a workload, end to end: transform, flush, attend.

Oracle module (test infrastructure only).  Follows the serving flow of the
pages ([WUSH] "方法步骤详情" inference algorithm: transform new keys and
queries, append at full precision, quantize S_flush-aligned spans beyond the
windows, mixed-precision attention; [OScaR] algorithm; [OSCAR] section 4):

1. rotate every key row with T_K (or H), every value row with T_V (or keep it),
   and the decode query with T_K^{-T} (or H), each rounded once to BF16;
2. cache state before the measured step: the context of ``ctx`` tokens with the
   flush rule applied from s_quant = S_sink;
3. the step appends ``n_new`` tokens and applies the flush rule again;
4. decode attention of the g query heads over the mixed cache.
"""

from __future__ import annotations

import math

import numpy as np

from . import attention, cache, transform
from .fp import bf16_to_f32, f32_to_bf16_bits


def rotate_unit(w, ui, tk, tkit, tv):
    """Transformed BF16 rows (bit patterns): k', v' [ctx + n_new, d], q' [g, d]."""
    h = ui.h
    if w.transform == "hadamard":
        k_rot = transform.rotate_rows(None, ui.k, "hadamard")
        q_rot = transform.rotate_rows(None, ui.q, "hadamard")
    else:
        k_rot = transform.rotate_rows(tk[h], ui.k)
        q_rot = transform.rotate_rows(tkit[h], ui.q)
    v_rot = transform.rotate_rows(None if tv is None else tv[h], ui.v)
    return f32_to_bf16_bits(k_rot), f32_to_bf16_bits(v_rot), f32_to_bf16_bits(q_rot)


def rotate_chunk_queries(w, h, q_bits, tkit):
    """q' for a chunk of queries [n, g, d] (bit patterns in, bit patterns out)."""
    if w.transform == "hadamard":
        return f32_to_bf16_bits(transform.rotate_rows(None, q_bits, "hadamard"))
    return f32_to_bf16_bits(transform.rotate_rows(tkit[h], q_bits))


def s_quant_schedule(w, ctx: int):
    """(s_quant before the step, s_quant after the step) under the flush rule."""
    before = cache.flush(ctx, w.s_sink, w.s_keep, w.s_flush)
    after = cache.flush(ctx + w.n_new, before, w.s_keep, w.s_flush)
    return before, after


def run_unit(w, ui, tk, tkit, tv, scale: float | None = None, attend: bool = True) -> dict:
    """Everything the hot path produces for one (sequence, kv head)."""
    k_rot, v_rot, q_rot = rotate_unit(w, ui, tk, tkit, tv)
    sq0, sq1 = s_quant_schedule(w, ui.ctx)
    L = ui.ctx + w.n_new
    unit = cache.build_unit(k_rot, v_rot, L, sq1, s_sink=w.s_sink, group=w.group_size,
                            kappa_k=w.kappa_k, kappa_v=w.kappa_v, quantizer=w.quantizer,
                            alpha=w.quest_alpha, key_l2norm=w.key_l2norm, key_axis=w.key_axis)
    res = {"k_rot": k_rot, "v_rot": v_rot, "q_rot": q_rot, "s_quant_before": sq0,
           "s_quant": sq1, "L": L, "unit": unit}
    if attend:
        kh, vh = cache.dequantized_kv(unit)
        sc = 1.0 / math.sqrt(w.head_dim) if scale is None else scale
        res["out"] = attention.decode(bf16_to_f32(q_rot).astype(np.float64), kh, vh, sc)
    return res


def run_unit_chunk_attention(w, ui, tk, tkit, tv, q_chunk_bits, scale: float | None = None) -> dict:
    """The step of run_unit with its appended chunk's queries q_chunk_bits [n_new, g, d]
    (bit patterns) attending causally to the cache after the step: query i at position
    ctx + i sees tokens [0, ctx + i] as the cache holds them (BF16 sink and recent rows,
    the INT2 middle dequantized)."""
    res = run_unit(w, ui, tk, tkit, tv, scale, attend=False)
    kh, vh = cache.dequantized_kv(res["unit"])
    q_rot = rotate_chunk_queries(w, ui.h, q_chunk_bits, tkit)
    sc = 1.0 / math.sqrt(w.head_dim) if scale is None else scale
    pos = ui.ctx + np.arange(q_chunk_bits.shape[0])
    res["q_chunk_rot"] = q_rot
    res["out_chunk"] = attention.chunk(bf16_to_f32(q_rot).astype(np.float64), pos, kh, vh, sc)
    return res
