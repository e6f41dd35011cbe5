"""Element-wise comparison of the GPU cache / outputs with the oracle, per (sequence, kv head)."""

from __future__ import annotations

import numpy as np

import synth
from oracle import pipeline
from tests import layout


def oracle_unit(w: synth.Workload, b: int, h: int, lengths, host_tr):
    tk, tkit, tv = host_tr
    ui = synth.unit_inputs(w, b, h, lengths)
    return pipeline.run_unit(w, ui, tk, tkit, tv)


def compare_unit(run: DeviceRun, snap: dict, b: int, h: int) -> dict:
    """Element-wise comparison of one (sequence, kv head) with the oracle."""
    w = run.w
    ref = oracle_unit(w, b, h, run.lengths, run.host_tr)
    g = w.gqa
    L, sq = ref["L"], ref["s_quant"]
    rep = {"L": L, "s_quant": sq}
    rep["seq_len_ok"] = int(snap["seq_len"][b]) == L
    rep["s_quant_ok"] = int(snap["s_quant"][b]) == sq
    rep["q_mismatch"] = int(np.sum(snap["q_out"][b, h * g:(h + 1) * g] != ref["q_rot"]))
    # BF16 windows: sink rows and recent ring rows
    ns = min(w.s_sink, L)
    mm = 0
    if ns:
        mm += int(np.sum(snap["sink_k"][b, h, :ns] != ref["k_rot"][:ns]))
        mm += int(np.sum(snap["sink_v"][b, h, :ns] != ref["v_rot"][:ns]))
    R = run.cfg.ring_cap
    toks = np.arange(max(sq, w.s_sink), L)
    if toks.size:
        mm += int(np.sum(snap["ring_k"][b, h, toks % R] != ref["k_rot"][toks]))
        mm += int(np.sum(snap["ring_v"][b, h, toks % R] != ref["v_rot"][toks]))
    rep["window_mismatch"] = mm
    # INT2 region
    axis = 1 if w.key_axis == "channel" else 0
    dec = layout.decode_unit(snap["pages"], run.table[b], h, w.s_sink, sq, w.group_size, w.key_l2norm, axis)
    qk, qv = ref["unit"]["qk"], ref["unit"]["qv"]
    rep["n_codes"] = int(qk["codes"].size + qv["codes"].size)
    rep["code_mismatch"] = int(np.sum(dec["codes_k"] != qk["codes"]) + np.sum(dec["codes_v"] != qv["codes"]))
    same16 = lambda a, b_: int(np.sum(a.view(np.uint16) != np.asarray(b_, np.float16).view(np.uint16)))
    rep["scale_mismatch"] = (same16(dec["delta_k"], qk["delta16"]) + same16(dec["zero_k"], qk["zero16"]) +
                             same16(dec["delta_v"], qv["delta16"]) + same16(dec["zero_v"], qv["zero16"]))
    if w.key_l2norm:
        rep["scale_mismatch"] += same16(dec["norm_k"], qk["norm16"])
    if axis:
        # the page exponent: that of the largest key Delta16 of the page, at least -14
        d = qk["delta16"].astype(np.float64)
        want = np.maximum(np.floor(np.log2(np.maximum(d.max(axis=1), 2.0 ** -30))).astype(np.int64), -14)
        rep["scale_mismatch"] += int(np.sum(dec["exp_k"] != want))
    # attention output: normwise max relative error per query head
    o = snap["out"][b, h * g:(h + 1) * g].astype(np.float64)
    r = ref["out"]
    rel = np.abs(o - r).max(axis=1) / np.maximum(np.abs(r).max(axis=1), 1e-30)
    rep["attn_rel"] = float(rel.max())
    return rep


