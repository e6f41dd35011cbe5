"""GPU parity of chunk attention (kv_attn_chunk): the queries of an appended chunk attend
causally to the cache as it stands after the append (BF16 sink, INT2 middle, BF16 ring) --
each row within 2e-3 of the oracle's float64 attention over the same dequantized prefix, on
chunks whose positions fall in the INT2 region and in the ring, per-token and per-channel keys,
l2 keys with Hadamard rotation, a context inside the sink, and ragged rows per sequence."""

import numpy as np
import pytest
import torch

import synth
from oracle import pipeline
from tests import harness

pytestmark = pytest.mark.gpu
ATTN_TOL = 2e-3


def _run(w, counts):
    """Prefill, append counts[b] rows per sequence (two calls), rotate the chunk queries and run
    kv_attn_chunk.  Returns (run, q' bits [rows, Hq, d], out [rows, Hq, d], raw chunk q bits)."""
    from bit_rotated_kv_gb300.runner import _rows_for
    run = harness.DeviceRun(w, do_step=False)
    r = run.runner
    counts = np.asarray(counts)
    ib, it = _rows_for(run.k_all, run.lengths, run.lengths + counts)
    r.append(run.k_all[ib, it].contiguous(), run.v_all[ib, it].contiguous(), ib.to(torch.int32), it.to(torch.int32))
    r.flush(int(counts.max()) + w.s_flush)
    g = w.gqa
    qc = []
    for b in range(w.batch):
        q = np.zeros((w.n_new, w.n_q_heads, w.head_dim), np.uint16)
        for h in range(w.n_kv_heads):
            q[:, h * g:(h + 1) * g] = synth.chunk_query_rows(w, b, h)
        qc.append(q[:counts[b]])
    qc = np.concatenate(qc)
    qd = harness._bf16_dev(qc, run.device)
    qo = torch.empty_like(qd)
    r.append(None, None, None, None, qd, qo)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device=run.device)
    out = torch.full((qc.shape[0], w.n_q_heads, w.head_dim), float("nan"), dtype=torch.float32, device=run.device)
    ws = r.chunk_workspace(qc.shape[0])
    r.attn_chunk(qo, cu, out, ws)
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0, int(r.status.item())
    return run, harness.bits(qo), out.cpu().numpy().astype(np.float64), qc


def _check(w, counts, units):
    run, qrot, out, qc = _run(w, counts)
    g = w.gqa
    starts = np.concatenate([[0], np.cumsum(counts)])
    worst = 0.0
    for b, h in units:
        n = int(counts[b])
        if n == 0:
            continue
        wb = w.replace(n_new=n)
        ui = synth.unit_inputs(w, b, h, run.lengths)        # the rows the harness generated
        rows = slice(int(starts[b]), int(starts[b]) + n)
        ref = pipeline.run_unit_chunk_attention(wb, ui, *run.host_tr, qc[rows, h * g:(h + 1) * g])
        assert np.array_equal(qrot[rows, h * g:(h + 1) * g], ref["q_chunk_rot"]), (b, h)
        o = out[rows, h * g:(h + 1) * g]
        rr = ref["out_chunk"]
        rel = np.abs(o - rr).max(-1) / np.maximum(np.abs(rr).max(-1), 1e-30)
        worst = max(worst, float(rel.max()))
        assert rel.max() <= ATTN_TOL, (b, h, float(rel.max()), np.unravel_index(rel.argmax(), rel.shape))
    return worst


CASES = {
    # WUSH windows (64 / 256 / 8): the chunk's positions reach into the INT2 region and the ring
    "wush_g128": (synth.WUSH_CHUNK_B16.replace(batch=2, ctx_lo=300, ctx_hi=500, n_new=400, chunk_queries=True), None),
    "oscar_hadamard_l2_g32": (synth.QWEN3_32B_128K.replace(batch=2, ctx_lo=700, ctx_hi=900, n_new=300), None),
    "per_channel_keys": (synth.QWEN3_32B_128K.replace(batch=1, ctx_lo=500, ctx_hi=500, n_new=260,
                                                      key_axis="channel"), None),
    "inside_sink": (synth.TINY_GQA4.replace(ctx_lo=3, ctx_hi=3, n_new=10), None),
    "ragged_rows": (synth.WUSH_CHUNK_B16.replace(batch=3, ctx_lo=100, ctx_hi=600, n_new=300, chunk_queries=True),
                    [300, 0, 77]),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_chunk_attention(name):
    w, counts = CASES[name]
    counts = np.full(w.batch, w.n_new) if counts is None else np.asarray(counts)
    units = harness.units_sample(w, 4, seed=13)
    _check(w, counts, units)
