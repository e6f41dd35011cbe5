"""kv_append_chunk -- a prefill chunk transformed and quantized on write in one pass -- against
the two-call path on the same rows (kv_rotate_qk at the appended positions, then
kv_quant_flush): every cache byte it writes must be the same, with a ring that holds only
the window.  Then the fused cache against the oracle per (sequence, kv head): codes, scales,
window rows, and the decode output that reads it."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
from tests import harness, parity

pytestmark = pytest.mark.gpu


class AppendRun:
    """A cache prefilled through the two-call path, then one step appending counts[b] rows to
    sequence b -- fused (kv_append_chunk) or not -- with its queries rotated and decoded."""

    def __init__(self, w: synth.Workload, counts, fused: bool, ring_cap: int | None = None, device="cuda",
                 edit_kv=None):
        import bit_rotated_kv_gb300 as kvq
        from bit_rotated_kv_gb300.runner import DecodeRunner, _rows_for
        self.w = w
        dev = torch.device(device)
        self.lengths = synth.context_lengths(w)
        self.counts = np.asarray(counts, np.int64)
        self.after = self.lengths + self.counts
        self.cfg, self.table = harness.kv_config(w, self.lengths + w.n_new)
        if ring_cap is not None:
            self.cfg.ring_cap = ring_cap
        self.tr, self.host_tr = harness.device_transform(w, dev)
        self.runner = DecodeRunner(self.cfg, self.tr, int(self.after.max()), dev)
        self.runner.set_page_table(self.table)
        k_all, v_all = harness.gen_kv(w, self.lengths, dev)
        if edit_kv is not None:
            edit_kv(k_all, v_all)
        q = harness.gen_q(w, dev)
        self.runner.prefill(k_all, v_all, self.lengths, self.cfg.ring_cap - w.s_keep - w.s_flush)
        ib, it = _rows_for(k_all, self.lengths, self.after)
        k, v = k_all[ib, it].contiguous(), v_all[ib, it].contiguous()
        if fused:
            cu = torch.tensor(np.concatenate([[0], np.cumsum(self.counts)]), dtype=torch.int32, device=dev)
            self.runner.step_fused(q, k, v, cu)
        else:
            self.runner.step(q, k, v, ib.to(torch.int32), it.to(torch.int32), int(self.counts.max()))
        torch.cuda.synchronize()
        c = self.runner.cache
        self.snap = {"pages": c.pages.cpu().numpy(), "seq_len": c.seq_len.cpu().numpy(),
                     "s_quant": c.s_quant.cpu().numpy(), "sink_k": harness.bits(c.sink_k),
                     "sink_v": harness.bits(c.sink_v), "ring_k": harness.bits(c.ring_k),
                     "ring_v": harness.bits(c.ring_v), "q_out": harness.bits(self.runner.q_out),
                     "out": self.runner.out.cpu().numpy(), "status": int(self.runner.status.item()),
                     "counters": c.counters.cpu().numpy()}


def _same_cache(a: AppendRun, f: AppendRun):
    sa, sf = a.snap, f.snap
    assert sa["status"] == 0 and sf["status"] == 0, (sa["status"], sf["status"])
    assert np.array_equal(sa["seq_len"], sf["seq_len"]), (sa["seq_len"], sf["seq_len"])
    assert np.array_equal(sa["s_quant"], sf["s_quant"]), (sa["s_quant"], sf["s_quant"])
    assert not sf["counters"].any()
    bad = np.argwhere(sa["pages"] != sf["pages"])
    assert bad.size == 0, (len(bad), bad[:4])
    assert np.array_equal(sa["sink_k"], sf["sink_k"]) and np.array_equal(sa["sink_v"], sf["sink_v"])
    w = a.w
    Ra, Rf = a.cfg.ring_cap, f.cfg.ring_cap
    for b in range(w.batch):
        toks = np.arange(max(int(sa["s_quant"][b]), w.s_sink), int(sa["seq_len"][b]))
        for name in ("ring_k", "ring_v"):
            assert np.array_equal(sa[name][b][:, toks % Ra], sf[name][b][:, toks % Rf]), (name, b)
    assert np.array_equal(sa["q_out"], sf["q_out"])
    assert np.array_equal(sa["out"].view(np.uint32), sf["out"].view(np.uint32))


CASES = {
    # invertible T_K (the chunk workload's transform), values copied, ragged contexts
    "wush_invertible_b3": (synth.WUSH_CHUNK_B16.replace(batch=3, ctx_lo=300, ctx_hi=900, n_new=700,
                                                        chunk_queries=False), None),
    # dense T_V, G = 64, kappa = 0.995; contexts shorter than the sink (rows land in all three places)
    "orth_dense_v_sinks": (synth.WUSH_CHUNK_B16.replace(batch=2, ctx_lo=10, ctx_hi=40, n_new=520,
                                                        transform="orthogonal", value_transform="orthogonal",
                                                        group_size=64, kappa_k=0.995, kappa_v=0.995,
                                                        chunk_queries=False), None),
    # l2-scaled keys, G = 32, min / max, no sink, S_keep = 0, S_flush = 128 (OScaR's windows)
    "l2_g32_flush128": (synth.QWEN3_32B_128K.replace(batch=2, ctx_lo=200, ctx_hi=330, n_new=600,
                                                     transform="orthogonal"), None),
    # QuEST quantizer, S_flush = 1
    "quest_flush1": (synth.WUSH_CHUNK_B16.replace(batch=2, ctx_lo=500, ctx_hi=620, n_new=333, quantizer="quest",
                                                  s_flush=1, chunk_queries=False), None),
    # kappa far from 1 (order statistics by extraction), G = 128
    "kappa_092": (synth.WUSH_CHUNK_B16.replace(batch=2, ctx_lo=280, ctx_hi=290, n_new=410, kappa_k=0.92,
                                               kappa_v=0.95, transform="orthogonal", chunk_queries=False), None),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fused_append_equals_two_call_path_and_oracle(name):
    w, _ = CASES[name]
    counts = np.full(w.batch, w.n_new)
    two = AppendRun(w, counts, fused=False)
    # the fused call needs the ring for the window only
    small_ring = harness.round16(w.s_keep + w.s_flush + 32)
    fused = AppendRun(w, counts, fused=True, ring_cap=small_ring)
    _same_cache(two, fused)
    for b, h in harness.units_sample(w, 3, seed=7):
        rep = parity.compare_unit(fused, fused.snap, b, h)
        assert rep["seq_len_ok"] and rep["s_quant_ok"], rep
        assert rep["window_mismatch"] == 0 and rep["code_mismatch"] == 0 and rep["scale_mismatch"] == 0, rep
        assert rep["q_mismatch"] == 0, rep
        assert rep["attn_rel"] <= 2e-3, rep


def test_fused_append_ragged_counts():
    """Sequences appending different numbers of rows, one appending none."""
    w = synth.WUSH_CHUNK_B16.replace(batch=4, ctx_lo=100, ctx_hi=700, n_new=700, chunk_queries=False)
    counts = np.array([0, 333, 57, 700])
    two = AppendRun(w, counts, fused=False)
    fused = AppendRun(w, counts, fused=True, ring_cap=harness.round16(w.s_keep + w.s_flush + 16))
    _same_cache(two, fused)


def test_fused_append_rejects_hadamard_keys():
    import bit_rotated_kv_gb300 as kvq
    w = synth.QWEN3_32B_128K.replace(batch=1, ctx_lo=16, ctx_hi=16, n_new=32)
    cfg, _ = harness.kv_config(w, [64])
    tr, _ = harness.device_transform(w, torch.device("cuda"))
    cache = kvq.KVCache(cfg, "cuda")
    k = torch.zeros((32, w.n_kv_heads, 128), dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 32], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(kvq.KVQError) as e:
        kvq.kv_append_chunk(cfg, tr, k, k, cu, cache, st)
    assert e.value.code == kvq.KVQ_ERR_UNSUPPORTED
