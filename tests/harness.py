"""GPU-side harness: build a workload's cache through the C ABI, run the measured step and
read everything back.  Imports nothing from the oracle (the bench's GPU arm uses it);
the comparisons with the oracle live in tests/parity.py."""

from __future__ import annotations

import math

import numpy as np
import torch

import synth


def round16(x: int) -> int:
    return (x + 15) // 16 * 16


def kv_config(w: synth.Workload, lengths_after, ring_extra: int = 1024, attn_splits: int = 0):
    import bit_rotated_kv_gb300 as kvq
    table, num_pages = synth.page_table(w, np.asarray(lengths_after))
    ring = round16(w.s_keep + w.s_flush + max(w.n_new, ring_extra))
    cfg = kvq.KVConfig(
        n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, batch=w.batch, max_pages_per_seq=table.shape[1],
        num_pages=num_pages, ring_cap=ring, group_size=w.group_size,
        quantizer=kvq.KVQ_QUANT_QUEST_RMS if w.quantizer == "quest" else kvq.KVQ_QUANT_AFFINE_KAPPA,
        key_l2norm=w.key_l2norm, s_sink=w.s_sink, s_keep=w.s_keep, s_flush=w.s_flush,
        attn_splits=attn_splits, kappa_k=w.kappa_k, kappa_v=w.kappa_v, quest_alpha=w.quest_alpha,
        key_axis=kvq.KVQ_KEY_PER_CHANNEL if w.key_axis == "channel" else kvq.KVQ_KEY_PER_TOKEN)
    return cfg, table


def device_transform(w: synth.Workload, device):
    import bit_rotated_kv_gb300 as kvq
    tk, tkit, tv = synth.transforms(w)
    dev = lambda a: None if a is None else torch.from_numpy(a).to(device)
    kind = kvq.KVQ_TRANSFORM_HADAMARD if w.transform == "hadamard" else kvq.KVQ_TRANSFORM_DENSE
    return kvq.Transform(kind, dev(tk), dev(tkit), dev(tv)), (tk, tkit, tv)


def _bf16_dev(a: np.ndarray, device):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def gen_kv(w: synth.Workload, lengths, device):
    """k_all, v_all: bf16 [B, T, Hkv, d] on device (rows beyond a sequence are zero)."""
    T = int(max(lengths)) + w.n_new
    k = np.zeros((w.batch, T, w.n_kv_heads, w.head_dim), np.uint16)
    v = np.zeros_like(k)
    for b in range(w.batch):
        n = int(lengths[b]) + w.n_new
        for h in range(w.n_kv_heads):
            k[b, :n, h] = synth.key_rows(w, b, h, n)
            v[b, :n, h] = synth.value_rows(w, b, h, n)
    return _bf16_dev(k, device), _bf16_dev(v, device)


def gen_q(w: synth.Workload, device):
    g = w.gqa
    q = np.zeros((w.batch, w.n_q_heads, w.head_dim), np.uint16)
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            q[b, h * g:(h + 1) * g] = synth.query_rows(w, b, h)
    return _bf16_dev(q, device)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceRun:
    """The workload's cache built through the library, then one measured step."""

    def __init__(self, w: synth.Workload, device="cuda", attn_splits=0, ring_extra=1024, do_step=True,
                 pool_fill=None, edit_kv=None):
        import bit_rotated_kv_gb300 as kvq
        from bit_rotated_kv_gb300.runner import DecodeRunner
        self.w = w
        self.device = torch.device(device)
        self.lengths = synth.context_lengths(w)
        self.after = self.lengths + w.n_new
        self.cfg, self.table = kv_config(w, self.after, ring_extra, attn_splits)
        self.tr, self.host_tr = device_transform(w, self.device)
        self.runner = DecodeRunner(self.cfg, self.tr, int(self.after.max()), self.device)
        self.runner.set_page_table(self.table)
        if pool_fill is not None:       # a pool that was never cleared: every byte pool_fill
            self.runner.cache.pages.fill_(pool_fill)
        self.k_all, self.v_all = gen_kv(w, self.lengths, self.device)
        if edit_kv is not None:         # planted rows (inputs the generator does not draw)
            edit_kv(self.k_all, self.v_all)
        self.q = gen_q(w, self.device)
        chunk = self.cfg.ring_cap - w.s_keep - w.s_flush
        self.runner.prefill(self.k_all, self.v_all, self.lengths, chunk)
        torch.cuda.synchronize()
        self.status_prefill = int(self.runner.status.item())
        if do_step:
            self.step_in = self.runner.step_inputs(self.k_all, self.v_all, self.lengths, w.n_new)
            self.runner.step(self.q, *self.step_in, n_new=w.n_new)
            torch.cuda.synchronize()
        self.kvq = kvq

    # ---- read-back ------------------------------------------------------------------
    def snapshot(self) -> dict:
        c = self.runner.cache
        return {"pages": c.pages.cpu().numpy(), "seq_len": c.seq_len.cpu().numpy(),
                "s_quant": c.s_quant.cpu().numpy(), "sink_k": bits(c.sink_k), "sink_v": bits(c.sink_v),
                "ring_k": bits(c.ring_k), "ring_v": bits(c.ring_v), "q_out": bits(self.runner.q_out),
                "out": self.runner.out.cpu().numpy(), "status": int(self.runner.status.item())}


def units_sample(w: synth.Workload, n: int, seed: int = 0):
    rng = np.random.default_rng(seed)
    all_units = [(b, h) for b in range(w.batch) for h in range(w.n_kv_heads)]
    if len(all_units) <= n:
        return all_units
    idx = rng.choice(len(all_units), size=n, replace=False)
    return [all_units[i] for i in sorted(idx)]
