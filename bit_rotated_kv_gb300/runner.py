"""Drive the C-ABI calls for a batch of sequences: chunked prefill of the cache and one
serving step (append n_new tokens, flush, decode -- or the fused append, then decode).  Argument marshalling only --
torch is used for device buffers, gathers of input rows and streams; every step of the
method runs in the library's kernels."""

from __future__ import annotations

import math

import numpy as np
import torch

from . import (KVCache, KVConfig, Transform, kv_append_chunk, kv_attn_chunk, kv_attn_chunk_workspace_bytes,
               kv_attn_decode, kv_quant_flush, kv_rotate_qk, workspace)


def _rows_for(k_all: torch.Tensor, lengths_lo, lengths_hi):
    """Gather rows [lo_b, hi_b) of every sequence from k_all [B, T, H, d] into [rows, H, d]
    plus int32 seq_idx / pos on the same device."""
    idx_b, idx_t = [], []
    for b, (lo, hi) in enumerate(zip(lengths_lo, lengths_hi)):
        if hi > lo:
            idx_b.append(np.full(hi - lo, b, np.int64))
            idx_t.append(np.arange(lo, hi, dtype=np.int64))
    if not idx_b:
        return None, None
    ib = torch.from_numpy(np.concatenate(idx_b)).to(k_all.device)
    it = torch.from_numpy(np.concatenate(idx_t)).to(k_all.device)
    return ib, it


class DecodeRunner:
    """Owns one cache plus the scratch of a decode step.

    Calls go to ``stream`` (default: the current stream of ``device`` when the runner is
    made, resolved once); a method's own ``stream`` argument overrides it for that call."""

    def __init__(self, cfg: KVConfig, transform: Transform, max_ctx: int, device="cuda", stream=None):
        self.cfg = cfg
        self.tr = transform
        self.device = torch.device(device)
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        self.stream = int(getattr(stream, "cuda_stream", stream))
        self.cache = KVCache(cfg, device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.max_ctx = int(max_ctx)
        self.ws = workspace(cfg, self.max_ctx, device)
        self.q_out = torch.empty((cfg.batch, cfg.n_q_heads, cfg.head_dim), dtype=torch.bfloat16,
                                 device=self.device)
        self.out = torch.empty((cfg.batch, cfg.n_q_heads, cfg.head_dim), dtype=torch.float32,
                               device=self.device)
        self.sm_scale = 1.0 / math.sqrt(cfg.head_dim)

    def set_page_table(self, table: np.ndarray) -> None:
        self.cache.page_table.copy_(torch.from_numpy(np.ascontiguousarray(table, np.int32)))

    def append(self, k_rows, v_rows, seq_idx, pos, q=None, q_out=None, stream=None) -> None:
        kv_rotate_qk(self.cfg, self.tr, q, q_out, k_rows, v_rows, seq_idx, pos, self.cache, self.status,
                     self.stream if stream is None else stream)

    def append_chunk(self, k_rows, v_rows, cu_rows, stream=None) -> None:
        """Rows cu_rows[b] .. cu_rows[b+1]-1 of k_rows / v_rows appended to sequence b, transformed
        and quantized on write in one pass (seq_len and s_quant advance)."""
        kv_append_chunk(self.cfg, self.tr, k_rows, v_rows, cu_rows, self.cache, self.status,
                        self.stream if stream is None else stream)

    def flush(self, max_tokens: int, stream=None) -> None:
        kv_quant_flush(self.cfg, self.cache, max_tokens, self.status, self.stream if stream is None else stream)

    def decode(self, q_rot, out, stream=None) -> None:
        kv_attn_decode(self.cfg, self.cache, q_rot, out, self.sm_scale, self.max_ctx, self.ws, self.status,
                       self.stream if stream is None else stream)

    def chunk_workspace(self, n_rows: int) -> torch.Tensor:
        """A zeroed workspace for kv_attn_chunk over n_rows query rows."""
        n = kv_attn_chunk_workspace_bytes(self.cfg, n_rows, self.max_ctx)
        return torch.zeros(max(n, 256), dtype=torch.uint8, device=self.device)

    def attn_chunk(self, q_rot, cu_rows, out, ws, stream=None) -> None:
        """Causal attention of chunk query rows q_rot [n, Hq, d] over the cache (after their
        tokens were appended) into out [n, Hq, d] float32."""
        kv_attn_chunk(self.cfg, self.cache, q_rot, cu_rows, out, self.sm_scale, self.max_ctx, ws, self.status,
                      self.stream if stream is None else stream)

    def prefill(self, k_all: torch.Tensor, v_all: torch.Tensor, lengths, chunk: int) -> None:
        """Append tokens [0, lengths[b]) of k_all / v_all [B, T, Hkv, d] (bf16, device) in chunks,
        flushing after each chunk."""
        lengths = [int(x) for x in lengths]
        T = max(lengths) if lengths else 0
        for c0 in range(0, T, chunk):
            lo = [min(c0, L) for L in lengths]
            hi = [min(c0 + chunk, L) for L in lengths]
            ib, it = _rows_for(k_all, lo, hi)
            if ib is None:
                continue
            k = k_all[ib, it].contiguous()
            v = v_all[ib, it].contiguous()
            self.append(k, v, ib.to(torch.int32), it.to(torch.int32))
            self.flush(chunk + self.cfg.s_flush)

    def step_inputs(self, k_all, v_all, ctx, n_new: int):
        """(k_rows, v_rows, seq_idx, pos) of the n_new tokens after ctx[b] of every sequence."""
        ctx = [int(x) for x in ctx]
        ib, it = _rows_for(k_all, ctx, [c + n_new for c in ctx])
        return (k_all[ib, it].contiguous(), v_all[ib, it].contiguous(), ib.to(torch.int32),
                it.to(torch.int32))

    def step_fused(self, q, k_rows, v_rows, cu_rows, stream=None) -> None:
        """The same serving step with the appended chunk transformed and quantized in one pass:
        append, rotate the queries, decode."""
        self.append_chunk(k_rows, v_rows, cu_rows, stream)
        kv_rotate_qk(self.cfg, self.tr, q, self.q_out, None, None, None, None, self.cache, self.status,
                     self.stream if stream is None else stream)
        self.decode(self.q_out, self.out, stream)

    def step(self, q, k_rows, v_rows, seq_idx, pos, n_new: int, stream=None) -> None:
        """One serving step: rotate the new rows and the queries, flush, decode."""
        self.append(k_rows, v_rows, seq_idx, pos, q, self.q_out, stream)
        self.flush(n_new + self.cfg.s_flush, stream)
        self.decode(self.q_out, self.out, stream)
