"""kv_attn_decode_noalloc: the decode entry point for callers that cannot allocate device
memory (e.g. inside a framework whose pool owns the device).  It must give what
kv_attn_decode gives with a caller workspace, call after call, while using only the
library's fixed internal scratch.  This file is collected last on purpose."""

import ctypes

import numpy as np
import pytest
import torch

import synth
from tests import harness

pytestmark = pytest.mark.gpu

ATTN_TOL = 2e-3          # the tolerance of the attention parity tests


def _rel(out: torch.Tensor, ref: torch.Tensor) -> float:
    o = out.double().cpu().numpy().reshape(-1, out.shape[-1])
    r = ref.double().cpu().numpy().reshape(-1, ref.shape[-1])
    return float((np.abs(o - r).max(axis=1) / np.maximum(np.abs(r).max(axis=1), 1e-30)).max())


@pytest.mark.parametrize("w", [
    synth.TINY_GQA4,
    synth.TINY_GQA4.replace(n_q_heads=16, n_kv_heads=2, batch=2, ctx_lo=300, ctx_hi=640, group_size=64),
], ids=["config1", "gqa8_b2_g64"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(w):
    import bit_rotated_kv_gb300 as kvq
    run = harness.DeviceRun(w)                 # cache built, one step decoded with a caller workspace
    r = run.runner
    torch.cuda.synchronize()
    ref = r.out.clone()
    assert int(r.status.item()) == 0
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        r.status.zero_()
        kvq.kv_attn_decode_noalloc(r.cfg, r.cache, r.q_out, out, r.sm_scale, r.max_ctx, r.status)
        torch.cuda.synchronize()
        assert int(r.status.item()) == 0, call
        assert torch.isfinite(out).all(), call
        assert _rel(out, ref) <= ATTN_TOL, (call, _rel(out, ref))


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    import bit_rotated_kv_gb300 as kvq
    cfg = kvq.KVConfig(n_q_heads=64, n_kv_heads=8, batch=512, max_pages_per_seq=1 << 16, num_pages=1 << 20,
                       ring_cap=272)
    assert kvq.kv_attn_workspace_bytes(cfg, 1 << 20) > kvq.NOALLOC_WORKSPACE_BYTES
    c = cfg.c()
    fake = kvq.CCache(*([1 << 20] * 9))      # never dereferenced: the size check comes first
    rc = kvq.lib().kv_attn_decode_noalloc(ctypes.byref(c), ctypes.byref(fake), 1 << 20, 1 << 20, 1.0, 1 << 20,
                                          None, None)
    assert rc == kvq.KVQ_ERR_WORKSPACE
