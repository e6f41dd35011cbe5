"""kv_attn_decode_bf16: the same decode with the output rounded once to bf16.

Checked bit for bit against the float32 output of kv_attn_decode rounded to nearest-even on
the host (the two calls share every step but the final store), and against the oracle's
float64 attention within the float32 bar plus one bf16 rounding (2^-8 of the row's largest
element), on a single-group workload, a batched ragged one and the l2-scaled Hadamard one.
"""

import numpy as np
import pytest
import torch

import synth
from tests import harness, parity

pytestmark = pytest.mark.gpu

ATTN_TOL = 2e-3


def _round_bf16(x: np.ndarray) -> np.ndarray:
    return synth.f32_to_bf16_bits(np.asarray(x, np.float32))


@pytest.mark.parametrize("w", [synth.TINY_GQA4,
                               synth.TINY_GQA4.replace(group_size=64, kappa_k=0.995, kappa_v=0.995, batch=3,
                                                       ctx_lo=300, ctx_hi=700, n_q_heads=16, n_kv_heads=2),
                               synth.QWEN3_32B_128K.replace(batch=1, ctx_lo=3000, ctx_hi=3000)],
                         ids=["tiny", "g64_ragged_gqa8", "l2_hadamard_g32"])
def test_bf16_output_is_rounded_float32_output(w):
    import bit_rotated_kv_gb300 as kvq
    run = harness.DeviceRun(w)
    r = run.runner
    snap = run.snapshot()
    assert snap["status"] == 0
    out16 = torch.zeros(r.out.shape, dtype=torch.bfloat16, device=r.device)
    kvq.kv_attn_decode_bf16(r.cfg, r.cache, r.q_out, out16, r.sm_scale, r.max_ctx, r.ws, r.status)
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    got = harness.bits(out16)
    want = _round_bf16(snap["out"])
    assert np.array_equal(got, want)
    # against the oracle: the float32 bar plus one bf16 rounding
    g = w.gqa
    o16 = synth.bf16_bits_to_f32(got).astype(np.float64)
    for b, h in harness.units_sample(w, 3, seed=7):
        ref = parity.oracle_unit(w, b, h, run.lengths, run.host_tr)["out"]
        o = o16[b, h * g:(h + 1) * g]
        rel = np.abs(o - ref).max(axis=1) / np.abs(ref).max(axis=1)
        assert rel.max() <= ATTN_TOL + 2.0 ** -8, (b, h, rel.max())


def test_bf16_output_rejects_misaligned_out():
    import bit_rotated_kv_gb300 as kvq
    w = synth.TINY_GQA4
    run = harness.DeviceRun(w)
    r = run.runner
    buf = torch.zeros(r.out.numel() + 8, dtype=torch.bfloat16, device=r.device)
    bad = buf[1:1 + r.out.numel()].view(r.out.shape)         # 2-byte aligned only
    with pytest.raises(kvq.KVQError) as e:
        kvq.kv_attn_decode_bf16(r.cfg, r.cache, r.q_out, bad, r.sm_scale, r.max_ctx, r.ws, r.status)
    assert e.value.code == kvq.KVQ_ERR_INVALID_ARG
