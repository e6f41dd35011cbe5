"""Scale data that overflows float16: every quantizing path reports KVQ_ERR_NONFINITE on the
device status word (include/kvq.h, error codes) -- the decode-size flush (4-warp CTAs), the
prefill-size flush (8-warp CTAs), per-channel keys and the fused chunk append -- and the
oracle's quantizer flags the same rows or blocks.

Planted rows have half their channels at +BIG and half at -BIG (per-channel blocks: the sign
alternates over the block's tokens instead), so a group's range is 2 BIG and Delta = 2 BIG / 3
(2-bit codes, 3 steps; the kappa = 0.99 quantile of such a group is still +-BIG): above the
float16 maximum 65504 for BIG = 3e5, finite for BIG = 6e4, the control that must leave the
status word at zero.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import quant
from tests import harness
from tests.test_gpu_append_chunk import AppendRun

pytestmark = pytest.mark.gpu

KVQ_ERR_NONFINITE = -5
OVER, FINITE = 3.0e5, 6.0e4
BASE = synth.TINY_GQA4.replace(transform="identity", value_transform="identity")
PER_CHANNEL = BASE.replace(key_axis="channel", s_flush=16)


def _row(big: float, sign: float = 1.0) -> np.ndarray:
    r = np.full(BASE.head_dim, sign * big, np.float32)
    r[1::2] = -sign * big
    return r


def _plant(tokens, big, which="k", alternate=False):
    """edit_kv hook: sequence 0, kv head 0, the given token positions of keys or values."""
    def edit(k_all, v_all):
        t = k_all if which == "k" else v_all
        for i, tok in enumerate(tokens):
            sign = -1.0 if (alternate and i % 2) else 1.0
            t[0, tok, 0] = torch.from_numpy(_row(big, sign)).to(torch.bfloat16).to(t.device)
    return edit


def _oracle_token_flag(big: float, kappa: float, group: int) -> bool:
    x = synth.f32_to_bf16_bits(_row(big)[None, :])
    return bool(quant.quantize_rows(x, group, kappa)["nonfinite"][0])


def _oracle_block_flag(big: float, kappa: float) -> bool:
    x = synth.f32_to_bf16_bits(np.stack([_row(big, -1.0 if i % 2 else 1.0) for i in range(16)]))
    return bool(quant.quantize_keys_per_channel(x, 16, kappa)["nonfinite"][0])


# (workload, planted tokens, K or V, per-channel block): tokens 40.. lie in the INT2 region
# after the prefill (s_sink 16, 504 tokens, s_keep 128)
CASES = {
    "flush_decode_size_keys": (BASE, [40], "k", False),
    "flush_decode_size_values": (BASE, [41], "v", False),
    # 8 sequences x 2 kv heads: the prefill flush takes the 8-warp, prefill-size kernel
    "flush_prefill_size_keys": (BASE.replace(batch=8, n_q_heads=8, n_kv_heads=2), [40], "k", False),
    "per_channel_key_block": (PER_CHANNEL, list(range(48, 64)), "k", True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_nonfinite_scales_reported(name):
    w, tokens, which, block = CASES[name]
    kappa = w.kappa_k if which == "k" else w.kappa_v
    for big, expect in ((OVER, KVQ_ERR_NONFINITE), (FINITE, 0)):
        flagged = _oracle_block_flag(big, kappa) if block else _oracle_token_flag(big, kappa, w.group_size)
        assert flagged == (expect != 0), (big, flagged)
        run = harness.DeviceRun(w, do_step=False, edit_kv=_plant(tokens, big, which, alternate=block))
        assert run.status_prefill == expect, (name, big, run.status_prefill)


@pytest.mark.parametrize("fused", [False, True])
def test_nonfinite_scales_reported_on_append(fused):
    """A planted row among 200 appended ones, quantized by the append itself (s_quant moves
    from 376 to 576): through kv_append_chunk, and through kv_rotate_qk + kv_quant_flush."""
    w = BASE.replace(n_new=200)
    pos = int(synth.context_lengths(w)[0]) + 10
    for big, expect in ((OVER, KVQ_ERR_NONFINITE), (FINITE, 0)):
        run = AppendRun(w, [200], fused=fused, edit_kv=_plant([pos], big, "k"))
        assert int(run.snap["s_quant"][0]) > pos
        assert run.snap["status"] == expect, (fused, big, run.snap["status"])
