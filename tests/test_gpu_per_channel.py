"""GPU parity of per-channel key quantization (KIVI blocks of one 16-token page; values per
token) against the oracle: key codes, per-channel Delta16 / z16, the page exponent and the
token norms bit-exact, the decode output within 2e-3 -- on the OScaR-shaped cache (Hadamard
keys, l2 scaling, S_keep = 0, S_flush = 128), plain orthogonal keys with outlier channels,
clipping quantiles below 1, flush spans of several pages, zero rows and keys spanning many
binades, and split counts."""

import numpy as np
import pytest

import synth
from tests import harness
from tests.test_gpu_parity import _check_units

pytestmark = pytest.mark.gpu

BASE = synth.TINY_GQA4.replace(key_axis="channel", s_flush=16, s_keep=64, s_sink=16, kappa_k=1.0)
CASES = {
    "oscar_hadamard_l2_g32": synth.QWEN3_32B_128K.replace(batch=2, ctx_lo=1100, ctx_hi=1500, n_new=1,
                                                          key_axis="channel"),
    "outlier_channels_g128": BASE.replace(ctx_lo=600, ctx_hi=600, n_new=20),
    "kappa_090_g64_gqa8": BASE.replace(kappa_k=0.90, kappa_v=0.95, group_size=64, n_q_heads=16, n_kv_heads=2,
                                       batch=2, ctx_lo=500, ctx_hi=900),
    "multi_page_spans": BASE.replace(s_flush=48, s_keep=32, ctx_lo=700, ctx_hi=700, n_new=100),
    "invertible_dense_v": BASE.replace(transform="invertible", value_transform="orthogonal", group_size=32,
                                       ctx_lo=400, ctx_hi=400, n_new=40),
    "zero_rows_l2": BASE.replace(key_dist="degenerate", key_l2norm=True, group_size=32, ctx_lo=300, ctx_hi=300),
    "wide_exponent": BASE.replace(key_dist="wide_exponent", transform="identity", group_size=32,
                                  ctx_lo=300, ctx_hi=300),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_per_channel_keys(name):
    w = CASES[name]
    run = harness.DeviceRun(w)
    _check_units(run, [(b, h) for b in range(w.batch) for h in range(w.n_kv_heads)])


@pytest.mark.parametrize("splits", [1, 7])
def test_per_channel_split_invariance(splits):
    w = BASE.replace(ctx_lo=900, ctx_hi=900)
    ref = harness.DeviceRun(w, attn_splits=1).snapshot()["out"]
    run = harness.DeviceRun(w, attn_splits=splits)
    out = run.snapshot()["out"]
    assert np.abs(out - ref).max() / np.abs(ref).max() < 5e-4
    _check_units(run, [(0, 0)])
