"""Seeded random configurations through the whole step (append, flush, decode) against the
oracle: shapes, quantizer, windows, transforms and key distributions drawn together, so that
combinations no hand-written case names are exercised too.  Every (sequence, kv head) unit
is compared (codes, scales, norms, windows and q' bit-exact; attention <= 2e-3)."""

import numpy as np
import pytest

import synth
from tests import harness
from tests.test_gpu_parity import _check_units

pytestmark = pytest.mark.gpu


def random_workload(seed: int) -> synth.Workload:
    rng = np.random.default_rng(1000 + seed)
    hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 4, 8]))
    quantizer = str(rng.choice(["affine", "affine", "quest"]))
    l2 = bool(quantizer == "affine" and rng.random() < 0.3)
    s_sink = int(rng.choice([0, 4, 16, 64]))
    s_keep = int(rng.choice([0, 16, 48, 128]))
    s_flush = int(rng.choice([1, 8, 16, 128]))
    ctx_hi = int(rng.integers(1, 900))
    return synth.Workload(
        name=f"random-{seed}", seed=100 + seed, batch=int(rng.integers(1, 4)), n_q_heads=hkv * g, n_kv_heads=hkv,
        ctx_lo=int(rng.integers(0, ctx_hi + 1)), ctx_hi=ctx_hi, n_new=int(rng.choice([1, 3, 17, 40, 100])),
        group_size=int(rng.choice([32, 64, 128])), kappa_k=float(rng.choice([1.0, 0.99, 0.95, 0.9])),
        kappa_v=float(rng.choice([1.0, 0.99, 0.95])), quantizer=quantizer, key_l2norm=l2,
        s_sink=s_sink, s_keep=s_keep, s_flush=s_flush,
        transform=str(rng.choice(["orthogonal", "hadamard", "invertible", "identity"])),
        value_transform=str(rng.choice(["orthogonal", "identity"])),
        key_dist=str(rng.choice(["outlier", "lognormal_norm", "degenerate", "wide_exponent"])))


@pytest.mark.parametrize("seed", range(24))
def test_random_configuration(seed):
    w = random_workload(seed)
    run = harness.DeviceRun(w)
    _check_units(run, [(b, h) for b in range(w.batch) for h in range(w.n_kv_heads)])
