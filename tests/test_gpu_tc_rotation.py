"""Prefill-sized rotations run their dense rows on the tensor cores (tcgen05): T and x written
as integer digits on a grid common to each dot product, so the tensor cores form exact integer
sums; the CUDA cores combine them, bound what was dropped, and decide each correctly rounded
output, recomputing the rest exactly.  Checked here: the exactness of those integer sums (a
device self-test), and q' rows bit-exact against the oracle at sizes that take that path --
ragged chunk tails, several GQA group sizes, inputs spanning many binades, matrices with
subnormal, tiny or huge entries, and zero rows."""

import numpy as np
import pytest
import torch

import synth
from oracle import transform
from tests import harness

pytestmark = pytest.mark.gpu

# dense (row, head) pairs from which kv_rotate_qk takes the tensor-core path: one 128-row chunk
# per SM of a 152-SM GB300
TC_MIN_PAIRS = 128 * 152


def test_tensor_core_integer_sums_are_exact():
    import bit_rotated_kv_gb300 as kvq
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    kvq.kvq_selftest_tc_integer_sums(bad)
    torch.cuda.synchronize()
    assert int(bad.item()) == 0


def _rotate_queries(x_bits: np.ndarray, tkit: np.ndarray, n_kv_heads: int) -> np.ndarray:
    """x_bits [n, Hq, d] uint16 -> q' bits from kv_rotate_qk with T_K^{-T} = tkit [Hkv, d, d]."""
    import bit_rotated_kv_gb300 as kvq
    n, hq, d = x_bits.shape
    w = synth.TINY_GQA4.replace(n_q_heads=hq, n_kv_heads=n_kv_heads, batch=1)
    dev = torch.device("cuda")
    cfg, _ = harness.kv_config(w, [512])
    t = torch.from_numpy(np.ascontiguousarray(tkit, np.float32)).to(dev)
    tr = kvq.Transform(kvq.KVQ_TRANSFORM_DENSE, t, t, None)
    cache = kvq.KVCache(cfg, dev)
    q = harness._bf16_dev(x_bits, dev)
    q_out = torch.full_like(q, float("nan"))
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    kvq.kv_rotate_qk(cfg, tr, q, q_out, None, None, None, None, cache, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return harness.bits(q_out)


def _oracle_queries(x_bits: np.ndarray, tkit: np.ndarray, n_kv_heads: int) -> np.ndarray:
    n, hq, d = x_bits.shape
    g = hq // n_kv_heads
    out = np.zeros_like(x_bits)
    for h in range(hq):
        out[:, h] = synth.f32_to_bf16_bits(transform.rotate_rows(tkit[h // g], x_bits[:, h]))
    return out


def _check(x_bits, tkit, hkv):
    assert x_bits.shape[0] * x_bits.shape[1] >= TC_MIN_PAIRS
    got = _rotate_queries(x_bits, tkit, hkv)
    ref = _oracle_queries(x_bits, tkit, hkv)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, (len(bad), bad[:5], got[tuple(bad[0])], ref[tuple(bad[0])])


def _gauss_rows(rng, shape, wide=False):
    x = rng.standard_normal(shape)
    if wide:
        x = x * np.exp2(rng.integers(-60, 61, size=shape[:-1] + (1,))) * np.exp2(rng.integers(-8, 9, size=shape))
    return synth.f32_to_bf16_bits(x.astype(np.float32))


@pytest.mark.parametrize("hq,hkv,n", [(32, 8, 650), (8, 8, 2437), (16, 2, 1300), (64, 8, 305)],
                         ids=["gqa4", "gqa1", "gqa8", "gqa8_h64"])
def test_invertible_queries_bit_exact(hq, hkv, n):
    w = synth.WUSH_CHUNK_B16.replace(n_q_heads=hq, n_kv_heads=hkv)
    _, tkit, _ = synth.transforms(w)
    rng = np.random.default_rng(hq * 1000 + n)
    _check(_gauss_rows(rng, (n, hq, 128)), tkit, hkv)


def test_orthogonal_queries_wide_exponents():
    w = synth.QWEN3_8B_32K
    tk, _, _ = synth.transforms(w)
    rng = np.random.default_rng(7)
    _check(_gauss_rows(rng, (700, 32, 128), wide=True), np.ascontiguousarray(tk), 8)


def test_subnormal_matrix_entries():
    """Subnormal float32 entries lie far below their row's largest: truncated at 2^-24 of the
    row's units, inside the bound -- still bit-exact.  One row is scaled by 2^-100 (its units
    follow its own exponent)."""
    w = synth.WUSH_CHUNK_B16
    _, tkit, _ = synth.transforms(w)
    tkit = tkit.copy()
    tkit[3, 5, 7] = np.float32(1e-39)
    tkit[3, 9, 100] = np.float32(-3e-41)
    tkit[6, 0, :] *= np.float32(2.0 ** -100)
    rng = np.random.default_rng(11)
    _check(_gauss_rows(rng, (640, 32, 128)), tkit, 8)


def test_zero_rows_and_zero_matrix_rows():
    w = synth.WUSH_CHUNK_B16
    _, tkit, _ = synth.transforms(w)
    tkit = tkit.copy()
    tkit[2, 17, :] = 0.0
    rng = np.random.default_rng(12)
    x = _gauss_rows(rng, (640, 32, 128))
    x[5] = 0
    x[77, 3] = 0x8000                                          # -0 everywhere in one head
    _check(x, tkit, 8)


def test_huge_matrix_entries_and_tiny_inputs():
    """Entries near 2^100 against inputs near 2^-120, some of them subnormal and some 20 binades
    below their row's largest (digits truncated: the row's bound covers it)."""
    rng = np.random.default_rng(13)
    tkit = (rng.standard_normal((8, 128, 128)) * 2.0 ** 100).astype(np.float32)
    x = rng.standard_normal((640, 32, 128)) * 2.0 ** -120
    x[:, :, ::3] *= 2.0 ** 20
    _check(synth.f32_to_bf16_bits(x.astype(np.float32)), tkit, 8)


def test_hadamard_keys_with_dense_values_at_chunk_size():
    """Hadamard keys and queries (warp items) with a dense T_V large enough for the tensor-core
    kernel: both launches of one call, through the whole step against the oracle."""
    from tests.test_gpu_parity import _check_units
    w = synth.QWEN3_32B_128K.replace(batch=1, ctx_lo=4500, ctx_hi=4500, value_transform="orthogonal")
    run = harness.DeviceRun(w, ring_extra=4096)            # prefill rotates 4096-row chunks
    assert 4096 * w.n_kv_heads >= TC_MIN_PAIRS
    _check_units(run, [(0, h) for h in range(w.n_kv_heads)])
