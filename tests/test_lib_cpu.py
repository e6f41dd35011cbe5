"""The C-ABI library without a GPU: it loads, exports exactly the symbols include/kvq.h
declares, and rejects bad arguments on the host before any CUDA call."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def kvq():
    import bit_rotated_kv_gb300 as m
    if not os.path.exists(m.LIB_PATH):
        from bit_rotated_kv_gb300 import build_lib
        build_lib.build()
    m.lib()
    return m


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^KVQ_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_three_calls():
    syms = declared_symbols()
    for s in ("kv_rotate_qk", "kv_quant_flush", "kv_attn_decode"):
        assert s in syms


def test_exports_match_header(kvq):
    out = subprocess.run(["nm", "-D", "--defined-only", kvq.LIB_PATH], capture_output=True, text=True).stdout
    exported = sorted({line.split()[-1] for line in out.splitlines() if " T " in line})
    assert exported == declared_symbols()
    for s in declared_symbols():
        assert hasattr(kvq.lib(), s)


def _cfg(kvq, **kw):
    base = dict(n_q_heads=32, n_kv_heads=8, batch=2, max_pages_per_seq=64, num_pages=128, ring_cap=272)
    base.update(kw)
    return kvq.KVConfig(**base)


def test_sizes(kvq):
    c = _cfg(kvq)
    assert kvq.kvq_page_head_bytes(c) == 1152             # 512 + 512 + 16*1*4*2
    assert kvq.kvq_page_bytes(c) == 8 * 1152
    assert kvq.kvq_page_head_bytes(_cfg(kvq, group_size=64)) == 1280
    assert kvq.kvq_page_head_bytes(_cfg(kvq, group_size=32, key_l2norm=True)) == 1568
    # per-channel keys: d Delta16 + d z16 instead of 16 x d/G pairs, plus the page exponent
    assert kvq.kvq_page_head_bytes(_cfg(kvq, group_size=32, key_l2norm=True, key_axis=1, s_flush=128, s_keep=0)) == 1856
    assert kvq.kv_attn_workspace_bytes(c, 4096) > 0
    assert kvq.kvq_page_head_bytes(_cfg(kvq, head_dim=64)) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=64), -2), (dict(group_size=16), -2), (dict(n_q_heads=12, n_kv_heads=8), -1),
    (dict(n_q_heads=24, n_kv_heads=2), -2), (dict(kappa_k=0.3), -1), (dict(kappa_v=1.5), -1),
    (dict(ring_cap=100), -1), (dict(ring_cap=16), -1), (dict(s_flush=0), -1),
    (dict(quantizer=1, key_l2norm=True), -2), (dict(quantizer=7), -1), (dict(batch=0), -1),
    (dict(key_axis=2), -1), (dict(key_axis=1, s_flush=8), -2), (dict(key_axis=1, s_flush=16, quantizer=1), -2),
])
def test_config_validation(kvq, kw, code):
    c = _cfg(kvq, **kw).c()
    cache = kvq.CCache()
    rc = kvq.lib().kv_quant_flush(ctypes.byref(c), ctypes.byref(cache), 8, None, None)
    assert rc == code


def test_null_cache_and_workspace_checks(kvq):
    c = _cfg(kvq).c()
    cache = kvq.CCache()                              # all NULL
    assert kvq.lib().kv_quant_flush(ctypes.byref(c), ctypes.byref(cache), 8, None, None) == -1
    assert kvq.lib().kv_attn_decode(ctypes.byref(c), None, None, None, 1.0, 10, None, 0, None, None) == -1
    fake = kvq.CCache(*([4096] * 9))                  # non-null, aligned host addresses (never dereferenced)
    rc = kvq.lib().kv_attn_decode(ctypes.byref(c), ctypes.byref(fake), 4096, 4096, 1.0, 4096, 4096, 16,
                                  None, None)
    assert rc == -7                                   # workspace too small: rejected before launch
    rc = kvq.lib().kv_attn_decode(ctypes.byref(c), ctypes.byref(fake), 4100, 4096, 1.0, 4096, 4096, 1 << 30,
                                  None, None)
    assert rc == -1                                   # misaligned query pointer


def test_rotate_validation(kvq):
    c = _cfg(kvq).c()
    t = kvq.CTransform(5, 0, None, None, None)
    assert kvq.lib().kv_rotate_qk(ctypes.byref(c), ctypes.byref(t), None, None, 0, None, None, None, None, 0,
                                  None, None, None) == -1
    t = kvq.CTransform(0, 0, None, None, None)
    # queries without T^{-T}
    assert kvq.lib().kv_rotate_qk(ctypes.byref(c), ctypes.byref(t), 4096, 4096, 1, None, None, None, None, 0,
                                  None, None, None) == -1
    # nothing to do: returns OK without touching the device
    assert kvq.lib().kv_rotate_qk(ctypes.byref(c), ctypes.byref(t), None, None, 0, None, None, None, None, 0,
                                  None, None, None) == 0
    assert kvq.lib().kv_rotate_qk(ctypes.byref(c), ctypes.byref(t), None, None, -1, None, None, None, None, 0,
                                  None, None, None) == -1
    # rows are read 16 bytes at a time: an 8-byte aligned query or key pointer is rejected on the host
    t = kvq.CTransform(0, 0, 4096, 4096, None)
    fake = kvq.CCache(*([4096] * 9))
    assert kvq.lib().kv_rotate_qk(ctypes.byref(c), ctypes.byref(t), 4104, 4096, 1, None, None, None, None, 0,
                                  ctypes.byref(fake), None, None) == -1
    assert kvq.lib().kv_rotate_qk(ctypes.byref(c), ctypes.byref(t), None, None, 0, 4104, 4096, 4096, 4096, 1,
                                  ctypes.byref(fake), None, None) == -1


def test_selftest_rejects_null(kvq):
    assert kvq.lib().kvq_selftest_scale_division(None, None) == -1
    assert kvq.lib().kvq_selftest_tc_integer_sums(None, None) == -1


def test_status_strings(kvq):
    for code in range(0, -8, -1):
        assert kvq.kvq_status_string(code) != "unknown status"
    assert kvq.lib().kvq_version() == 100


def test_append_chunk_validation(kvq):
    """kv_append_chunk's host checks, before any launch (fake device addresses are never used)."""
    c = _cfg(kvq).c()
    fake = kvq.CCache(*([4096] * 9))
    had = kvq.CTransform(1, 0, None, None, None)
    dense = kvq.CTransform(0, 0, 4096, 4096, None)
    # Hadamard keys are not fused (their exact butterflies stay on the two-call path)
    assert kvq.lib().kv_append_chunk(ctypes.byref(c), ctypes.byref(had), 4096, 4096, 4096, 1,
                                     ctypes.byref(fake), None, None) == -2
    # per-channel keys are not fused either
    cp = _cfg(kvq, key_axis=1, s_flush=16).c()
    assert kvq.lib().kv_append_chunk(ctypes.byref(cp), ctypes.byref(dense), 4096, 4096, 4096, 1,
                                     ctypes.byref(fake), None, None) == -2
    # missing cu_rows, misaligned rows, negative count
    assert kvq.lib().kv_append_chunk(ctypes.byref(c), ctypes.byref(dense), 4096, 4096, None, 1,
                                     ctypes.byref(fake), None, None) == -1
    assert kvq.lib().kv_append_chunk(ctypes.byref(c), ctypes.byref(dense), 4104, 4096, 4096, 1,
                                     ctypes.byref(fake), None, None) == -1
    assert kvq.lib().kv_append_chunk(ctypes.byref(c), ctypes.byref(dense), 4096, 4096, 4096, -1,
                                     ctypes.byref(fake), None, None) == -1


def test_attn_chunk_validation(kvq):
    """kv_attn_chunk's host checks: row limit, workspace size, alignment, empty calls."""
    c = _cfg(kvq).c()
    fake = kvq.CCache(*([4096] * 9))
    lib = kvq.lib()
    need = lib.kv_attn_chunk_workspace_bytes(ctypes.byref(c), 64, 4096)
    assert need > lib.kv_attn_workspace_bytes(ctypes.byref(c), 4096)   # 64 rows vs 2 sequences
    assert lib.kv_attn_chunk_workspace_bytes(ctypes.byref(c), 70000, 4096) == 0
    call = lambda q, cu, n, out, ws, nbytes: lib.kv_attn_chunk(ctypes.byref(c), ctypes.byref(fake), q, cu, n, out,
                                                               ctypes.c_float(0.1), 4096, ws, nbytes, None, None)
    assert call(4096, 4096, 0, 4096, None, 0) == 0                   # nothing to do
    assert call(4096, 4096, 70000, 4096, 4096, 1 << 40) == -2        # one grid row per query row
    assert call(4096, None, 64, 4096, 4096, 1 << 40) == -1           # no cu_rows
    assert call(4096, 4096, 64, 4096, 4096, 16) == -7                # workspace too small
    assert call(4104, 4096, 64, 4096, 4096, 1 << 40) == -1           # misaligned queries
