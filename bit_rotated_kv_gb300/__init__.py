"""Python binding of the rotated INT2 paged KV-cache library (libkvq.so, sm_103a).

Argument marshalling only: every step of the hot path runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  The shared library is built
in-tree (``bit_rotated_kv_gb300/_build/libkvq.so``, see ``build_lib.py``); importing
this module fails loudly when it is missing -- there is no CPU fallback.

Entry points (same names as the C ABI in include/kvq.h):
  kv_rotate_qk, kv_quant_flush, kv_attn_decode, kv_attn_decode_bf16, kv_attn_workspace_bytes,
  kvq_page_head_bytes, kvq_page_bytes, kvq_status_string
plus ``KVConfig`` / ``KVCache`` helpers that allocate the caller-owned buffers.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkvq.so")

KVQ_OK = 0
KVQ_ERR_INVALID_ARG = -1
KVQ_ERR_UNSUPPORTED = -2
KVQ_ERR_CUDA = -3
KVQ_ERR_BOUNDS = -4
KVQ_ERR_NONFINITE = -5
KVQ_ERR_TIMEOUT = -6
KVQ_ERR_WORKSPACE = -7

KVQ_QUANT_AFFINE_KAPPA = 0
KVQ_QUANT_QUEST_RMS = 1
KVQ_TRANSFORM_DENSE = 0
KVQ_TRANSFORM_HADAMARD = 1
KVQ_KEY_PER_TOKEN = 0
KVQ_KEY_PER_CHANNEL = 1

EXPORTED = ("kv_rotate_qk", "kv_quant_flush", "kv_append_chunk", "kv_attn_chunk", "kv_attn_chunk_workspace_bytes", "kv_attn_decode", "kv_attn_decode_bf16", "kv_attn_decode_noalloc",
            "kv_attn_workspace_bytes",
            "kvq_page_head_bytes", "kvq_page_bytes", "kvq_status_string", "kvq_version",
            "kvq_selftest_scale_division", "kvq_selftest_tc_integer_sums")


class CConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "head_dim", "n_q_heads", "n_kv_heads", "page_size", "group_size", "quantizer", "key_l2norm",
        "s_sink", "s_keep", "s_flush", "ring_cap", "batch", "max_pages_per_seq", "num_pages",
        "attn_splits", "key_axis")] + [("kappa_k", ctypes.c_double), ("kappa_v", ctypes.c_double),
                                       ("quest_alpha", ctypes.c_double)]


class CCache(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "pages", "page_table", "seq_len", "s_quant", "sink_k", "sink_v", "ring_k", "ring_v", "counters")]


class CTransform(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("reserved", ctypes.c_int32), ("t_k", ctypes.c_void_p),
                ("t_k_inv_t", ctypes.c_void_p), ("t_v", ctypes.c_void_p)]


class KVQError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {kvq_status_string(code)} ({code})")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        l = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        P = ctypes.POINTER
        l.kv_rotate_qk.argtypes = [P(CConfig), P(CTransform), vp, vp, i32, vp, vp, vp, vp, i32, P(CCache), vp, vp]
        l.kv_rotate_qk.restype = ctypes.c_int
        l.kv_quant_flush.argtypes = [P(CConfig), P(CCache), i32, vp, vp]
        l.kv_append_chunk.restype = ctypes.c_int
        l.kv_attn_chunk.argtypes = [P(CConfig), P(CCache), vp, vp, i32, vp, ctypes.c_float, i32, vp, sz, vp, vp]
        l.kv_attn_chunk.restype = ctypes.c_int
        l.kv_attn_chunk_workspace_bytes.argtypes = [P(CConfig), i32, i32]
        l.kv_attn_chunk_workspace_bytes.restype = sz
        l.kv_append_chunk.argtypes = [P(CConfig), P(CTransform), vp, vp, vp, i32, P(CCache), vp, vp]
        l.kv_quant_flush.restype = ctypes.c_int
        l.kv_attn_decode.argtypes = [P(CConfig), P(CCache), vp, vp, ctypes.c_float, i32, vp, sz, vp, vp]
        l.kv_attn_decode.restype = ctypes.c_int
        l.kv_attn_decode_bf16.argtypes = [P(CConfig), P(CCache), vp, vp, ctypes.c_float, i32, vp, sz, vp, vp]
        l.kv_attn_decode_bf16.restype = ctypes.c_int
        l.kv_attn_decode_noalloc.argtypes = [P(CConfig), P(CCache), vp, vp, ctypes.c_float, i32, vp, vp]
        l.kv_attn_decode_noalloc.restype = ctypes.c_int
        l.kv_attn_workspace_bytes.argtypes = [P(CConfig), i32]
        l.kv_attn_workspace_bytes.restype = sz
        l.kvq_page_head_bytes.argtypes = [P(CConfig)]
        l.kvq_page_head_bytes.restype = sz
        l.kvq_page_bytes.argtypes = [P(CConfig)]
        l.kvq_page_bytes.restype = sz
        l.kvq_status_string.argtypes = [ctypes.c_int]
        l.kvq_status_string.restype = ctypes.c_char_p
        l.kvq_version.argtypes = []
        l.kvq_version.restype = ctypes.c_int
        l.kvq_selftest_scale_division.argtypes = [vp, vp]
        l.kvq_selftest_scale_division.restype = ctypes.c_int
        l.kvq_selftest_tc_integer_sums.argtypes = [vp, vp]
        l.kvq_selftest_tc_integer_sums.restype = ctypes.c_int
        _lib = l
    return _lib


def kvq_status_string(code: int) -> str:
    return lib().kvq_status_string(int(code)).decode()


def _check(rc: int, where: str) -> None:
    if rc != KVQ_OK:
        raise KVQError(rc, where)


@dataclass
class KVConfig:
    """Python mirror of kvq_config (see include/kvq.h for every field)."""
    n_q_heads: int
    n_kv_heads: int
    batch: int
    max_pages_per_seq: int
    num_pages: int
    ring_cap: int
    head_dim: int = 128
    page_size: int = 16
    group_size: int = 128
    quantizer: int = KVQ_QUANT_AFFINE_KAPPA
    key_l2norm: bool = False
    s_sink: int = 64
    s_keep: int = 256
    s_flush: int = 8
    attn_splits: int = 0
    kappa_k: float = 0.99
    kappa_v: float = 0.99
    quest_alpha: float = 1.4935705
    key_axis: int = 0                    # KVQ_KEY_PER_TOKEN / KVQ_KEY_PER_CHANNEL

    def __setattr__(self, name, value):
        object.__setattr__(self, name, value)
        if name != "_cc":                    # any change rebuilds the C struct on next use
            object.__setattr__(self, "_cc", None)

    def c(self) -> CConfig:
        """The C struct (built once, rebuilt only after a field changes)."""
        cc = self.__dict__.get("_cc")
        if cc is None:
            cc = CConfig(self.head_dim, self.n_q_heads, self.n_kv_heads, self.page_size, self.group_size,
                         self.quantizer, int(bool(self.key_l2norm)), self.s_sink, self.s_keep, self.s_flush,
                         self.ring_cap, self.batch, self.max_pages_per_seq, self.num_pages, self.attn_splits,
                         int(self.key_axis), float(self.kappa_k), float(self.kappa_v), float(self.quest_alpha))
            object.__setattr__(self, "_cc", cc)
        return cc

    @property
    def gqa(self) -> int:
        return self.n_q_heads // self.n_kv_heads


def kvq_page_head_bytes(cfg: KVConfig) -> int:
    c = cfg.c()
    return int(lib().kvq_page_head_bytes(ctypes.byref(c)))


def kvq_page_bytes(cfg: KVConfig) -> int:
    c = cfg.c()
    return int(lib().kvq_page_bytes(ctypes.byref(c)))


def kv_attn_workspace_bytes(cfg: KVConfig, max_ctx: int) -> int:
    c = cfg.c()
    return int(lib().kv_attn_workspace_bytes(ctypes.byref(c), int(max_ctx)))


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        return int(torch.cuda.current_stream().cuda_stream)
    return int(getattr(stream, "cuda_stream", stream))


class KVCache:
    """Caller-owned device buffers of one cache (all zero-initialised; s_quant = s_sink)."""

    def __init__(self, cfg: KVConfig, device="cuda"):
        self.cfg = cfg
        dev = torch.device(device)
        B, H, d = cfg.batch, cfg.n_kv_heads, cfg.head_dim
        phb = kvq_page_head_bytes(cfg)
        if phb == 0:
            raise KVQError(KVQ_ERR_UNSUPPORTED, "KVCache")
        self.page_head_bytes = phb
        self.pages = torch.zeros((cfg.num_pages, H, phb), dtype=torch.uint8, device=dev)
        self.page_table = torch.full((B, cfg.max_pages_per_seq), -1, dtype=torch.int32, device=dev)
        self.seq_len = torch.zeros(B, dtype=torch.int32, device=dev)
        self.s_quant = torch.full((B,), cfg.s_sink, dtype=torch.int32, device=dev)
        ns = max(cfg.s_sink, 1)
        self.sink_k = torch.zeros((B, H, ns, d), dtype=torch.bfloat16, device=dev)
        self.sink_v = torch.zeros((B, H, ns, d), dtype=torch.bfloat16, device=dev)
        self.ring_k = torch.zeros((B, H, cfg.ring_cap, d), dtype=torch.bfloat16, device=dev)
        self.ring_v = torch.zeros((B, H, cfg.ring_cap, d), dtype=torch.bfloat16, device=dev)
        self.counters = torch.zeros(B, dtype=torch.int32, device=dev)

    def __setattr__(self, name, value):
        object.__setattr__(self, name, value)
        if name != "_cc":                    # a replaced buffer rebuilds the C struct on next use
            object.__setattr__(self, "_cc", None)

    def c(self) -> CCache:
        """The C struct of device pointers (built once, rebuilt only after a buffer is replaced)."""
        cc = self.__dict__.get("_cc")
        if cc is None:
            cc = CCache(_ptr(self.pages), _ptr(self.page_table), _ptr(self.seq_len), _ptr(self.s_quant),
                        _ptr(self.sink_k), _ptr(self.sink_v), _ptr(self.ring_k), _ptr(self.ring_v),
                        _ptr(self.counters))
            object.__setattr__(self, "_cc", cc)
        return cc


@dataclass
class Transform:
    """Per-head transforms as device float32 tensors [Hkv, d, d] (or Hadamard)."""
    kind: int = KVQ_TRANSFORM_DENSE
    t_k: torch.Tensor | None = None
    t_k_inv_t: torch.Tensor | None = None
    t_v: torch.Tensor | None = None

    def __setattr__(self, name, value):
        object.__setattr__(self, name, value)
        if name != "_cc":
            object.__setattr__(self, "_cc", None)

    def c(self) -> CTransform:
        """The C struct (built once, rebuilt only after a field changes)."""
        cc = self.__dict__.get("_cc")
        if cc is None:
            cc = CTransform(self.kind, 0, _ptr(self.t_k), _ptr(self.t_k_inv_t), _ptr(self.t_v))
            object.__setattr__(self, "_cc", cc)
        return cc


def kv_rotate_qk(cfg: KVConfig, tr: Transform, q, q_out, k, v, seq_idx, pos, cache: KVCache,
                 status, stream=None) -> None:
    """q [n, Hq, d] -> q_out; k, v [m, Hkv, d] into the cache at (seq_idx[r], pos[r])."""
    c, t = cfg.c(), tr.c()
    n_q = 0 if q is None else int(q.shape[0])
    n_kv = 0 if k is None else int(k.shape[0])
    cc = cache.c()
    rc = lib().kv_rotate_qk(ctypes.byref(c), ctypes.byref(t), _ptr(q), _ptr(q_out), n_q, _ptr(k), _ptr(v),
                            _ptr(seq_idx), _ptr(pos), n_kv, ctypes.byref(cc), _ptr(status), _stream(stream))
    _check(rc, "kv_rotate_qk")


def kv_append_chunk(cfg: KVConfig, tr: Transform, k, v, cu_rows, cache: KVCache, status, stream=None) -> None:
    """k, v [n, Hkv, d]: rows cu_rows[b] .. cu_rows[b+1]-1 appended to sequence b, transformed
    and quantized on write in one pass (the effect of kv_rotate_qk + kv_quant_flush)."""
    c, t = cfg.c(), tr.c()
    n = 0 if k is None else int(k.shape[0])
    cc = cache.c()
    rc = lib().kv_append_chunk(ctypes.byref(c), ctypes.byref(t), _ptr(k), _ptr(v), _ptr(cu_rows), n,
                               ctypes.byref(cc), _ptr(status), _stream(stream))
    _check(rc, "kv_append_chunk")


def kv_attn_chunk_workspace_bytes(cfg: KVConfig, n_rows: int, max_ctx: int) -> int:
    return int(lib().kv_attn_chunk_workspace_bytes(ctypes.byref(cfg.c()), int(n_rows), int(max_ctx)))


def kv_attn_chunk(cfg: KVConfig, cache: KVCache, q_rot, cu_rows, out, sm_scale: float, max_ctx: int, workspace,
                  status, stream=None) -> None:
    """q_rot [n, Hq, d] (rows cu_rows[b] .. cu_rows[b+1]-1 the last tokens of sequence b) ->
    out [n, Hq, d] float32: causal attention over the cache after the append."""
    n = int(q_rot.shape[0])
    c, cc = cfg.c(), cache.c()
    rc = lib().kv_attn_chunk(ctypes.byref(c), ctypes.byref(cc), _ptr(q_rot), _ptr(cu_rows), n, _ptr(out),
                             float(sm_scale), int(max_ctx), _ptr(workspace), int(workspace.numel()), _ptr(status),
                             _stream(stream))
    _check(rc, "kv_attn_chunk")


def kv_quant_flush(cfg: KVConfig, cache: KVCache, max_tokens_per_seq: int, status, stream=None) -> None:
    c, cc = cfg.c(), cache.c()
    rc = lib().kv_quant_flush(ctypes.byref(c), ctypes.byref(cc), int(max_tokens_per_seq), _ptr(status),
                              _stream(stream))
    _check(rc, "kv_quant_flush")


def kv_attn_decode(cfg: KVConfig, cache: KVCache, q_rot, out, sm_scale: float, max_ctx: int, workspace,
                   status, stream=None) -> None:
    c, cc = cfg.c(), cache.c()
    nbytes = int(workspace.numel() * workspace.element_size())
    rc = lib().kv_attn_decode(ctypes.byref(c), ctypes.byref(cc), _ptr(q_rot), _ptr(out), float(sm_scale),
                              int(max_ctx), _ptr(workspace), nbytes, _ptr(status), _stream(stream))
    _check(rc, "kv_attn_decode")


def kv_attn_decode_bf16(cfg: KVConfig, cache: KVCache, q_rot, out, sm_scale: float, max_ctx: int, workspace,
                        status, stream=None) -> None:
    """kv_attn_decode with a bf16 output tensor [B, Hq, d] (the float32 result rounded once)."""
    c, cc = cfg.c(), cache.c()
    nbytes = int(workspace.numel() * workspace.element_size())
    rc = lib().kv_attn_decode_bf16(ctypes.byref(c), ctypes.byref(cc), _ptr(q_rot), _ptr(out), float(sm_scale),
                                   int(max_ctx), _ptr(workspace), nbytes, _ptr(status), _stream(stream))
    _check(rc, "kv_attn_decode_bf16")


NOALLOC_WORKSPACE_BYTES = 8 << 20


def kv_attn_decode_noalloc(cfg: KVConfig, cache: KVCache, q_rot, out, sm_scale: float, max_ctx: int, status,
                           stream=None) -> None:
    """kv_attn_decode with the library's fixed internal scratch (no workspace argument)."""
    c, cc = cfg.c(), cache.c()
    rc = lib().kv_attn_decode_noalloc(ctypes.byref(c), ctypes.byref(cc), _ptr(q_rot), _ptr(out), float(sm_scale),
                                      int(max_ctx), _ptr(status), _stream(stream))
    _check(rc, "kv_attn_decode_noalloc")


def kvq_selftest_scale_division(mismatches, stream=None) -> None:
    """Device self-check of the quantizer's scale division against IEEE division; adds the
    number of differing results to `mismatches` (a zeroed int64 device tensor of one element)."""
    rc = lib().kvq_selftest_scale_division(_ptr(mismatches), _stream(stream))
    _check(rc, "kvq_selftest_scale_division")


def kvq_selftest_tc_integer_sums(mismatches, stream=None) -> None:
    """Device self-check that the tensor cores add the rotation's integer digit products exactly;
    adds the number of differing sums to `mismatches` (a zeroed int64 device tensor of one
    element)."""
    rc = lib().kvq_selftest_tc_integer_sums(_ptr(mismatches), _stream(stream))
    _check(rc, "kvq_selftest_tc_integer_sums")


def workspace(cfg: KVConfig, max_ctx: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace tensor for kv_attn_decode."""
    n = kv_attn_workspace_bytes(cfg, max_ctx)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)
