"""Seeded synthetic inputs for the rotated INT2 paged KV cache.

This module is shared by the tests, the bench and the oracle's callers.  It
holds no step of the method itself: it only draws random tensors, rounds them
once to bfloat16, builds the fixed per-head transforms a calibration pass would
hand to the serving path (and their inverse-transpose, which the caller of the
library supplies), and lays out page tables.  Everything is a pure function of
the workload and its seed, drawn from numpy's PCG64 through SeedSequence
sub-streams keyed by (seed, tag, sequence, kv_head), so any (sequence, head)
slice can be regenerated alone.

Workloads follow the head layouts and context lengths of the Qwen3 models the
pages evaluate on (OSCAR summary, section 5 "Experiments"; OScaR note,
"效率基准（H20 GPU）"; WUSH-KV digest, "实验结果").  The models, their weights
and the benchmark suites are not used: the tensors below stand in for them.
"""

from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import numpy as np

# ---- sub-stream tags ---------------------------------------------------------
_TAG_K, _TAG_V, _TAG_Q, _TAG_TK, _TAG_TV, _TAG_LEN, _TAG_OUT, _TAG_PAGES, _TAG_QCHUNK = range(1, 10)


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(k) for k in key]))


# ---- bfloat16 rounding of drawn float32 values (input preparation) -----------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest-even) and return the 16-bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint32)
    nan = np.isnan(x)
    if nan.any():
        r = np.where(nan, (u >> 16).astype(np.uint32) | 0x40, r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---- workloads -----------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    """One synthetic configuration of the hot path.

    ``ctx_lo``/``ctx_hi`` bound the context already in the cache before the
    measured step (inclusive, drawn uniformly per sequence when they differ);
    the measured step then appends ``n_new`` tokens per sequence, flushes, and
    runs one decode step with one query token per sequence.
    """

    name: str
    seed: int
    batch: int
    n_q_heads: int
    n_kv_heads: int
    ctx_lo: int
    ctx_hi: int
    n_new: int
    head_dim: int = 128
    page_size: int = 16
    group_size: int = 128
    kappa_k: float = 0.99
    kappa_v: float = 0.99
    quantizer: str = "affine"          # "affine" (kappa-quantile clipped) | "quest"
    quest_alpha: float = 1.4935705     # outer level (in RMS units) of the MSE-optimal uniform 4-level quantizer of N(0,1)
    key_l2norm: bool = False
    key_axis: str = "token"            # "token" (groups of G channels per token) | "channel" (per channel per page)
    s_sink: int = 64
    s_keep: int = 256
    s_flush: int = 8
    transform: str = "orthogonal"      # "orthogonal" | "hadamard" | "invertible" | "identity"
    value_transform: str = "orthogonal"  # "orthogonal" | "identity"
    key_dist: str = "outlier"          # "outlier" | "fixed_outlier" | "lognormal_norm" | "degenerate" | "wide_exponent"
    outlier_scale: float = 15.0
    n_outlier: int = 2
    fixed_outlier_channels: tuple = ()
    sink_tokens: int = 4
    sink_scale: float = 0.05
    lognormal_sigma: float = 1.5
    low_norm_frac: float = 0.01
    low_norm_scale: float = 0.03
    spd_cond: float = 100.0
    chunk_queries: bool = False        # the appended chunk also carries its queries (prefill-sized rotation)

    @property
    def gqa(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def ring_cap(self) -> int:
        """BF16 recent-window capacity in tokens (multiple of the page size)."""
        need = self.s_keep + self.s_flush + self.n_new
        p = self.page_size
        return max(p, (need + p - 1) // p * p)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The pages' workloads (shapes and distributions follow the hot-path scope table), by name;
# WORKLOADS numbers them for the bench's --config option.
TINY_GQA4 = Workload(name="tiny-gqa4-ctx512", seed=0, batch=1, n_q_heads=4, n_kv_heads=1,
                     ctx_lo=504, ctx_hi=504, n_new=8, group_size=128, kappa_k=0.99, kappa_v=0.99,
                     s_sink=16, s_keep=128, s_flush=8, key_dist="fixed_outlier", outlier_scale=20.0,
                     fixed_outlier_channels=(3, 77))
QWEN3_8B_32K = Workload(name="qwen3-8b-ctx32k-b1", seed=2, batch=1, n_q_heads=32, n_kv_heads=8,
                        ctx_lo=32760, ctx_hi=32760, n_new=8, group_size=128, kappa_k=0.99, kappa_v=0.99)
QWEN3_4B_B64 = Workload(name="qwen3-4b-b64-ctx4k-8k", seed=3, batch=64, n_q_heads=32, n_kv_heads=8,
                        ctx_lo=4096, ctx_hi=8192, n_new=1, group_size=64, kappa_k=0.995, kappa_v=0.995)
QWEN3_32B_128K = Workload(name="qwen3-32b-ctx128k-b4-oscar", seed=4, batch=4, n_q_heads=64, n_kv_heads=8,
                          ctx_lo=131072, ctx_hi=131072, n_new=1, group_size=32, kappa_k=1.0, kappa_v=1.0,
                          key_l2norm=True, s_sink=0, s_keep=0, s_flush=128, transform="hadamard",
                          value_transform="identity", key_dist="lognormal_norm")
WUSH_CHUNK_B16 = Workload(name="wush-qwen3-8b-b16-chunk2048-on-16k", seed=5, batch=16, n_q_heads=32,
                          n_kv_heads=8, ctx_lo=16384, ctx_hi=16384, n_new=2048, group_size=128,
                          kappa_k=0.99, kappa_v=0.99, transform="invertible", value_transform="identity",
                          chunk_queries=True)
# the 128K OScaR cache with KIVI's per-channel keys (Delta, z per channel per 16-token page)
QWEN3_32B_128K_KIVI = QWEN3_32B_128K.replace(name="qwen3-32b-ctx128k-b4-oscar-kivi", seed=6, key_axis="channel")
WORKLOADS: dict[int, Workload] = {1: TINY_GQA4, 2: QWEN3_8B_32K, 3: QWEN3_4B_B64, 4: QWEN3_32B_128K,
                                  5: WUSH_CHUNK_B16, 6: QWEN3_32B_128K_KIVI}


# ---- transforms handed over by offline calibration -----------------------------
def random_orthogonal(d: int, rng: np.random.Generator) -> np.ndarray:
    """Haar-random orthogonal matrix: QR of a Gaussian with the sign fix Q*diag(sign(diag R))."""
    a = rng.standard_normal((d, d))
    q, r = np.linalg.qr(a)
    return q * np.sign(np.diag(r))[None, :]


def spd_invertible(d: int, rng: np.random.Generator, cond: float) -> np.ndarray:
    """A general invertible per-head transform L diag(lam^-1/4) U^T.

    U is random orthogonal, lam is log-spaced in [1, cond], A = U diag(lam) U^T
    is symmetric positive definite and L its Cholesky factor.  This stands in
    for a calibrated WUSH transform, which needs model activations.
    """
    u = random_orthogonal(d, rng)
    lam = np.logspace(0.0, math.log10(cond), d)
    a = (u * lam[None, :]) @ u.T
    a = 0.5 * (a + a.T)
    l = np.linalg.cholesky(a)
    return (l * (lam ** -0.25)[None, :]) @ u.T


def transforms(w: Workload):
    """Return (T_K, T_K^{-T}, T_V) as float32 [Hkv, d, d] arrays (T_V may be None).

    T^{-T} is computed in float64 from the float32-rounded T and then rounded
    once more, so that q'^T k' = q^T k holds to float32 accuracy for any T.
    For "hadamard" the library applies the normalised Walsh-Hadamard transform
    itself and no matrix is passed (None, None).
    """
    d, hkv = w.head_dim, w.n_kv_heads
    if w.transform in ("hadamard",):
        tk = tkit = None
    else:
        tk = np.empty((hkv, d, d), np.float32)
        tkit = np.empty((hkv, d, d), np.float32)
        for h in range(hkv):
            rng = _rng(w.seed, _TAG_TK, h)
            if w.transform == "orthogonal":
                t = random_orthogonal(d, rng)
            elif w.transform == "invertible":
                t = spd_invertible(d, rng, w.spd_cond)
            elif w.transform == "identity":
                t = np.eye(d)
            else:
                raise ValueError(w.transform)
            t32 = t.astype(np.float32)
            tk[h] = t32
            tkit[h] = np.linalg.inv(t32.astype(np.float64)).T.astype(np.float32)
    if w.value_transform == "orthogonal":
        tv = np.empty((hkv, d, d), np.float32)
        for h in range(hkv):
            tv[h] = random_orthogonal(d, _rng(w.seed, _TAG_TV, h)).astype(np.float32)
    elif w.value_transform == "identity":
        tv = None
    else:
        raise ValueError(w.value_transform)
    return tk, tkit, tv


# ---- lengths and pages -----------------------------------------------------------
def context_lengths(w: Workload) -> np.ndarray:
    """Tokens already cached per sequence before the measured step."""
    if w.ctx_lo == w.ctx_hi:
        return np.full(w.batch, w.ctx_lo, np.int64)
    return _rng(w.seed, _TAG_LEN).integers(w.ctx_lo, w.ctx_hi, size=w.batch, endpoint=True).astype(np.int64)


def max_pages_per_seq(w: Workload, total_len: int | None = None) -> int:
    total = (w.ctx_hi + w.n_new) if total_len is None else total_len
    return max(1, -(-max(0, total - w.s_sink) // w.page_size))


def page_table(w: Workload, lengths_after: np.ndarray, spare: int = 0):
    """Seeded random assignment of physical pages: (table [B, max_pages] int32, num_pages).

    Every logical INT2 page a sequence can reach (tokens S_sink.. total) gets a
    distinct physical page; unused table slots hold -1.
    """
    mp = max_pages_per_seq(w, int(lengths_after.max()))
    need = [max(0, -(-max(0, int(n) - w.s_sink) // w.page_size)) for n in lengths_after]
    total = int(sum(need)) + spare
    perm = _rng(w.seed, _TAG_PAGES).permutation(max(total, 1)).astype(np.int32)
    table = np.full((w.batch, mp), -1, np.int32)
    o = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[o:o + n]
        o += n
    return table, max(total, 1)


# ---- K, V, Q rows ----------------------------------------------------------------
def _outlier_channels(w: Workload, h: int) -> np.ndarray:
    if w.key_dist == "fixed_outlier":
        return np.asarray(w.fixed_outlier_channels, np.int64)
    return _rng(w.seed, _TAG_OUT, h).choice(w.head_dim, size=w.n_outlier, replace=False)


def key_rows(w: Workload, b: int, h: int, n_tokens: int) -> np.ndarray:
    """Raw (pre-transform) keys of one (sequence, kv head): bf16 bits [n_tokens, d]."""
    rng = _rng(w.seed, _TAG_K, b, h)
    d = w.head_dim
    if w.key_dist in ("outlier", "fixed_outlier"):
        x = rng.standard_normal((n_tokens, d), dtype=np.float32)
        x[:, _outlier_channels(w, h)] *= np.float32(w.outlier_scale)
        ns = min(w.sink_tokens, n_tokens)
        x[:ns] *= np.float32(w.sink_scale)
    elif w.key_dist == "degenerate":
        # outlier keys plus degenerate rows: tokens 10..17 constant, 18..25 all zero
        x = rng.standard_normal((n_tokens, d), dtype=np.float32)
        x[:, _outlier_channels(w, h)] *= np.float32(w.outlier_scale)
        x[10:18] = np.float32(1.25)
        x[18:26] = np.float32(0.0)
    elif w.key_dist == "lognormal_norm":
        dirs = rng.standard_normal((n_tokens, d), dtype=np.float32)
        dirs /= np.linalg.norm(dirs, axis=1, keepdims=True).astype(np.float32)
        norms = np.exp(rng.standard_normal(n_tokens) * w.lognormal_sigma) * math.sqrt(d)
        n_low = int(round(w.low_norm_frac * n_tokens))
        if n_low:
            low = rng.choice(n_tokens, size=n_low, replace=False)
            norms[low] *= w.low_norm_scale
        x = dirs * norms.astype(np.float32)[:, None]
    elif w.key_dist == "wide_exponent":
        # every token at its own binary scale 2^e, e in [-120, 8]; half the channels of a row
        # pushed down a further 2^0 .. 2^-110, so rows mix normal and tiny magnitudes
        x = rng.standard_normal((n_tokens, d), dtype=np.float32).astype(np.float64)
        e = rng.integers(-120, 9, size=n_tokens)
        f = np.where(rng.random((n_tokens, d)) < 0.5, rng.integers(-110, 1, size=(n_tokens, d)), 0)
        x = np.ldexp(x, e[:, None] + f).astype(np.float32)
    else:
        raise ValueError(w.key_dist)
    return f32_to_bf16_bits(x)


def value_rows(w: Workload, b: int, h: int, n_tokens: int) -> np.ndarray:
    rng = _rng(w.seed, _TAG_V, b, h)
    x = rng.standard_normal((n_tokens, w.head_dim), dtype=np.float32)
    if w.key_dist == "degenerate":
        x[30:36] = np.float32(-0.5)
    return f32_to_bf16_bits(x)


def query_rows(w: Workload, b: int, h: int) -> np.ndarray:
    """Decode-step queries of the g query heads reading kv head h: bf16 bits [g, d]."""
    rng = _rng(w.seed, _TAG_Q, b, h)
    return f32_to_bf16_bits(rng.standard_normal((w.gqa, w.head_dim), dtype=np.float32))


def chunk_query_rows(w: Workload, b: int, h: int) -> np.ndarray:
    """Queries of an appended chunk (prefill-sized rotation): bf16 bits [n_new, g, d]."""
    rng = _rng(w.seed, _TAG_QCHUNK, b, h)
    return f32_to_bf16_bits(rng.standard_normal((w.n_new, w.gqa, w.head_dim), dtype=np.float32))


@dataclass
class UnitInputs:
    """Raw inputs of one (sequence b, kv head h): context + appended tokens."""
    b: int
    h: int
    ctx: int
    k: np.ndarray      # bf16 bits [ctx + n_new, d]
    v: np.ndarray      # bf16 bits [ctx + n_new, d]
    q: np.ndarray      # bf16 bits [g, d]


def unit_inputs(w: Workload, b: int, h: int, lengths: np.ndarray | None = None) -> UnitInputs:
    if lengths is None:
        lengths = context_lengths(w)
    ctx = int(lengths[b])
    n = ctx + w.n_new
    return UnitInputs(b=b, h=h, ctx=ctx, k=key_rows(w, b, h, n), v=value_rows(w, b, h, n),
                      q=query_rows(w, b, h))
