"""Quantize-on-write: per-token, per-group INT2 codes with a scale and a zero point.

Oracle module (test infrastructure only).  Steps, in the pages' order:

1. Optional l2 token scaling of keys, after the rotation ([OScaR] "步骤二：
   Omni-Token Scaling"; ordering rule in "正确的修复顺序"):
   s = ||k'||_2, y = k' / s, and s is stored beside the codes.  Here s is the
   float64 square root of the float64 sum of squares (exact for BF16 inputs of
   moderate dynamic range), stored as float16; y = fp32(k') / fp32(s16) with one
   IEEE float32 division.  A zero row keeps s16 = 0 and y = 0.
2. Group range, per token and per group of G channels ([OSCAR] section 3
   "Scale Determination and Clipping" and appendix A.5, per-token per-group
   with percentile clipping; [WUSH] "方法步骤详情", kappa-quantile clipped
   affine scale and zero point).  Reading taken: two-sided, hi = the
   kappa-quantile and lo = the (1-kappa)-quantile of the group's own values,
   linear interpolation between order statistics: sorted a[0..G-1],
   pos = (G-1)*kappa in float64, i = floor(pos), f = fp32(pos - i),
   q = a[i] + f*(a[i+1] - a[i]) with float32 operations (q = a[G-1] if
   i = G-1).  kappa = 1 gives min / max.
3. Scale and zero point ([OScaR] "整数量化基础": Delta = (max - min)/(2^b - 1);
   "背景：KIVI": z = -min/Delta).  Delta = (hi - lo)/3 in float32, stored as
   Delta16 = fp16(Delta) (Delta16 := 1 when it rounds to 0); z = -(lo/Delta16)
   in float32, stored as z16 = fp16(z).
   QuEST variant ([WUSH] "方法步骤详情", Delta = 2 alpha ||x|| / (sqrt(d)(2^b-1))
   read per group: rms = ||x_group|| / sqrt(G)): Delta16 = fp16(2*alpha*rms/3)
   from float64, z16 = 1.5, i.e. the symmetric mid-rise grid Delta (c - 1.5)
   spanning +-alpha*rms.
4. Codes ([OScaR] "整数量化基础": Q(x) = clamp(round(x/Delta + z), 0, 2^b - 1)):
   u = fp32(y / Delta16) + fp32(z16) (two float32 operations), c = clamp(
   round_half_even(u), 0, 3).  Computed from the stored Delta16 and z16, so
   dequantisation x_hat = Delta16 (c - z16) (times s16 for l2-scaled keys)
   satisfies |x - x_hat| <= Delta16/2 for unclipped values.
"""

from __future__ import annotations

import math

import numpy as np

from .fp import bf16_to_f32, to_f16

F32 = np.float32


def kappa_position(g: int, kappa: float):
    """Index and float32 fraction of the kappa-quantile among g sorted values."""
    pos = (g - 1) * float(kappa)
    i = int(math.floor(pos))
    return i, F32(pos - i)


def quantile_sorted(a: np.ndarray, i: int, f: np.float32) -> np.ndarray:
    """Linear interpolation between order statistics a[..., i] and a[..., i+1] in float32."""
    g = a.shape[-1]
    if i >= g - 1:
        return a[..., g - 1].copy()
    lo = a[..., i]
    hi = a[..., i + 1]
    return lo + f * (hi - lo)


def group_range(y: np.ndarray, kappa: float):
    """(lo, hi) float32 of every group: y [..., G] float32."""
    a = np.sort(y.astype(F32), axis=-1)
    g = a.shape[-1]
    i_hi, f_hi = kappa_position(g, kappa)
    i_lo, f_lo = kappa_position(g, 1.0 - float(kappa))
    return quantile_sorted(a, i_lo, f_lo), quantile_sorted(a, i_hi, f_hi)


def affine_params(lo: np.ndarray, hi: np.ndarray):
    """Delta16, z16 (float16) from the group range."""
    delta = (hi.astype(F32) - lo.astype(F32)) / F32(3.0)
    d16 = to_f16(delta)
    d16 = np.where(d16 == 0, np.float16(1.0), d16)
    z = -(lo.astype(F32) / d16.astype(F32))
    return d16, to_f16(z)


def quest_params(y: np.ndarray, alpha: float):
    """Delta16, z16 of the QuEST RMS grid for groups y [..., G] (float32 values)."""
    g = y.shape[-1]
    y64 = y.astype(np.float64)
    rms = np.sqrt(np.sum(y64 * y64, axis=-1) / g)
    delta = (2.0 * float(alpha) * rms) / 3.0
    d16 = to_f16(delta)
    d16 = np.where(d16 == 0, np.float16(1.0), d16)
    return d16, np.full(d16.shape, np.float16(1.5))


def codes_from_params(y: np.ndarray, d16: np.ndarray, z16: np.ndarray) -> np.ndarray:
    """INT2 codes for groups y [..., G] float32 with per-group Delta16, z16 [...]."""
    u = y.astype(F32) / d16.astype(F32)[..., None] + z16.astype(F32)[..., None]
    return np.clip(np.rint(u), 0, 3).astype(np.uint8)


def l2_scale(x: np.ndarray):
    """(y float32 [..., d], s16 float16 [...]) for rows x [..., d] float32."""
    x64 = x.astype(np.float64)
    s = np.sqrt(np.sum(x64 * x64, axis=-1))
    s16 = to_f16(s)
    sf = s16.astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = x.astype(F32) / sf[..., None]
    y = np.where((sf == 0)[..., None], F32(0.0), y)
    return y.astype(F32), s16


def quantize_rows(x_bits: np.ndarray, group: int, kappa: float = 1.0, quantizer: str = "affine",
                  alpha: float = 1.4935705, l2: bool = False) -> dict:
    """Quantize BF16 rows x_bits [n, d] (bit patterns) to INT2.

    Returns codes [n, d] uint8, delta16 / zero16 [n, d/G] float16, norm16 [n]
    float16 (or None) and a per-row flag for non-finite scale data.
    """
    x = bf16_to_f32(x_bits)
    n, d = x.shape
    if d % group:
        raise ValueError("group size must divide head_dim")
    norm16 = None
    y = x
    if l2:
        y, norm16 = l2_scale(x)
    yg = y.reshape(n, d // group, group)
    if quantizer == "affine":
        lo, hi = group_range(yg, kappa)
        d16, z16 = affine_params(lo, hi)
    elif quantizer == "quest":
        d16, z16 = quest_params(yg, alpha)
    else:
        raise ValueError(quantizer)
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        c = codes_from_params(yg, d16, z16).reshape(n, d)
    bad = ~np.isfinite(d16.astype(np.float64)).all(-1) | ~np.isfinite(z16.astype(np.float64)).all(-1)
    if norm16 is not None:
        bad |= ~np.isfinite(norm16.astype(np.float64))
    return {"codes": c, "delta16": d16, "zero16": z16, "norm16": norm16, "nonfinite": bad}


def dequantize(q: dict) -> np.ndarray:
    """x_hat = s16 * Delta16 * (c - z16) in float64, [n, d] ([OScaR] "步骤二" dequantisation;
    the OScaR algorithm's attention part for per-channel keys: k_hat_t = s_t Delta (Q(k_t) - z))."""
    c = q["codes"].astype(np.float64)
    n, d = c.shape
    dd = q["delta16"].astype(np.float64)
    zz = q["zero16"].astype(np.float64)
    if q.get("axis") == "channel":
        blk = q["block"]
        xh = (dd[:, None, :] * (c.reshape(n // blk, blk, d) - zz[:, None, :])).reshape(n, d)
    else:
        ng = q["delta16"].shape[-1]
        g = d // ng
        xh = (dd[..., None] * (c.reshape(n, ng, g) - zz[..., None])).reshape(n, d)
    if q.get("norm16") is not None:
        xh = xh * q["norm16"].astype(np.float64)[:, None]
    return xh


def quantize_keys_per_channel(x_bits: np.ndarray, block: int, kappa: float = 1.0, l2: bool = False) -> dict:
    """KIVI's per-channel key quantization of BF16 rows x_bits [n, d] (bit patterns).

    [OScaR] "背景：KIVI 与逐通道量化范式" and "理论分析：TNI 如何破坏逐通道量化": a block of G
    consecutive tokens, and for channel j the block's G values K_{1,j} .. K_{G,j} give
    Delta_{j,g} = (max - min)/(2^b - 1), z_{j,g} = -min/Delta_{j,g}, Q and K_hat as for
    per-token groups; [OScaR] algorithm, key processing: the buffered, l2-scaled keys are
    quantized per channel in blocks when the residual buffer is full.  Here the block is `block` tokens (n a multiple of it; block b holds
    rows [b*block, (b+1)*block)), the optional l2 token scaling comes first (as in
    quantize_rows), and the range, Delta16 / z16 and code steps are those of the per-token
    groups (two-sided kappa-quantile, kappa = 1 giving min / max) applied to channel j's
    `block` values instead of a token's G channels.

    Returns codes [n, d] uint8, delta16 / zero16 [n/block, d] float16 (per block and
    channel), norm16 [n] float16 (or None) and a per-block flag for non-finite scale data.
    """
    x = bf16_to_f32(x_bits)
    n, d = x.shape
    if n % block:
        raise ValueError("the rows must be whole blocks")
    norm16 = None
    y = x
    if l2:
        y, norm16 = l2_scale(x)
    # [blocks, channels, tokens of the block]: one group per (block, channel)
    yc = np.swapaxes(y.reshape(n // block, block, d), 1, 2)
    lo, hi = group_range(yc, kappa)
    d16, z16 = affine_params(lo, hi)
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        c = np.swapaxes(codes_from_params(yc, d16, z16), 1, 2).reshape(n, d)
    bad = ~np.isfinite(d16.astype(np.float64)).all(-1) | ~np.isfinite(z16.astype(np.float64)).all(-1)
    if norm16 is not None:
        bad |= ~np.isfinite(norm16.astype(np.float64)).reshape(n // block, block).all(-1)
    return {"codes": c, "delta16": d16, "zero16": z16, "norm16": norm16, "nonfinite": bad,
            "axis": "channel", "block": block}


def pack_lsb(codes: np.ndarray) -> np.ndarray:
    """Logical packing used for byte-level comparison: word w of a row holds
    codes 16w .. 16w+15, code 16w+i at bits 2i..2i+1 (four 2-bit values per byte,
    least significant first; [OSCAR] section 4 "KV Cache Update")."""
    c = codes.astype(np.uint32)
    n, d = c.shape
    c = c.reshape(n, d // 16, 16)
    shifts = (2 * np.arange(16, dtype=np.uint32))
    return np.bitwise_or.reduce(c << shifts, axis=-1).astype(np.uint32)


def unpack_lsb(words: np.ndarray) -> np.ndarray:
    n, nw = words.shape
    shifts = (2 * np.arange(16, dtype=np.uint32))
    return ((words[..., None].astype(np.uint32) >> shifts) & 3).reshape(n, nw * 16).astype(np.uint8)
