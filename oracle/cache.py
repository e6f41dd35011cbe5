"""Mixed-precision cache of one (sequence, kv head) and its flush schedule.

Oracle module (test infrastructure only).

Regions ([OSCAR] section 4 "KV Cache Layout": BF16 sink of the first S0 tokens,
BF16 recent window, INT2 middle; [WUSH] "方法步骤详情": full-precision S_sink and
S_keep windows, quantization right edge S_quant advanced over S_flush-aligned
spans; [OScaR] algorithm, key processing: residual buffer quantized when full):

    tokens [0, S_sink)          BF16 sink, never quantized
    tokens [S_sink, s_quant)    INT2 (codes + scale/zero-point [+ norm])
    tokens [s_quant, L)         BF16 recent window

Flush rule: starting from s_quant = S_sink, after tokens are appended, while
L - s_quant >= S_keep + S_flush quantize [s_quant, s_quant + S_flush) and
advance s_quant by S_flush.  S_flush = 1 is OSCAR's one-token demotion,
S_flush = 8 WUSH's downstream setting, and S_keep = 0 with S_flush = 128 is
OScaR's R = 128 residual buffer flushed when full.
"""

from __future__ import annotations

import numpy as np

from . import quant
from .fp import bf16_to_f32


def flush(L: int, s_quant: int, s_keep: int, s_flush: int) -> int:
    """Apply the flush rule once (as many spans as it allows); returns the new s_quant."""
    while L - s_quant >= s_keep + s_flush:
        s_quant += s_flush
    return s_quant


def build_unit(k_rot_bits: np.ndarray, v_rot_bits: np.ndarray, L: int, s_quant: int, *,
               s_sink: int, group: int, kappa_k: float, kappa_v: float,
               quantizer: str = "affine", alpha: float = 1.4935705, key_l2norm: bool = False,
               key_axis: str = "token", key_block: int = 16) -> dict:
    """The cache of one (sequence, kv head) holding tokens [0, L) with INT2 region [S_sink, s_quant).

    k_rot_bits / v_rot_bits: transformed BF16 rows [>= L, d] (bit patterns).
    Per-token groups make a token's codes independent of when it was flushed.  Per-channel
    keys (key_axis "channel", [OScaR] algorithm, key processing) take blocks of key_block tokens from
    S_sink on; the flush spans are then whole blocks, so a block is quantized once, complete.
    """
    lo = min(s_sink, L)
    hi = max(lo, min(s_quant, L))
    if key_axis == "channel":
        qk = quant.quantize_keys_per_channel(k_rot_bits[lo:hi], key_block, kappa_k, key_l2norm)
    else:
        qk = quant.quantize_rows(k_rot_bits[lo:hi], group, kappa_k, quantizer, alpha, key_l2norm)
    qv = quant.quantize_rows(v_rot_bits[lo:hi], group, kappa_v, quantizer, alpha, False)
    return {"L": L, "s_sink": lo, "s_quant": hi, "k_rot": k_rot_bits[:L], "v_rot": v_rot_bits[:L],
            "qk": qk, "qv": qv}


def dequantized_kv(unit: dict):
    """(K_hat, V_hat) float64 [L, d] as attention reads them: BF16 rows in the
    windows, Delta16 (c - z16) (times s16) in the INT2 region."""
    L, lo, hi = unit["L"], unit["s_sink"], unit["s_quant"]
    k = bf16_to_f32(unit["k_rot"]).astype(np.float64).copy()
    v = bf16_to_f32(unit["v_rot"]).astype(np.float64).copy()
    if hi > lo:
        k[lo:hi] = quant.dequantize(unit["qk"])
        v[lo:hi] = quant.dequantize(unit["qv"])
    return k[:L], v[:L]
