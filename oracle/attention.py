"""Decode attention over the mixed cache, in float64.

Oracle module (test infrastructure only).  softmax(q K^T * scale) V for the new
query token ([OScaR] "KV 缓存的工作原理", decode-step attention; [OSCAR] section 2
"Attention and KV cache"), with grouped-query attention: query head (h, i)
reads kv head h, i.e. query head index h*g + i for g = Hq / Hkv ([WUSH]
"分组查询注意力(GQA)").  Keys and values are the dequantized cache
([OScaR] algorithm, attention phase).  The output stays in the value
transform's space; the caller's folded output projection undoes T_V ([WUSH]
"方法步骤详情", W_O^c = W_O T_V^{-1}).
"""

from __future__ import annotations

import numpy as np


def chunk(q: np.ndarray, pos: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Causal attention of chunk queries: q [n, g, d], query i at position pos[i] attends to
    tokens [0, pos[i]] of k / v [L, d] (the cache as it stands after the chunk was appended:
    [WUSH] "方法步骤详情", mixed-precision attention over the windows and the INT2 middle;
    [OSCAR] section 4 "Decoding Attention Kernel", BF16 and INT2 segments).  -> [n, g, d]."""
    return np.stack([decode(q[i], k[:int(pos[i]) + 1], v[:int(pos[i]) + 1], scale) for i in range(len(pos))])


def decode(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """q [g, d], k / v [L, d] (float64 values) -> out [g, d] float64.

    Max-subtracted softmax; an empty context gives zeros.
    """
    q = np.asarray(q, np.float64)
    if k.shape[0] == 0:
        return np.zeros_like(q)
    s = (q @ np.asarray(k, np.float64).T) * float(scale)          # [g, L]
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    return p @ np.asarray(v, np.float64)
