"""Decoder of the library's INT2 page layout, written from the layout documented in
include/kvq.h (not from the CUDA sources): turns one (page, kv head) chunk back into
logical per-token codes and float16 scale data for comparison with the oracle."""

from __future__ import annotations

import numpy as np

D = 128
P = 16


def _maps():
    # key words: u32 4l + r, bits 2s + 16e -> token l/4 + 8(r%2), channel 16s + 2(l%4) + 8(r/2) + e
    kt = np.zeros((128, 16), np.int64)
    kc = np.zeros((128, 16), np.int64)
    vt = np.zeros((128, 16), np.int64)
    vc = np.zeros((128, 16), np.int64)
    for l in range(32):
        for r in range(4):
            w = 4 * l + r
            for s in range(8):
                for e in range(2):
                    bit = s + 8 * e            # code slot index = bit position / 2
                    kt[w, bit] = l // 4 + 8 * (r % 2)
                    kc[w, bit] = 16 * s + 2 * (l % 4) + 8 * (r // 2) + e
                    # value words: bits 2m + 16e -> channel 16m + l/4 + 8(r%2), token 2(l%4) + 8(r/2) + e
                    vt[w, bit] = 2 * (l % 4) + 8 * (r // 2) + e
                    vc[w, bit] = 16 * s + l // 4 + 8 * (r % 2)
    return kt, kc, vt, vc


KT, KC, VT, VC = _maps()
SHIFTS = (2 * np.arange(16)).astype(np.uint32)


def chunk_bytes(group: int, l2: bool) -> int:
    ng = D // group
    b = 1024 + 2 * P * ng * 4 + (P * 2 if l2 else 0)
    return (b + 31) // 32 * 32


def decode_chunk(chunk: np.ndarray, group: int, l2: bool) -> dict:
    """chunk: uint8 [chunk_bytes] of one (page, kv head)."""
    ng = D // group
    words = chunk[:1024].view(np.uint32)
    codes = (words[:, None] >> SHIFTS[None, :]) & 3            # [256 words, 16 slots]
    ck = np.zeros((P, D), np.uint8)
    cv = np.zeros((P, D), np.uint8)
    ck[KT, KC] = codes[:128]
    cv[VT, VC] = codes[128:]
    ks = chunk[1024:1024 + P * ng * 4].view(np.float16).reshape(P, ng, 2)          # [token][group](D, z)
    vs = chunk[1024 + P * ng * 4:1024 + 2 * P * ng * 4].view(np.float16).reshape(2, P // 2, ng, 2)
    vd = vs[0].transpose(0, 2, 1).reshape(P, ng)                                     # [pair][group][2] -> [token][group]
    vz = vs[1].transpose(0, 2, 1).reshape(P, ng)
    out = {"ck": ck, "cv": cv, "dk": ks[:, :, 0], "zk": ks[:, :, 1], "dv": vd, "zv": vz, "nk": None}
    if l2:
        o = 1024 + 2 * P * ng * 4
        out["nk"] = chunk[o:o + 2 * P].view(np.float16)
    return out


def decode_unit(pages: np.ndarray, table_row: np.ndarray, h: int, s_sink: int, s_quant: int,
                group: int, l2: bool) -> dict:
    """Logical INT2 data of tokens [s_sink, s_quant) of one (sequence, kv head).

    pages: uint8 [num_pages, Hkv, chunk_bytes]; table_row: the sequence's page-table row.
    """
    n = max(0, s_quant - s_sink)
    ng = D // group
    res = {k: [] for k in ("ck", "cv", "dk", "zk", "dv", "zv", "nk")}
    for p in range(-(-n // P)):
        dec = decode_chunk(pages[int(table_row[p]), h], group, l2)
        m = min(P, n - P * p)
        for k in res:
            if dec[k] is not None:
                res[k].append(dec[k][:m])
    cat = lambda k, shape: np.concatenate(res[k]) if res[k] else np.zeros(shape, np.float16)
    return {"codes_k": cat("ck", (0, D)).astype(np.uint8), "codes_v": cat("cv", (0, D)).astype(np.uint8),
            "delta_k": cat("dk", (0, ng)), "zero_k": cat("zk", (0, ng)),
            "delta_v": cat("dv", (0, ng)), "zero_v": cat("zv", (0, ng)),
            "norm_k": cat("nk", (0,)) if l2 else None}
