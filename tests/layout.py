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


def _key_scale_bytes(ng: int, key_axis: int) -> int:
    return 4 * D if key_axis else P * ng * 4


def chunk_bytes(group: int, l2: bool, key_axis: int = 0) -> int:
    ng = D // group
    b = 1024 + _key_scale_bytes(ng, key_axis) + P * ng * 4 + (P * 2 if l2 else 0) + (4 if key_axis else 0)
    return (b + 31) // 32 * 32


def _channel_pairs():
    # per-channel key scales: u32 pair 16 q + 2 s + h holds channels 16 s + 8 h + 2 q and + 1
    byte = np.zeros(D, np.int64)
    for q in range(4):
        for s_ in range(8):
            for h in range(2):
                c = 16 * s_ + 8 * h + 2 * q
                byte[c] = 4 * (16 * q + 2 * s_ + h)
                byte[c + 1] = byte[c] + 2
    return byte


CH_BYTE = _channel_pairs()


def decode_chunk(chunk: np.ndarray, group: int, l2: bool, key_axis: int = 0) -> dict:
    """chunk: uint8 [chunk_bytes] of one (page, kv head).  Per-token keys: dk / zk [token][group];
    per-channel keys (key_axis 1): dk / zk [channel] and the page exponent ek."""
    ng = D // group
    words = chunk[:1024].view(np.uint32)
    codes = (words[:, None] >> SHIFTS[None, :]) & 3            # [256 words, 16 slots]
    ck = np.zeros((P, D), np.uint8)
    cv = np.zeros((P, D), np.uint8)
    ck[KT, KC] = codes[:128]
    cv[VT, VC] = codes[128:]
    kb = _key_scale_bytes(ng, key_axis)
    if key_axis:
        f16 = lambda off: np.array([chunk[off + b:off + b + 2].view(np.float16)[0] for b in CH_BYTE])
        dk, zk = f16(1024), f16(1024 + 2 * D)
    else:
        ks = chunk[1024:1024 + kb].view(np.float16).reshape(P, ng, 2)                # [token][group](D, z)
        dk, zk = ks[:, :, 0], ks[:, :, 1]
    vs = chunk[1024 + kb:1024 + kb + P * ng * 4].view(np.float16).reshape(2, P // 2, ng, 2)
    vd = vs[0].transpose(0, 2, 1).reshape(P, ng)                                     # [pair][group][2] -> [token][group]
    vz = vs[1].transpose(0, 2, 1).reshape(P, ng)
    out = {"ck": ck, "cv": cv, "dk": dk, "zk": zk, "dv": vd, "zv": vz, "nk": None, "ek": None}
    o = 1024 + kb + P * ng * 4
    if l2:
        out["nk"] = chunk[o:o + 2 * P].view(np.float16)
        o += 2 * P
    if key_axis:
        out["ek"] = int(chunk[o:o + 4].view(np.int32)[0])
    return out


def decode_unit(pages: np.ndarray, table_row: np.ndarray, h: int, s_sink: int, s_quant: int,
                group: int, l2: bool, key_axis: int = 0) -> dict:
    """Logical INT2 data of tokens [s_sink, s_quant) of one (sequence, kv head).

    pages: uint8 [num_pages, Hkv, chunk_bytes]; table_row: the sequence's page-table row.
    Per-channel keys: delta_k / zero_k [pages, D] and exp_k [pages].
    """
    n = max(0, s_quant - s_sink)
    ng = D // group
    res = {k: [] for k in ("ck", "cv", "dk", "zk", "dv", "zv", "nk")}
    ek = []
    for p in range(-(-n // P)):
        dec = decode_chunk(pages[int(table_row[p]), h], group, l2, key_axis)
        m = min(P, n - P * p)
        for k in res:
            if dec[k] is not None:
                res[k].append(dec[k][None] if (key_axis and k in ("dk", "zk")) else dec[k][:m])
        ek.append(dec["ek"])
    kshape = (0, D) if key_axis else (0, ng)
    cat = lambda k, shape: np.concatenate(res[k]) if res[k] else np.zeros(shape, np.float16)
    return {"codes_k": cat("ck", (0, D)).astype(np.uint8), "codes_v": cat("cv", (0, D)).astype(np.uint8),
            "delta_k": cat("dk", kshape), "zero_k": cat("zk", kshape),
            "delta_v": cat("dv", (0, ng)), "zero_v": cat("zv", (0, ng)),
            "norm_k": cat("nk", (0,)) if l2 else None, "exp_k": np.array(ek) if key_axis else None}
