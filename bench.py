"""Benchmark of the rotated INT2 paged KV-cache hot path on GB300.

One step = one pass of the whole hot path over one batch: rotate the n_new new key /
value rows per sequence and the decode queries (kv_rotate_qk), quantize-on-write flush
(kv_quant_flush), GQA decode attention over the mixed cache (kv_attn_decode).  The cache
is built once (untimed); before every timed step the cache's seq_len / s_quant are reset
to the pre-step state and L2 is flushed by a 512 MB memset (both untimed), so every step
does identical work from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C | --configs C1,C2,..]
                  [--impl reference]

The headline is the 128K-context workload (qwen3-32b-ctx128k-b4-oscar); the 32K, batched
and chunk-append workloads are measured in the same run and reported as "sub_configs"
(each with its roofline, end-to-end figure and oracle baseline; the chunk workload also
times its K/V chunk rotate+quantize and its chunk query rotation on their own).

Prints one JSON line (rank 0).  Multi-GPU runs are independent replicas, one per rank
(weak scaling): the decode units (sequence, kv head) need no exchange.
"""

from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "INT2 paged decode attention: effective HBM GB/s (% of ~8 TB/s), tokens/s"
UNIT = "GB/s"
DEFAULT_CONFIG = 4                 # the largest single-GPU workload (128K context)
SUB_CONFIGS = "2,3,5,6"            # measured in the same run, reported as sub-records
NOMINAL_HBM_GBS = 7900.0
FALLBACK_HBM_GBS = 6800.0


# ---- algorithmic bytes ---------------------------------------------------------------------
def step_bytes(w: synth.Workload, ctx: np.ndarray, sq_before: np.ndarray, sq_after: np.ndarray) -> dict:
    """Minimum bytes one step must move (per the cache layout): decode reads + the
    rotate / flush traffic of the new tokens."""
    d, hkv, g, B = w.head_dim, w.n_kv_heads, w.gqa, w.batch
    ng = d // w.group_size
    # K + V bytes of one INT2 token: codes, scales (per-channel keys: d Delta16 + d z16 and the
    # 4-byte page exponent per 16 tokens), key norm
    chan = w.key_axis == "channel"
    int2_tok = (2 * (d // 4) + 4 * ng + (4 * d / w.page_size + 4 / w.page_size if chan else 4 * ng)
                + (2 if w.key_l2norm else 0))
    L = ctx + w.n_new
    dec_int2 = dec_win = ptab = 0
    for Lb, sqb in zip(L, sq_after):
        Lb, sqb = int(Lb), int(sqb)
        n_int2 = max(0, min(sqb, Lb) - w.s_sink)
        n_win = min(w.s_sink, Lb) + max(0, Lb - max(sqb, w.s_sink))
        dec_int2 += int(round(n_int2 * hkv * int2_tok))
        dec_win += n_win * hkv * 4 * d
        ptab += -(-n_int2 // w.page_size) * 4
    qb = B * w.n_q_heads * d * 2
    decode = dec_int2 + dec_win + ptab + qb + B * w.n_q_heads * d * 4
    n_new_rows = B * w.n_new * hkv
    mats = 0
    if w.transform != "hadamard":
        mats += 2 * hkv * d * d * 4                  # T_K (keys) and T_K^{-T} (queries)
    if w.value_transform != "identity":
        mats += hkv * d * d * 4
    rotate = mats + 2 * qb + 2 * n_new_rows * d * 2 * 2
    n_fl = int(np.sum(sq_after - sq_before)) * hkv
    flush = int(round(n_fl * (2 * d * 2 + int2_tok)))
    return {"decode": int(decode), "decode_int2": int(dec_int2), "decode_window": int(dec_win),
            "rotate": int(rotate), "flush": int(flush), "total": int(decode + rotate + flush)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            j = json.load(open(p))
            return float(j["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in ("attn.cu", "common.cuh"):
        h.update(open(os.path.join(ROOT, "bit_rotated_kv_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        j = json.load(open(p))
        e = j.get(workload)
        if e and e.get("kernel_hash") == kernel_hash():
            return int(e["dram_bytes_per_launch"])
    except Exception:
        return None
    return None


@contextlib.contextmanager
def nvtx_range(name: str):
    """An NVTX range around the timed steps when torch has NVTX support (no-op otherwise)."""
    import torch
    pushed = False
    try:
        torch.cuda.nvtx.range_push(name)
        pushed = True
    except Exception:
        pass
    try:
        yield
    finally:
        if pushed:
            torch.cuda.nvtx.range_pop()


# ---- clocks --------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self._stop = threading.Event()
        self._thr = None

    def _run(self):
        while not self._stop.is_set():
            try:
                out = subprocess.run(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                      "--format=csv,noheader,nounits"], capture_output=True, text=True,
                                     timeout=5).stdout.strip()
                if out:
                    self.samples.append((time.time(), out))
            except Exception:
                pass
            self._stop.wait(0.1)

    def start(self):
        self._thr = threading.Thread(target=self._run, daemon=True)
        self._thr.start()

    def stop(self):
        self._stop.set()
        if self._thr:
            self._thr.join(timeout=10)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, line in self.samples:
            parts = [x.strip() for x in line.split(",")]
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- the GPU arm ----------------------------------------------------------------------------
def _timed_avg(fn, steps: int, stream, reset=None):
    """Average ms of fn() over `steps` runs, CUDA events on `stream` around each run."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        if reset is not None:
            reset()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / steps


def measure_config(args, w: synth.Workload, rank: int, world: int, local_rank: int, headline: bool):
    """One workload: the step timed as a user runs it, per-kernel times, end to end through the
    C ABI from pinned host buffers, and (chunk workloads) the chunk rotate+quantize and the
    chunk query rotation timed on their own."""
    import torch
    from tests import harness

    dev = torch.device("cuda", local_rank)
    # the realistic ring capacity (S_keep + S_flush + n_new): window splits are sized by it
    run = harness.DeviceRun(w, device=dev, do_step=False, ring_extra=0, attn_splits=args.splits)
    r = run.runner
    stream = torch.cuda.current_stream()
    seq0, sq0 = r.cache.seq_len.clone(), r.cache.s_quant.clone()
    k_new, v_new, sidx, pos = r.step_inputs(run.k_all, run.v_all, run.lengths, w.n_new)
    q = run.q
    ctx = run.lengths
    sq_before = sq0.cpu().numpy().astype(np.int64)
    sq_after = np.array([synth_sq(w, int(c)) for c in ctx], np.int64)
    nbytes = step_bytes(w, ctx, sq_before, sq_after)
    flush_buf = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def reset():
        r.cache.seq_len.copy_(seq0)
        r.cache.s_quant.copy_(sq0)
        flush_buf.zero_()

    def step(ev=None):
        # ev: (after rotate, after flush) events, or None
        r.append(k_new, v_new, sidx, pos, q, r.q_out)
        if ev is not None:
            ev[0].record(stream)
        r.flush(w.n_new + w.s_flush)
        if ev is not None:
            ev[1].record(stream)
        r.decode(r.q_out, r.out)

    # warm-up (untimed)
    for _ in range(args.warmup):
        reset()
        step()
    torch.cuda.synchronize()
    if int(r.status.item()) != 0:
        raise RuntimeError(f"{w.name}: device status {int(r.status.item())}")

    sampler = ClockSampler(local_rank)
    sampler.start()
    # clock soak: keep the GPU on this step while the sampler warms up (untimed)
    t_end = time.time() + args.soak
    while time.time() < t_end:
        for _ in range(50):
            reset()
            step()
        torch.cuda.synchronize()

    mk = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    avg = lambda a, b: sum(a[i].elapsed_time(b[i]) for i in range(args.steps)) / args.steps
    # the step as a user runs it: events only at step boundaries, so each launch overlaps its
    # predecessor's tail (programmatic dependent launch)
    ev_s, ev_e = mk(), mk()
    barrier(world)
    torch.cuda.synchronize()
    with nvtx_range("timed_steps" if headline else "timed_steps_" + w.name):
        for i in range(args.steps):
            reset()
            ev_s[i].record(stream)
            step()
            ev_e[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_step = avg(ev_s, ev_e)
    # per-kernel durations: the same steps with events between the launches (which forgoes the
    # overlap); the decode roofline is taken from these
    ev_s2, ev_r, ev_f, ev_e2 = mk(), mk(), mk(), mk()
    torch.cuda.synchronize()
    for i in range(args.steps):
        reset()
        ev_s2[i].record(stream)
        step((ev_r[i], ev_f[i]))
        ev_e2[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    sampler.stop()
    t_dec = avg(ev_f, ev_e2)
    kernel_ms = {"kv_rotate_qk": round(avg(ev_s2, ev_r), 5), "kv_quant_flush": round(avg(ev_r, ev_f), 5),
                 "kv_attn_decode": round(t_dec, 5), "step_with_events_between": round(avg(ev_s2, ev_e2), 5)}
    t_step_max = allreduce_max(t_step, world)
    status = int(r.status.item())

    # ---- end to end through the C ABI with host buffers: H2D of the step's inputs from
    # pinned memory, the three calls, D2H of the attention output, every step.  The step's
    # inputs are packed into one pinned host buffer (256-byte aligned segments), so the
    # upload is a single copy.
    parts = [x.contiguous() for x in (k_new, v_new, sidx, pos, q)]
    offs, nb = [], 0
    for x in parts:
        offs.append(nb)
        nb += (x.numel() * x.element_size() + 255) // 256 * 256
    h_buf = torch.empty(nb, dtype=torch.uint8).pin_memory()
    d_buf = torch.empty(nb, dtype=torch.uint8, device=dev)
    views = []
    for x, o in zip(parts, offs):
        n = x.numel() * x.element_size()
        h_buf[o:o + n].copy_(x.cpu().contiguous().view(-1).view(torch.uint8))
        views.append(d_buf[o:o + n].view(x.dtype).view(x.shape))
    d_k, d_v, d_s, d_p, d_q = views
    h_out = torch.empty(r.out.shape, dtype=r.out.dtype).pin_memory()
    h2d = nb
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        d_buf.copy_(h_buf, non_blocking=True)
        r.append(d_k, d_v, d_s, d_p, d_q, r.q_out)
        r.flush(w.n_new + w.s_flush)
        r.decode(r.q_out, r.out)
        h_out.copy_(r.out, non_blocking=True)

    for _ in range(max(3, args.warmup)):
        reset()
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for i in range(args.steps):
        reset()
        torch.cuda.synchronize()
        s_ev = torch.cuda.Event(enable_timing=True); e_ev = torch.cuda.Event(enable_timing=True)
        s_ev.record(stream)
        e2e_step()
        e_ev.record(stream)
        torch.cuda.synchronize()
        e2e_ms.append(s_ev.elapsed_time(e_ev))
    t_e2e = allreduce_max(sum(e2e_ms) / len(e2e_ms), world)

    peak, peak_kind = measured_peaks()
    achieved = nbytes["decode"] / (t_dec * 1e-3) / 1e9
    value = world * nbytes["total"] / (t_step_max * 1e-3) / 1e9
    res = {
        "value": round(value, 2), "ms_per_step": round(t_step_max, 5),
        "config": {"workload": w.name, "batch": w.batch, "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
                   "head_dim": w.head_dim, "context": int(ctx.max()) + w.n_new, "n_new_tokens": w.n_new,
                   "group_size": w.group_size, "kappa": [w.kappa_k, w.kappa_v],
                   "windows_sink_keep_flush": [w.s_sink, w.s_keep, w.s_flush], "transform": w.transform,
                   "key_l2norm": bool(w.key_l2norm), "key_axis": w.key_axis,
                   "l2": "flushed between timed steps (512 MB memset, untimed)",
                   "bytes_per_step": nbytes, "parallelism": f"replicas x{world}"},
        "tokens_per_s": round(world * w.batch / (t_step_max * 1e-3), 1),
        "hbm_frac_of_nominal_8tbs": round(value / NOMINAL_HBM_GBS, 4),
        "roofline": {"kernel": "kv_attn_decode", "bound": "hbm", "achieved": round(achieved, 2),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s", "traffic": profiled_traffic(w.name),
                     "decode_ms": round(t_dec, 5), "bytes_per_launch": nbytes["decode"],
                     "timing": "CUDA events around each kv_attn_decode launch, second timed pass"},
        "e2e": {"value": round(world * nbytes["total"] / (t_e2e * 1e-3) / 1e9, 2), "unit": UNIT,
                "ms_per_step": round(t_e2e, 5), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "kernel_ms": kernel_ms,
        "gpu_launches": args.steps * step_launches(w, int(q.shape[0]), int(k_new.shape[0]), run.cfg.ring_cap),
        "clocks": sampler.summary(),
        "device_status": status,
    }
    if w.chunk_queries:
        res["chunk"] = measure_chunk(args, w, run, k_new, v_new, sidx, pos, reset, stream, peak)
    del run, r, flush_buf, d_buf
    torch.cuda.empty_cache()
    return res


def chunk_bytes(w: synth.Workload) -> dict:
    """Algorithmic bytes of a chunk append: the K/V rotate + quantize (the fused minimum: each
    appended row read once, the quantized tokens written as INT2 and the rest as BF16 ring
    rows, the ring rows pushed out of the window read once), and the chunk query rotation."""
    d, hkv, B, n = w.head_dim, w.n_kv_heads, w.batch, w.n_new
    ng = d // w.group_size
    int2 = d // 4 + 4 * ng + (2 if w.key_l2norm else 0)      # one K or V row
    ctx = int(w.ctx_lo)
    sq0 = synth_sq(w.replace(n_new=0), ctx)
    sq1 = synth_sq(w, ctx)
    n_q = sq1 - sq0                                          # tokens quantized by the step
    from_ring = max(0, min(n_q, ctx - sq0))                  # of them, rows already in the ring
    from_new = n_q - from_ring
    stay = n - from_new                                      # appended rows that stay BF16
    per_tensor = (n * d * 2 + from_ring * d * 2 + n_q * int2 + stay * d * 2)
    mats = hkv * d * d * 4 * (1 if w.transform != "hadamard" else 0)
    kv = B * hkv * 2 * per_tensor + mats
    qrows = B * n * w.n_q_heads
    q = 2 * qrows * d * 2 + mats
    return {"kv_rotate_quantize": int(kv), "query_rotation": int(q), "query_rows": int(qrows),
            "kv_rows": int(B * n * hkv), "quantized_tokens_per_seq": int(n_q)}


def measure_chunk(args, w, run, k_new, v_new, sidx, pos, reset, stream, peak):
    """Chunk append of a prefill-sized step, timed on its own: (a) the new keys / values
    rotated on the tensor cores and quantized by the flush (two calls), (b) the chunk's
    queries (n_new x Hq rows per sequence) compensated with T_K^{-T}."""
    import torch
    r = run.runner
    cb = chunk_bytes(w)

    def kv():
        r.append(k_new, v_new, sidx, pos)
        r.flush(w.n_new + w.s_flush)
    for _ in range(args.warmup):
        reset()
        kv()
    t_kv = _timed_avg(kv, args.steps, stream, reset)
    # the same append through the fused call (transform and quantize-on-write in one pass)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(np.full(w.batch, w.n_new))]), dtype=torch.int32,
                      device=r.device)
    fused = lambda: r.append_chunk(k_new, v_new, cu)
    for _ in range(args.warmup):
        reset()
        fused()
    t_fused = _timed_avg(fused, args.steps, stream, reset)
    # the chunk queries, [B * n_new, Hq, d] (sequence-major, then token)
    g = w.gqa
    qc = np.zeros((w.batch, w.n_new, w.n_q_heads, w.head_dim), np.uint16)
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            qc[b, :, h * g:(h + 1) * g] = synth.chunk_query_rows(w, b, h)
    qd = torch.from_numpy(qc.reshape(-1, w.n_q_heads, w.head_dim).view(np.int16)).to(r.device).view(torch.bfloat16)
    del qc
    qo = torch.empty_like(qd)
    flush_buf = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=r.device)
    qrun = lambda: r.append(None, None, None, None, qd, qo)
    for _ in range(args.warmup):
        qrun()
    t_q = _timed_avg(qrun, args.steps, stream, lambda: flush_buf.zero_())
    # chunk attention: the last n_att rotated chunk queries of every sequence over the cache as
    # the append left it (each row streams its own causal prefix)
    n_att = min(128, w.n_new)
    rows = torch.cat([qo[b * w.n_new + w.n_new - n_att:(b + 1) * w.n_new] for b in range(w.batch)]).contiguous()
    cu_att = torch.arange(0, (w.batch + 1) * n_att, n_att, dtype=torch.int32, device=r.device)
    out_att = torch.empty((rows.shape[0], w.n_q_heads, w.head_dim), dtype=torch.float32, device=r.device)
    ws_att = r.chunk_workspace(rows.shape[0])
    arun = lambda: r.attn_chunk(rows, cu_att, out_att, ws_att)
    for _ in range(args.warmup):
        arun()
    t_att = _timed_avg(arun, args.steps, stream, lambda: flush_buf.zero_())
    att_bytes = chunk_attention_bytes(w, n_att)
    if int(r.status.item()) != 0:
        raise RuntimeError(f"{w.name}: device status {int(r.status.item())} after the chunk timings")
    flops_q = 2.0 * w.head_dim * w.head_dim * cb["query_rows"]
    flops_kv = 2.0 * w.head_dim * w.head_dim * cb["kv_rows"] * (1 if w.transform != "hadamard" else 0)
    out = {
        "kv_rotate_quantize": {"calls": "kv_rotate_qk (keys, values) + kv_quant_flush", "ms": round(t_kv, 5),
                               "bytes": cb["kv_rotate_quantize"],
                               "achieved_gbs": round(cb["kv_rotate_quantize"] / (t_kv * 1e-3) / 1e9, 2),
                               "frac_of_peak": round(cb["kv_rotate_quantize"] / (t_kv * 1e-3) / 1e9 / peak, 4),
                               "key_tflops": round(flops_kv / (t_kv * 1e-3) / 1e12, 2),
                               "bytes_basis": "fused minimum (each new row read once, INT2 / BF16 written once)",
                               "quantized_tokens_per_seq": cb["quantized_tokens_per_seq"]},
        "kv_append_fused": {"calls": "kv_append_chunk", "ms": round(t_fused, 5),
                            "bytes": cb["kv_rotate_quantize"],
                            "achieved_gbs": round(cb["kv_rotate_quantize"] / (t_fused * 1e-3) / 1e9, 2),
                            "frac_of_peak": round(cb["kv_rotate_quantize"] / (t_fused * 1e-3) / 1e9 / peak, 4),
                            "key_tflops": round(flops_kv / (t_fused * 1e-3) / 1e12, 2),
                            "bytes_basis": "fused minimum (each new row read once, INT2 / BF16 written once)"},
        "query_rotation": {"calls": "kv_rotate_qk (queries only)", "rows": cb["query_rows"], "ms": round(t_q, 5),
                           "bytes": cb["query_rotation"],
                           "achieved_gbs": round(cb["query_rotation"] / (t_q * 1e-3) / 1e9, 2),
                           "frac_of_peak": round(cb["query_rotation"] / (t_q * 1e-3) / 1e9 / peak, 4),
                           "tflops": round(flops_q / (t_q * 1e-3) / 1e12, 2)},
    }
    out["chunk_attention"] = {"calls": "kv_attn_chunk", "rows": int(rows.shape[0]),
                              "rows_per_seq": n_att, "ms": round(t_att, 5),
                              "queries_per_s": round(rows.shape[0] / (t_att * 1e-3), 1),
                              "prefix_bytes": att_bytes,
                              "prefix_gbs": round(att_bytes / (t_att * 1e-3) / 1e9, 2),
                              "bytes_basis": "each row's causal prefix of the cache (INT2 pages, BF16 rows), "
                                             "counted once per row: the rows share pages through L2"}
    del qd, qo, flush_buf, rows, out_att, ws_att
    return out


def chunk_attention_bytes(w, n_att: int) -> int:
    """Bytes the last n_att chunk queries of every sequence read (each its own causal prefix,
    all kv heads): INT2 tokens below the post-append s_quant, BF16 sink and ring rows, q' and out."""
    d, hkv, ng = w.head_dim, w.n_kv_heads, w.head_dim // w.group_size
    int2_tok = 2 * (d // 4) + 4 * ng + (4 * d / w.page_size + 4 / w.page_size if w.key_axis == "channel" else 4 * ng)
    int2_tok += 2 if w.key_l2norm else 0
    ctx = int(w.ctx_lo)
    L = ctx + w.n_new
    sq = synth_sq(w, ctx)
    total = 0.0
    for p in range(L - n_att, L):
        n_int2 = max(0, min(sq, p + 1) - w.s_sink)
        n_win = min(w.s_sink, p + 1) + max(0, p + 1 - max(sq, w.s_sink))
        total += hkv * (n_int2 * int2_tok + n_win * 4 * d + -(-n_int2 // w.page_size) * 4)
        total += w.n_q_heads * d * (2 + 4)
    return int(total * w.batch)


def run_ours(args, rank: int, world: int, local_rank: int):
    import torch
    torch.cuda.set_device(torch.device("cuda", local_rank))
    chosen = [int(c) for c in str(args.configs).split(",") if c.strip()] if args.configs else [args.config]
    head = measure_config(args, workload(args, chosen[0]), rank, world, local_rank, True)
    res = {"metric": METRIC, "value": head.pop("value"), "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": head.pop("ms_per_step"), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "int2 codes x f16 tensor-core MMA, f32 accumulate",
           "data": "synthetic (seeded; shapes of the pages' Qwen3 workloads, random transforms)"}
    res.update(head)
    subs = {}
    for c in chosen[1:]:
        wc = workload(args, c)
        if world > 1:                   # every rank takes the same barriers: no partial records
            sub = measure_config(args, wc, rank, world, local_rank, False)
            subs[sub["config"]["workload"]] = sub
            continue
        try:
            sub = measure_config(args, wc, rank, world, local_rank, False)
            subs[sub["config"]["workload"]] = sub
        except Exception as e:          # the headline record stands; the failure is reported
            msg = str(e).strip().splitlines()
            subs[wc.name] = {"config": {"workload": wc.name}, "error": f"{type(e).__name__}: {msg[0] if msg else ''}"}
    if subs:
        res["sub_configs"] = subs
    return res


def workload(args, config: int | None = None) -> synth.Workload:
    """The configuration, optionally shrunk (--batch) for a profiler capture of the same kernel."""
    w = synth.WORKLOADS[args.config if config is None else config]
    if args.batch:
        w = w.replace(batch=args.batch)
    return w


def synth_sq(w, ctx: int) -> int:
    s = w.s_sink
    L = ctx
    while L - s >= w.s_keep + w.s_flush:
        s += w.s_flush
    L += w.n_new
    while L - s >= w.s_keep + w.s_flush:
        s += w.s_flush
    return s


# ---- launches per step ---------------------------------------------------------------------
# kv_rotate_qk's dispatch (include/kvq.h): from this many dense (row, head) pairs on, the dense
# rows run on the tensor cores and the exact copies / Hadamard rows in a second launch
TC_MIN_PAIRS = 128 * 152


def rotate_launches(w, n_q_rows: int, n_kv_rows: int) -> int:
    """Kernel launches of one kv_rotate_qk call (the library's dispatch rule)."""
    had = w.transform == "hadamard"
    q_pairs, kv_pairs = n_q_rows * w.n_q_heads, n_kv_rows * w.n_kv_heads
    dense = (0 if had else q_pairs + kv_pairs) + (kv_pairs if w.value_transform != "identity" else 0)
    items = (q_pairs + kv_pairs if had else 0) + (kv_pairs if w.value_transform == "identity" else 0)
    if dense < TC_MIN_PAIRS:
        return 1 if dense + items > 0 else 0
    return 2 if items > 0 else 1


def step_launches(w, n_q_rows: int, n_kv_rows: int, ring_cap: int) -> int:
    """Kernel launches of one bench step: rotate, flush (when it may quantize anything), decode."""
    max_tokens = min(w.n_new + w.s_flush, ring_cap - w.s_keep)
    flush = 1 if (max_tokens // w.s_flush) * w.s_flush > 0 else 0
    return rotate_launches(w, n_q_rows, n_kv_rows) + flush + 1


# ---- CPU baseline: the oracle as it stands on a bounded sample -----------------------------
def oracle_step_sample(config: int, budget_s: float) -> dict:
    """Time the oracle's step work (rotate the new rows and queries, quantize the flushed
    tokens, dequantize the cache, float64 attention) on whole (sequence, kv head) units of
    the workload until about budget_s of CPU time has been spent; returns GB/s equivalent."""
    from oracle import attention, cache, quant, transform
    from oracle.fp import bf16_to_f32, f32_to_bf16_bits
    w = synth.WORKLOADS[config]
    tk, tkit, tv = synth.transforms(w)
    lengths = synth.context_lengths(w)
    ctx = lengths
    sq_b = np.array([synth_sq(w.replace(n_new=0), int(c)) for c in ctx])
    sq_a = np.array([synth_sq(w, int(c)) for c in ctx])
    full = step_bytes(w, ctx, sq_b, sq_a)["total"]
    units = [(b, h) for b in range(w.batch) for h in range(w.n_kv_heads)]
    per_unit = full / len(units)
    done = 0
    spent = 0.0
    i = 0
    # the untimed cache build of each sampled unit costs several times its timed step, so the
    # sample also stops after 3 x budget_s of wall time
    wall_end = time.time() + 3.0 * budget_s
    while spent < budget_s and i < 100000 and (done == 0 or time.time() < wall_end):
        b, h = units[i % len(units)]
        i += 1
        ui = synth.unit_inputs(w, b, h, lengths)
        L = ui.ctx + w.n_new
        kind = "hadamard" if w.transform == "hadamard" else "dense"
        # state before the step (untimed): rotated rows and quantized cache of the context
        k_rot = f32_to_bf16_bits(transform.rotate_rows(None if tk is None else tk[h], ui.k[:ui.ctx], kind))
        v_rot = f32_to_bf16_bits(transform.rotate_rows(None if tv is None else tv[h], ui.v[:ui.ctx]))
        sqb = int(sq_b[b])
        unit = cache.build_unit(k_rot, v_rot, ui.ctx, sqb, s_sink=w.s_sink, group=w.group_size,
                                kappa_k=w.kappa_k, kappa_v=w.kappa_v, quantizer=w.quantizer,
                                alpha=w.quest_alpha, key_l2norm=w.key_l2norm, key_axis=w.key_axis)
        t0 = time.process_time()
        # the step: rotate new rows + queries, flush, dequantize the cache, attend
        kn = f32_to_bf16_bits(transform.rotate_rows(None if tk is None else tk[h], ui.k[ui.ctx:L], kind))
        vn = f32_to_bf16_bits(transform.rotate_rows(None if tv is None else tv[h], ui.v[ui.ctx:L]))
        qr = transform.rotate_rows(None if tkit is None else tkit[h], ui.q, kind)
        k_all = np.concatenate([k_rot, kn])
        v_all = np.concatenate([v_rot, vn])
        sqa = cache.flush(L, sqb, w.s_keep, w.s_flush)
        kh = bf16_to_f32(k_all).astype(np.float64)
        vh = bf16_to_f32(v_all).astype(np.float64)
        lo = min(w.s_sink, L)
        if sqb > lo:
            kh[lo:sqb] = quant.dequantize(unit["qk"])
            vh[lo:sqb] = quant.dequantize(unit["qv"])
        if sqa > sqb:
            if w.key_axis == "channel":
                qk = quant.quantize_keys_per_channel(k_all[sqb:sqa], w.page_size, w.kappa_k, w.key_l2norm)
            else:
                qk = quant.quantize_rows(k_all[sqb:sqa], w.group_size, w.kappa_k, w.quantizer, w.quest_alpha,
                                         w.key_l2norm)
            kh[sqb:sqa] = quant.dequantize(qk)
            vh[sqb:sqa] = quant.dequantize(quant.quantize_rows(v_all[sqb:sqa], w.group_size, w.kappa_v, w.quantizer,
                                                               w.quest_alpha, False))
        attention.decode(qr.astype(np.float64), kh, vh, 1.0 / math.sqrt(w.head_dim))
        spent += time.process_time() - t0
        done += 1
    gbs = done * per_unit / spent / 1e9
    return {"value": gbs, "units": done, "seconds": spent, "workload": w.name}


def cpu_baseline(config: int, budget_s: float) -> dict:
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = (f"import sys, json; sys.path.insert(0, {ROOT!r}); import bench; "
            f"print(json.dumps(bench.oracle_step_sample({config}, {budget_s})))")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=1800)
    if out.returncode:
        raise RuntimeError(out.stderr[-2000:])
    j = json.loads(out.stdout.strip().splitlines()[-1])
    return {"value": round(j["value"], 6), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{j['units']} (sequence, kv head) units of {j['workload']}: rotate new rows + queries, "
                      f"quantize flushed tokens, dequantize cache, float64 attention; {j['seconds']:.1f} s CPU, "
                      f"1 thread"}


# ---- distributed helpers --------------------------------------------------------------------
_PG = None


def init_dist():
    global _PG
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if _cuda_ok() else "gloo"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        _PG = dist
    return rank, world, local


def _cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def barrier(world):
    if world > 1 and _PG is not None:
        _PG.barrier()


def allreduce_max(x: float, world: int) -> float:
    if world > 1 and _PG is not None:
        import torch
        dev = torch.device("cuda", torch.cuda.current_device()) if _cuda_ok() else torch.device("cpu")
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        _PG.all_reduce(t, op=_PG.ReduceOp.MAX)
        return float(t.item())
    return x


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG, help="headline workload (synth.WORKLOADS)")
    ap.add_argument("--configs", default=None,
                    help="comma list: headline first, the rest as sub-records (default: headline + "
                         f"{SUB_CONFIGS} when --config is the default, else the headline alone)")
    ap.add_argument("--sub-cpu-budget", type=float, default=5.0, help="oracle seconds per sub-record")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak", type=float, default=1.0, help="untimed seconds on the step while clocks are sampled")
    ap.add_argument("--batch", type=int, default=0, help="override the batch (smaller profiler captures)")
    ap.add_argument("--splits", type=int, default=0, help="INT2 splits per (sequence, kv head); 0 = library default")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.configs is None:
        args.configs = (f"{args.config}," + SUB_CONFIGS) if (args.config == DEFAULT_CONFIG and not args.batch) \
            else str(args.config)
    args.config = int(args.configs.split(",")[0])
    rank, world, local = init_dist()
    if args.impl == "reference":
        if rank == 0:
            cb = cpu_baseline(args.config, args.cpu_budget)
            w = synth.WORKLOADS[args.config]
            res = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": world,
                   "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
                   "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
                   "config": {"workload": w.name}, "cpu_baseline": cb,
                   "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
            print(json.dumps(res), flush=True)
        return
    res = run_ours(args, rank, world, local)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            res["cpu_baseline"] = cpu_baseline(args.config, args.cpu_budget)
            for name, sub in res.get("sub_configs", {}).items():
                cid = next(k for k, v in synth.WORKLOADS.items() if v.name == name)
                sub["cpu_baseline"] = cpu_baseline(cid, args.sub_cpu_budget)
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
