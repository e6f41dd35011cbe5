// kv_quant_flush: quantize-on-write of tokens leaving the BF16 recent window into
// INT2 pages (per token, per group: range -> Delta16, z16 -> 2-bit codes).
//
// Source: WUSH-KV digest, inference algorithm (maintain S_quant; quantize S_flush-
// aligned spans beyond S_sink / S_keep in place; per-group QuEST or kappa-quantile
// affine quantizer); OSCAR summary, section 3 "Scale Determination and Clipping"
// (per-token affine scale + zero point, percentile clipping) and section 4 "KV Cache
// Update" (demotion reuses the clip-quantize step); OScaR reading note, "整数量化基础"
// (Q(x), Delta = (max - min)/(2^b - 1)), KIVI background (z = -min/Delta) and step 2
// "Omni-Token Scaling" (s = ||k||, k / s quantized, s stored).
//
// Design (GB300): one warp per (token, kv head, K|V) row; lane l owns channels 4l..4l+3,
// a group of G channels is G/4 lanes.  The quantile needs only a few order statistics
// near the ends: up to the 4th most extreme by a butterfly merge of per-lane sorted
// quadruples, beyond that by repeated warp-level extraction with exact ties -- no sort.
// Codes are OR-reduced across lanes straight into the MMA-fragment layout the decode
// kernel reads with one 128-bit load per thread.  Every float operation is an explicit
// IEEE round-to-nearest intrinsic (divisions by a scale use a correctly rounded
// reciprocal and one exact-remainder correction), so the results are bit-identical to the
// float32 / float64 definition.
#include "common.cuh"
#include "launch.h"
#include "quant.cuh"

#include <algorithm>

namespace kvq {

struct FlushParams {
  uint8_t* pages;
  const int32_t* page_table;
  int32_t* seq_len;
  int32_t* s_quant;
  // kv_append_chunk: cu_rows[b + 1] - cu_rows[b] rows are appended to sequence b by this
  // call; the flush schedule runs on the advanced length, only the tokens already in the ring
  // are quantized here (the appended ones are quantized as they are transformed), and the
  // last CTA of a sequence publishes both seq_len and s_quant.  nullptr: kv_quant_flush.
  const int32_t* cu_rows;
  const uint16_t* ring_k;
  const uint16_t* ring_v;
  int32_t* counters;
  int32_t* status;
  int batch, hkv, s_sink, s_keep, s_flush, ring_cap, max_pages, num_pages, max_tokens;
  int group, quantizer, l2, page_bytes, items_per_cta;
  int i_lo[2], i_hi[2], n_lo[2], n_hi[2];   // [0] keys, [1] values
  float f_lo[2], f_hi[2];
  double alpha;
  // per-channel keys: quantile positions among the 16 values of a channel in a page
  int key_axis, kc_i_lo, kc_i_hi;
  float kc_f_lo, kc_f_hi;
};

__device__ __forceinline__ void sort4(float& a, float& b, float& c, float& d) {
  float t;
  t = fminf(a, b); b = fmaxf(a, b); a = t;
  t = fminf(c, d); d = fmaxf(c, d); c = t;
  t = fminf(a, c); c = fmaxf(a, c); a = t;
  t = fminf(b, d); d = fmaxf(b, d); b = t;
  t = fminf(b, c); c = fmaxf(b, c); b = t;
}

// Extract n values from the top (largest first) of the group's 4*NL values; returns the
// last two extracted: cur = n-th largest, prev = (n-1)-th largest.
template <bool TOP>
__device__ __forceinline__ void extract(const float s[4], int n, int nl, unsigned gmask, int lane,
                                        float& cur, float& prev) {
  int ptr = TOP ? 3 : 0;
  float cand = TOP ? s[3] : s[0];
  cur = prev = cand;
  for (int it = 0; it < n; ++it) {
    float m = cand;
    for (int o = nl >> 1; o > 0; o >>= 1) {
      float other = __shfl_xor_sync(0xffffffffu, m, o);
      m = TOP ? fmaxf(m, other) : fminf(m, other);
    }
    unsigned bal = __ballot_sync(0xffffffffu, cand == m) & gmask;
    int owner = __ffs(bal) - 1;
    if (lane == owner) {
      ptr += TOP ? -1 : 1;
      float inf = TOP ? -INFINITY : INFINITY;
      cand = (ptr == 0) ? s[0] : (ptr == 1) ? s[1] : (ptr == 2) ? s[2] : (ptr == 3) ? s[3] : inf;
    }
    prev = cur;
    cur = m;
  }
}

// The K most extreme values of the group (largest when TOP), most extreme first, on every
// lane of the group: each lane starts from its own 4 sorted values and merges with its
// butterfly partner at every stage; the k-th most extreme of two sorted lists v, w is
// ext_{i=0..k+1} inner(v[i-1], w[k-i]) with v[-1] = w[-1] = the most extreme value.
template <int K, bool TOP>
__device__ __forceinline__ void group_topk(const float s[4], int nl, float (&r)[K]) {
#pragma unroll
  for (int i = 0; i < K; ++i) r[i] = TOP ? s[3 - i] : s[i];
  for (int o = nl >> 1; o > 0; o >>= 1) {
    float w[K], m[K];
#pragma unroll
    for (int i = 0; i < K; ++i) w[i] = __shfl_xor_sync(0xffffffffu, r[i], o);
#pragma unroll
    for (int k = 0; k < K; ++k) {
      float best = TOP ? fmaxf(r[k], w[k]) : fminf(r[k], w[k]);
#pragma unroll
      for (int i = 1; i <= k; ++i) {
        const float t = TOP ? fminf(r[i - 1], w[k - i]) : fmaxf(r[i - 1], w[k - i]);
        best = TOP ? fmaxf(best, t) : fminf(best, t);
      }
      m[k] = best;
    }
#pragma unroll
    for (int k = 0; k < K; ++k) r[k] = m[k];
  }
}

// n-th and (n-1)-th most extreme values of the group (butterfly merge for n <= 4, repeated
// extraction beyond).
template <bool TOP>
__device__ __forceinline__ void order_stats(const float s[4], int n, int nl, unsigned gmask, int lane,
                                            float& cur, float& prev) {
  switch (n) {
    case 1: { float r[1]; group_topk<1, TOP>(s, nl, r); cur = prev = r[0]; break; }
    case 2: { float r[2]; group_topk<2, TOP>(s, nl, r); cur = r[1]; prev = r[0]; break; }
    case 3: { float r[3]; group_topk<3, TOP>(s, nl, r); cur = r[2]; prev = r[1]; break; }
    case 4: { float r[4]; group_topk<4, TOP>(s, nl, r); cur = r[3]; prev = r[2]; break; }
    default: extract<TOP>(s, n, nl, gmask, lane, cur, prev); break;
  }
}

// Quantize one row held as 4 float32 values per lane; returns the lane's 4 codes and the
// group's Delta16 / z16 in dz (valid on all lanes).
__device__ __forceinline__ void quant_row(const QuantConsts& Q, const float (&y)[4], int lane,
                                          uint32_t (&code)[4], __half2& dz, bool& bad) {
  const int nl = Q.nl;
  const unsigned gmask = nl == 32 ? 0xffffffffu : (((1u << nl) - 1u) << (lane & ~(nl - 1)));
  __half d16, z16;
  if (Q.affine) {
    float s[4] = {y[0], y[1], y[2], y[3]};
    sort4(s[0], s[1], s[2], s[3]);
    float hc, hp, lc, lp;
    order_stats<true>(s, Q.n_hi, nl, gmask, lane, hc, hp);
    order_stats<false>(s, Q.n_lo, nl, gmask, lane, lc, lp);
    const int g = Q.group;
    float hi = (Q.i_hi >= g - 1) ? hc : __fadd_rn(hc, __fmul_rn(Q.f_hi, __fsub_rn(hp, hc)));
    float lo = (Q.i_lo >= g - 1) ? lc : __fadd_rn(lp, __fmul_rn(Q.f_lo, __fsub_rn(lc, lp)));
    float delta = __fdiv_rn(__fsub_rn(hi, lo), 3.0f);
    d16 = __float2half_rn(delta);
    if (__half2float(d16) == 0.0f) d16 = __float2half_rn(1.0f);
    float z = -__fdiv_rn(lo, __half2float(d16));
    z16 = __float2half_rn(z);
  } else {
    double ss = 0.0;
#pragma unroll
    for (int m = 0; m < 4; ++m) ss = __dadd_rn(ss, __dmul_rn((double)y[m], (double)y[m]));
    for (int o = nl >> 1; o > 0; o >>= 1) ss = __dadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    double rms = __dsqrt_rn(__ddiv_rn(ss, (double)Q.group));
    double delta = __ddiv_rn(__dmul_rn(__dmul_rn(2.0, Q.alpha), rms), 3.0);
    d16 = double_to_half_rn(delta);
    if (__half2float(d16) == 0.0f) d16 = __float2half_rn(1.0f);
    z16 = __float2half_rn(1.5f);
  }
  float df = __half2float(d16), zf = __half2float(z16);
  if (!isfinite(df) || !isfinite(zf)) bad = true;
  float qv[4];
  div4_by_scale(y, df, qv);
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int c = __float2int_rn(__fadd_rn(qv[m], zf));
    code[m] = (uint32_t)min(max(c, 0), 3);
  }
  dz = __halves2half2(d16, z16);
}

// The flush span of sequence b from its length L_in and s_quant sq (both as read after the
// dependency wait): n tokens from sq on are quantized from the ring by this launch, s_quant
// advances by n_adv, and the length becomes L_new.  Invalid states quantize nothing.
__device__ __forceinline__ void flush_span(const FlushParams& P, int b, int L_in, int sq, bool leader, int& n,
                                           int& n_adv, int& L_new) {
  const int nb = P.cu_rows ? __ldg(P.cu_rows + b + 1) - __ldg(P.cu_rows + b) : 0;
  L_new = L_in + nb;
  const int avail = L_new - sq - P.s_keep;
  n_adv = avail >= P.s_flush ? (avail / P.s_flush) * P.s_flush : 0;
  if (P.cu_rows) {
    n = min(n_adv, max(0, L_in - sq));       // the rest of the span arrives with this call
    if (n > P.max_tokens) {                  // more than the ring can hold: not a valid state
      if (leader) set_status(P.status, KVQ_ERR_BOUNDS);
      n = P.max_tokens;
    }
  } else {
    const int cap = (P.max_tokens / P.s_flush) * P.s_flush;
    n_adv = n_adv < cap ? n_adv : cap;
    n = n_adv;
  }
  if (sq < P.s_sink || L_in < 0 || nb < 0) {
    if (leader) set_status(P.status, KVQ_ERR_BOUNDS);
    n = n_adv = 0;
    L_new = L_in;
  }
}

// Publication of the new state of sequence b (s_quant, and seq_len for an append).
__device__ __forceinline__ void flush_publish(const FlushParams& P, int b, int sq, int n_adv, int L_new) {
  P.s_quant[b] = sq + n_adv;
  if (P.cu_rows) P.seq_len[b] = L_new;
}

// The parameter block is a grid constant: device functions read it by reference, with
// run-time indices, straight from the launch's parameter space (no per-CTA copy).
__global__ void __launch_bounds__(256, 3) flush_kernel(const __grid_constant__ FlushParams P) {
  pdl_trigger();
  const int b = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  {
    // Before waiting for the producer kernels: warm L2 with this warp's first ring row and
    // page-table entry, located from the s_quant seen now (a prefetch only: everything that
    // counts is read again after the wait).
    const int sq_g = P.s_quant[b];
    const int r0 = (blockIdx.x * P.items_per_cta + warp) >> 1;
    const int t = r0 / P.hkv, hh = r0 - t * P.hkv;
    const int tok = sq_g + t;
    if (lane < 2 && tok >= P.s_sink) {
      const uint16_t* ring = (warp & 1) ? P.ring_v : P.ring_k;
      prefetch_l2_line(ring + (((size_t)b * P.hkv + hh) * P.ring_cap + tok % P.ring_cap) * kHeadDim + 64 * lane);
      const int pidx = (tok - P.s_sink) >> 4;
      if (lane == 0 && pidx < P.max_pages) prefetch_l2_line(P.page_table + (size_t)b * P.max_pages + pidx);
    }
  }
  pdl_wait();
  const int nwarps = blockDim.x >> 5;
  // every warp derives the span itself (no block barrier before the first load)
  const int L = P.seq_len[b], sq = P.s_quant[b];
  int n, n_adv, L_new;
  flush_span(P, b, L, sq, lane == 0 && warp == 0, n, n_adv, L_new);
  // Nothing to quantize or publish this step (every CTA of the sequence derives that from the
  // same L and s_quant, so the whole CTA leaves here): a decode step's grid is sized for the
  // largest flush, and most steps flush nothing.
  if (n_adv == 0 && L_new == L) return;
  // Every warp has read s_quant once the CTA passes this barrier.  A single CTA publishes the
  // new value at once (later kernels read it only after this grid completes); otherwise each
  // CTA takes a ticket now -- a release atomic whose result is only needed at the end, so its
  // latency hides behind the work -- and the last reader publishes.
  __syncthreads();
  int ticket = -1;
  if (threadIdx.x == 0) {
    if (gridDim.x == 1) flush_publish(P, b, sq, n_adv, L_new);
    else ticket = atomic_add_release_gpu(P.counters + b, 1);
  }
  const int ng = kHeadDim / P.group;
  // work items: (token, kv head, K|V) in that order, a contiguous range per CTA, strided over
  // the CTA's warps.  Ranges and strides are even, so a warp always handles keys (even warps)
  // or values (odd warps), and its (token, head, ring slot) advance without divisions.  The
  // page-table entry and ring row of a warp's next item are fetched while the current one is
  // quantized.
  const int n_items = n * P.hkv * 2;
  const int i0 = blockIdx.x * P.items_per_cta;
  // an append's grid covers the usual ring occupancy; the last CTA takes whatever is beyond;
  // per-channel keys are quantized by their own kernel (the key warps have nothing to do)
  const int i1 = ((warp & 1) == 0 && P.key_axis) ? i0
                 : (P.cu_rows && blockIdx.x == gridDim.x - 1) ? n_items
                                                              : min(n_items, i0 + P.items_per_cta);
  const int which = warp & 1;
  const uint16_t* ring = which ? P.ring_v : P.ring_k;
  const int hkv = P.hkv, rcap = P.ring_cap, dh = nwarps >> 1;
  // everything the row loop needs, in registers (the parameter block is shared memory, which
  // the compiler would re-read after every store through a generic pointer)
  QuantConsts Q;
  Q.nl = P.group >> 2;
  Q.group = P.group;
  Q.affine = P.quantizer == KVQ_QUANT_AFFINE_KAPPA;
  Q.n_hi = P.n_hi[which];
  Q.n_lo = P.n_lo[which];
  Q.i_hi = P.i_hi[which];
  Q.i_lo = P.i_lo[which];
  Q.f_hi = P.f_hi[which];
  Q.f_lo = P.f_lo[which];
  Q.alpha = P.alpha;
  const bool key_norm = which == 0 && P.l2;
  const int s_sink = P.s_sink, max_pages = P.max_pages, num_pages = P.num_pages, page_bytes = P.page_bytes;
  const int32_t* ptab = P.page_table + (size_t)b * max_pages;
  uint8_t* const pages = P.pages;
  int it = i0 + warp;
  int nx_h = 0, nx_tok = 0, nx_slot = 0, pid_n = -1;
  uint2 raw_n = make_uint2(0u, 0u);
  auto fetch = [&]() {
    const int pidx = (nx_tok - s_sink) >> 4;
    pid_n = (pidx < max_pages) ? ptab[pidx] : -1;
    raw_n = *reinterpret_cast<const uint2*>(
        ring + (((size_t)b * hkv + nx_h) * rcap + nx_slot) * kHeadDim + 4 * lane);
  };
  if (it < i1) {
    const int r0 = it >> 1, t = r0 / hkv;
    nx_h = r0 - t * hkv;
    nx_tok = sq + t;
    nx_slot = nx_tok % rcap;
    fetch();
  }
  for (; it < i1; it += nwarps) {
    const int tok = nx_tok, h = nx_h, pid = pid_n;
    const uint2 raw = raw_n;
    nx_h += dh;
    while (nx_h >= hkv) {
      nx_h -= hkv;
      ++nx_tok;
      if (++nx_slot == rcap) nx_slot = 0;
    }
    if (it + nwarps < i1) fetch();
    const int tp = (tok - s_sink) & (kPage - 1);
    if (pid < 0 || pid >= num_pages) {
      if (lane == 0) set_status(P.status, KVQ_ERR_BOUNDS);
      continue;
    }
    uint8_t* chunk = pages + ((size_t)pid * hkv + h) * page_bytes;
    bool bad = false;
    float y[4];
    y[0] = __uint_as_float(raw.x << 16);
    y[1] = __uint_as_float(raw.x & 0xffff0000u);
    y[2] = __uint_as_float(raw.y << 16);
    y[3] = __uint_as_float(raw.y & 0xffff0000u);
    if (key_norm) {
      double ss = 0.0;
#pragma unroll
      for (int m = 0; m < 4; ++m) ss = __dadd_rn(ss, __dmul_rn((double)y[m], (double)y[m]));
      for (int o = 16; o > 0; o >>= 1) ss = __dadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
      __half s16 = double_to_half_rn(__dsqrt_rn(ss));
      float sf = __half2float(s16);
      if (!isfinite(sf)) bad = true;
      // the division's warp vote stays outside any branch; a zero norm gives a zero row
      const float sdiv = sf == 0.0f ? 1.0f : sf;
      float yn[4];
      div4_by_scale(y, sdiv, yn);
#pragma unroll
      for (int m = 0; m < 4; ++m) y[m] = sf == 0.0f ? 0.0f : yn[m];
      if (lane == 0) reinterpret_cast<__half*>(chunk + norm_off(ng))[tp] = s16;
    }
    __half2 dz;
    uint32_t c[4];
    quant_row(Q, y, lane, c, dz, bad);
    const int nl = Q.nl;
    if ((lane & (nl - 1)) == 0) {
      const int g = lane / nl;
      if (which == 0) {
        *reinterpret_cast<__half2*>(chunk + k_scale_off() + (tp * ng + g) * 4) = dz;
      } else {
        *reinterpret_cast<__half*>(chunk + v_delta_off(ng, tp, g, P.key_axis)) = __low2half(dz);
        *reinterpret_cast<__half*>(chunk + v_zero_off(ng, tp, g, P.key_axis)) = __high2half(dz);
      }
    }
    // Pack the codes with shuffles.  Lane l holds channels 4l..4l+3; with s = l / 4 its pairs
    // (4l, 4l+1) and (4l+2, 4l+3) land at bits 2s and 16 + 2s of two 32-bit words (keys) or
    // of two pairs of 16-bit half-words (values), OR-ed over the 8 lanes of equal l % 4.
    const int sh = 2 * (lane >> 2);
    uint32_t u0 = (c[0] << sh) | (c[1] << (16 + sh));
    uint32_t u1 = (c[2] << sh) | (c[3] << (16 + sh));
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      u0 |= __shfl_xor_sync(0xffffffffu, u0, o);
      u1 |= __shfl_xor_sync(0xffffffffu, u1, o);
    }
    if (lane < 4) {
      const int hi = lane >> 1, lo = lane & 1;
      if (which == 0) {
        // key word (p, r2) = (2 lo + {0, 1}, hi): u0, u1
        uint32_t* kw = reinterpret_cast<uint32_t*>(chunk);
        const int base = (4 * (tp & 7) + 2 * lo) * 4 + 2 * hi + (tp >> 3);
        kw[base] = u0;
        kw[base + 4] = u1;
      } else {
        // value half-words (rr, hh) = (4 lo + {0, 1, 2, 3}, hi): u0 low / high, u1 low / high
        uint16_t* vw = reinterpret_cast<uint16_t*>(chunk + kCodeBytes);
        const int off = 2 * (((tp & 7) >> 1) * 4 + 2 * (tp >> 3) + hi) + (tp & 1);
        const int rr = 4 * lo;
        vw[2 * (4 * rr) * 4 + off] = (uint16_t)(u0 & 0xffffu);
        vw[2 * (4 * (rr + 1)) * 4 + off] = (uint16_t)(u0 >> 16);
        vw[2 * (4 * (rr + 2)) * 4 + off] = (uint16_t)(u1 & 0xffffu);
        vw[2 * (4 * (rr + 3)) * 4 + off] = (uint16_t)(u1 >> 16);
      }
    }
    if (bad && lane == 0) set_status(P.status, KVQ_ERR_NONFINITE);
  }
  // the last CTA of this sequence to have read s_quant publishes the new value and re-zeroes
  // the ticket (its fence orders that store after every other CTA's read)
  if (threadIdx.x == 0 && ticket == (int)gridDim.x - 1) {
    __threadfence();
    flush_publish(P, b, sq, n_adv, L_new);
    P.counters[b] = 0;
  }
}

// ---- per-channel keys: one warp per (page, kv head) of the flush span -------------------------
// Lane l owns channels 4l .. 4l+3 of the page's 16 tokens, so each channel's 16 values sit in
// one lane: its range, Delta16, z16 and codes need no other lane.  The token norms (l2 keys)
// are summed by a reduce-scatter whose additions are those of the one-row flush's butterfly
// (partners 16, 8, 4, 2, 1 in that order), so the norms equal the per-token path's bit for bit.
// Runs before the value flush of the same call, which publishes s_quant: both see the same
// span.  Source: OScaR reading note, "背景：KIVI 与逐通道量化范式" (Delta_{j,g}, z_{j,g} over a
// block of tokens) and the algorithm's key processing (l2-scaled keys quantized per channel).
__global__ void __launch_bounds__(128) flush_keys_channel_kernel(const __grid_constant__ FlushParams P) {
  pdl_trigger();
  const int b = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_wait();
  const int L = P.seq_len[b], sq = P.s_quant[b];
  int n, n_adv, L_new;
  flush_span(P, b, L, sq, false, n, n_adv, L_new);      // the value flush reports bad states
  const int item = blockIdx.x * (blockDim.x >> 5) + warp;
  if (item >= (n / kPage) * P.hkv) return;
  const int pi = item / P.hkv, h = item - pi * P.hkv;
  const int tok0 = sq + kPage * pi;
  const int lp = tok0 - P.s_sink;
  const int pidx = lp >> 4;
  const int pid = (pidx < P.max_pages) ? P.page_table[(size_t)b * P.max_pages + pidx] : -1;
  if (pid < 0 || pid >= P.num_pages || (lp & (kPage - 1))) {
    if (lane == 0) set_status(P.status, KVQ_ERR_BOUNDS);
    return;
  }
  const int ng = kHeadDim / P.group;
  uint8_t* chunk = P.pages + ((size_t)pid * P.hkv + h) * P.page_bytes;
  const uint16_t* ring = P.ring_k + ((size_t)b * P.hkv + h) * P.ring_cap * kHeadDim + 4 * lane;
  float y[kPage][4];
#pragma unroll
  for (int t = 0; t < kPage; ++t) {
    const uint2 raw = *reinterpret_cast<const uint2*>(ring + (size_t)((tok0 + t) % P.ring_cap) * kHeadDim);
    y[t][0] = __uint_as_float(raw.x << 16);
    y[t][1] = __uint_as_float(raw.x & 0xffff0000u);
    y[t][2] = __uint_as_float(raw.y << 16);
    y[t][3] = __uint_as_float(raw.y & 0xffff0000u);
  }
  bool bad = false;
  if (P.l2) {
    // sums of squares: lane l ends with token (l >> 1) & 15 (both lanes of a pair)
    double v[kPage];
#pragma unroll
    for (int t = 0; t < kPage; ++t) {
      double ss = 0.0;
#pragma unroll
      for (int m = 0; m < 4; ++m) ss = __dadd_rn(ss, __dmul_rn((double)y[t][m], (double)y[t][m]));
      v[t] = ss;
    }
#pragma unroll
    for (int st = 0; st < 4; ++st) {
      const int o = 16 >> st, half = 8 >> st;
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const double send = up ? v[i] : v[half + i];
        const double keep = up ? v[half + i] : v[i];
        v[i] = __dadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, o));
      }
    }
    const double ss = __dadd_rn(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1));
    const __half s16 = double_to_half_rn(__dsqrt_rn(ss));
    const float sf_mine = __half2float(s16);
    if (!isfinite(sf_mine)) bad = true;
    if ((lane & 1) == 0) reinterpret_cast<__half*>(chunk + norm_off(ng, 1))[lane >> 1] = s16;
    const uint32_t s16b = __half_as_ushort(s16);
#pragma unroll
    for (int t = 0; t < kPage; ++t) {
      const float sf = __half2float(__ushort_as_half((unsigned short)__shfl_sync(0xffffffffu, s16b, 2 * t)));
      const float sdiv = sf == 0.0f ? 1.0f : sf;
      float yn[4];
      div4_by_scale(y[t], sdiv, yn);
#pragma unroll
      for (int m = 0; m < 4; ++m) y[t][m] = sf == 0.0f ? 0.0f : yn[m];
    }
  }
  const int s = lane >> 2;                               // the lane's 16-channel block
  uint32_t W[kPage][2];                                  // key words 2 (lane & 3) + k' of each token
#pragma unroll
  for (int t = 0; t < kPage; ++t) W[t][0] = W[t][1] = 0u;
  uint32_t dpair[2] = {0u, 0u}, zpair[2] = {0u, 0u};
  int emax = -14;
  const bool minmax = P.kc_i_hi >= kPage - 1 && P.kc_i_lo == 0 && P.kc_f_lo == 0.0f;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    float v[kPage];
#pragma unroll
    for (int t = 0; t < kPage; ++t) v[t] = y[t][m];
    float hi, lo;
    if (minmax) {
      hi = lo = v[0];
#pragma unroll
      for (int t = 1; t < kPage; ++t) {
        hi = fmaxf(hi, v[t]);
        lo = fminf(lo, v[t]);
      }
    } else {
      float a[kPage];
#pragma unroll
      for (int t = 0; t < kPage; ++t) a[t] = v[t];
      sort16(a);
      float h0 = a[kPage - 1], h1 = a[kPage - 1], l0 = a[0], l1 = a[0];
#pragma unroll
      for (int q = 0; q < kPage - 1; ++q) {
        if (q == P.kc_i_hi) { h0 = a[q]; h1 = a[q + 1]; }
        if (q == P.kc_i_lo) { l0 = a[q]; l1 = a[q + 1]; }
      }
      hi = (P.kc_i_hi >= kPage - 1) ? a[kPage - 1] : __fadd_rn(h0, __fmul_rn(P.kc_f_hi, __fsub_rn(h1, h0)));
      lo = (P.kc_i_lo >= kPage - 1) ? a[kPage - 1] : __fadd_rn(l0, __fmul_rn(P.kc_f_lo, __fsub_rn(l1, l0)));
    }
    __half d16 = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), 3.0f));
    if (__half2float(d16) == 0.0f) d16 = __float2half_rn(1.0f);
    const __half z16 = __float2half_rn(-__fdiv_rn(lo, __half2float(d16)));
    const float df = __half2float(d16), zf = __half2float(z16);
    if (!isfinite(df) || !isfinite(zf)) bad = true;
    float qv[kPage];
    divn_by_scale<kPage>(v, df, qv);
#pragma unroll
    for (int t = 0; t < kPage; ++t) {
      const uint32_t c = (uint32_t)min(max(__float2int_rn(__fadd_rn(qv[t], zf)), 0), 3);
      W[t][m >> 1] |= c << ((m & 1) ? 16 + 2 * s : 2 * s);
    }
    const uint32_t db = __half_as_ushort(d16), zb = __half_as_ushort(z16);
    dpair[m >> 1] |= db << (16 * (m & 1));
    zpair[m >> 1] |= zb << (16 * (m & 1));
    emax = max(emax, (int)((db >> 10) & 31u) - 15);
  }
  // OR over the 8 lanes of equal lane % 4, scattered: lane l keeps tokens 2 (l >> 2), + 1
  uint32_t W8[8][2], W4[4][2], W2[2][2];
  {
    const bool up = (lane & 16) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint32_t send = up ? W[i][k] : W[8 + i][k];
        W8[i][k] = (up ? W[8 + i][k] : W[i][k]) | __shfl_xor_sync(0xffffffffu, send, 16);
      }
  }
  {
    const bool up = (lane & 8) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint32_t send = up ? W8[i][k] : W8[4 + i][k];
        W4[i][k] = (up ? W8[4 + i][k] : W8[i][k]) | __shfl_xor_sync(0xffffffffu, send, 8);
      }
  }
  {
    const bool up = (lane & 4) != 0;
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint32_t send = up ? W4[i][k] : W4[2 + i][k];
        W2[i][k] = (up ? W4[2 + i][k] : W4[i][k]) | __shfl_xor_sync(0xffffffffu, send, 4);
      }
  }
  uint32_t* kw = reinterpret_cast<uint32_t*>(chunk);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int t = 2 * (lane >> 2) + i;
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
      const int k = 2 * (lane & 3) + k2;                 // word k: channel offset 2k in each block
      kw[16 * (t & 7) + 4 * (k & 3) + 2 * (k >> 2) + (t >> 3)] = W2[i][k2];
    }
  }
  uint32_t* dk = reinterpret_cast<uint32_t*>(chunk + kc_delta_off());
  uint32_t* zk = reinterpret_cast<uint32_t*>(chunk + kc_zero_off());
  dk[kc_pair_index(4 * lane)] = dpair[0];
  dk[kc_pair_index(4 * lane + 2)] = dpair[1];
  zk[kc_pair_index(4 * lane)] = zpair[0];
  zk[kc_pair_index(4 * lane + 2)] = zpair[1];
  emax = __reduce_max_sync(0xffffffffu, (unsigned)(emax + 64)) - 64;
  if (lane == 0) *reinterpret_cast<int*>(chunk + kc_exp_off(ng, P.l2)) = emax;
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(P.status, KVQ_ERR_NONFINITE);
}

// ---- prefill-sized flushes: two rows per warp -----------------------------------------------
// Half-warp hr = lane / 16 takes one row; lane hl = lane % 16 of it owns channels 8 hl ..
// 8 hl + 7, so a group of G channels spans G / 8 lanes.  Every per-row step that the whole
// warp executes once per row (order-statistic merges, the scale arithmetic, the code packing,
// the stores) is shared by two rows.  The arithmetic is the one-row kernel's, step for step.

// ascending; an optimal 19-comparator network for 8 inputs
__device__ __forceinline__ void sort8(float (&s)[8]) {
  cswap(s[0], s[1]); cswap(s[2], s[3]); cswap(s[4], s[5]); cswap(s[6], s[7]);
  cswap(s[0], s[2]); cswap(s[1], s[3]); cswap(s[4], s[6]); cswap(s[5], s[7]);
  cswap(s[1], s[2]); cswap(s[5], s[6]); cswap(s[0], s[4]); cswap(s[3], s[7]);
  cswap(s[1], s[5]); cswap(s[2], s[6]);
  cswap(s[1], s[4]); cswap(s[3], s[6]);
  cswap(s[2], s[4]); cswap(s[3], s[5]);
  cswap(s[3], s[4]);
}

// as group_topk, from each lane's 8 sorted values
template <int K, bool TOP>
__device__ __forceinline__ void group_topk8(const float (&s)[8], int nl, float (&r)[K]) {
#pragma unroll
  for (int i = 0; i < K; ++i) r[i] = TOP ? s[7 - i] : s[i];
  for (int o = nl >> 1; o > 0; o >>= 1) {
    float w[K], m[K];
#pragma unroll
    for (int i = 0; i < K; ++i) w[i] = __shfl_xor_sync(0xffffffffu, r[i], o);
#pragma unroll
    for (int k = 0; k < K; ++k) {
      float best = TOP ? fmaxf(r[k], w[k]) : fminf(r[k], w[k]);
#pragma unroll
      for (int i = 1; i <= k; ++i) {
        const float t = TOP ? fminf(r[i - 1], w[k - i]) : fmaxf(r[i - 1], w[k - i]);
        best = TOP ? fmaxf(best, t) : fminf(best, t);
      }
      m[k] = best;
    }
#pragma unroll
    for (int k = 0; k < K; ++k) r[k] = m[k];
  }
}

// as extract, from each lane's 8 sorted values
template <bool TOP>
__device__ __forceinline__ void extract8(const float (&s)[8], int n, int nl, unsigned gmask, int lane,
                                         float& cur, float& prev) {
  int ptr = TOP ? 7 : 0;
  float cand = TOP ? s[7] : s[0];
  cur = prev = cand;
  for (int it = 0; it < n; ++it) {
    float m = cand;
    for (int o = nl >> 1; o > 0; o >>= 1) {
      const float other = __shfl_xor_sync(0xffffffffu, m, o);
      m = TOP ? fmaxf(m, other) : fminf(m, other);
    }
    const unsigned bal = __ballot_sync(0xffffffffu, cand == m) & gmask;
    if (lane == __ffs(bal) - 1) {
      ptr += TOP ? -1 : 1;
      float next = TOP ? -INFINITY : INFINITY;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (ptr == q) next = s[q];
      cand = next;
    }
    prev = cur;
    cur = m;
  }
}

template <bool TOP>
__device__ __forceinline__ void order_stats8(const float (&s)[8], int n, int nl, unsigned gmask, int lane,
                                             float& cur, float& prev) {
  switch (n) {
    case 1: { float r[1]; group_topk8<1, TOP>(s, nl, r); cur = prev = r[0]; break; }
    case 2: { float r[2]; group_topk8<2, TOP>(s, nl, r); cur = r[1]; prev = r[0]; break; }
    case 3: { float r[3]; group_topk8<3, TOP>(s, nl, r); cur = r[2]; prev = r[1]; break; }
    case 4: { float r[4]; group_topk8<4, TOP>(s, nl, r); cur = r[3]; prev = r[2]; break; }
    default: extract8<TOP>(s, n, nl, gmask, lane, cur, prev); break;
  }
}

// quant_row for a half-warp row: 8 values per lane, Q.nl = G / 8 lanes per group
__device__ __forceinline__ void quant_row8(const QuantConsts& Q, const float (&y)[8], int lane,
                                           uint32_t (&code)[8], __half2& dz, bool& bad) {
  const int nl = Q.nl;
  const unsigned gmask = ((1u << nl) - 1u) << ((lane & 16) + ((lane & 15) & ~(nl - 1)));
  __half d16, z16;
  if (Q.affine) {
    float s[8] = {y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]};
    sort8(s);
    float hc, hp, lc, lp;
    order_stats8<true>(s, Q.n_hi, nl, gmask, lane, hc, hp);
    order_stats8<false>(s, Q.n_lo, nl, gmask, lane, lc, lp);
    const int g = Q.group;
    float hi = (Q.i_hi >= g - 1) ? hc : __fadd_rn(hc, __fmul_rn(Q.f_hi, __fsub_rn(hp, hc)));
    float lo = (Q.i_lo >= g - 1) ? lc : __fadd_rn(lp, __fmul_rn(Q.f_lo, __fsub_rn(lc, lp)));
    float delta = __fdiv_rn(__fsub_rn(hi, lo), 3.0f);
    d16 = __float2half_rn(delta);
    if (__half2float(d16) == 0.0f) d16 = __float2half_rn(1.0f);
    float z = -__fdiv_rn(lo, __half2float(d16));
    z16 = __float2half_rn(z);
  } else {
    double ss = 0.0;
#pragma unroll
    for (int m = 0; m < 8; ++m) ss = __dadd_rn(ss, __dmul_rn((double)y[m], (double)y[m]));
    for (int o = nl >> 1; o > 0; o >>= 1) ss = __dadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    double rms = __dsqrt_rn(__ddiv_rn(ss, (double)Q.group));
    double delta = __ddiv_rn(__dmul_rn(__dmul_rn(2.0, Q.alpha), rms), 3.0);
    d16 = double_to_half_rn(delta);
    if (__half2float(d16) == 0.0f) d16 = __float2half_rn(1.0f);
    z16 = __float2half_rn(1.5f);
  }
  float df = __half2float(d16), zf = __half2float(z16);
  if (!isfinite(df) || !isfinite(zf)) bad = true;
  float qv[8];
  div4_by_scale(*reinterpret_cast<const float(*)[4]>(&y[0]), df, *reinterpret_cast<float(*)[4]>(&qv[0]));
  div4_by_scale(*reinterpret_cast<const float(*)[4]>(&y[4]), df, *reinterpret_cast<float(*)[4]>(&qv[4]));
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int c = __float2int_rn(__fadd_rn(qv[m], zf));
    code[m] = (uint32_t)min(max(c, 0), 3);
  }
  dz = __halves2half2(d16, z16);
}

__global__ void __launch_bounds__(256, 3) flush_kernel2(const __grid_constant__ FlushParams P) {
  pdl_trigger();
  const int b = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int hr = lane >> 4, hl = lane & 15;
  const int nwarps = blockDim.x >> 5;
  {
    // warm L2 with this half's first ring row (a prefetch only; see flush_kernel)
    const int sq_g = P.s_quant[b];
    const int r0 = (blockIdx.x * P.items_per_cta + warp + hr * nwarps) >> 1;
    const int t = r0 / P.hkv, hh = r0 - t * P.hkv;
    const int tok = sq_g + t;
    if (hl < 2 && tok >= P.s_sink) {
      const uint16_t* ring = (warp & 1) ? P.ring_v : P.ring_k;
      prefetch_l2_line(ring + (((size_t)b * P.hkv + hh) * P.ring_cap + tok % P.ring_cap) * kHeadDim + 64 * hl);
    }
  }
  pdl_wait();
  const int L = P.seq_len[b], sq = P.s_quant[b];
  int n, n_adv, L_new;
  flush_span(P, b, L, sq, lane == 0 && warp == 0, n, n_adv, L_new);
  if (n_adv == 0 && L_new == L) return;                 // nothing to do (see flush_kernel)
  __syncthreads();
  int ticket = -1;
  if (threadIdx.x == 0) {
    if (gridDim.x == 1) flush_publish(P, b, sq, n_adv, L_new);
    else ticket = atomic_add_release_gpu(P.counters + b, 1);
  }
  const int ng = kHeadDim / P.group;
  // items (token, kv head, K|V) as in flush_kernel; warp w takes items i0 + w + k nwarps
  // (all of kind w & 1), half hr the ones with k = hr mod 2
  const int n_items = n * P.hkv * 2;
  const int i0 = blockIdx.x * P.items_per_cta;
  // an append's grid covers the usual ring occupancy; the last CTA takes whatever is beyond;
  // per-channel keys are quantized by their own kernel (the key warps have nothing to do)
  const int i1 = ((warp & 1) == 0 && P.key_axis) ? i0
                 : (P.cu_rows && blockIdx.x == gridDim.x - 1) ? n_items
                                                              : min(n_items, i0 + P.items_per_cta);
  const int which = warp & 1;
  const uint16_t* ring = which ? P.ring_v : P.ring_k;
  const int hkv = P.hkv, rcap = P.ring_cap;
  QuantConsts Q;
  Q.nl = P.group >> 3;
  Q.group = P.group;
  Q.affine = P.quantizer == KVQ_QUANT_AFFINE_KAPPA;
  Q.n_hi = P.n_hi[which];
  Q.n_lo = P.n_lo[which];
  Q.i_hi = P.i_hi[which];
  Q.i_lo = P.i_lo[which];
  Q.f_hi = P.f_hi[which];
  Q.f_lo = P.f_lo[which];
  Q.alpha = P.alpha;
  const bool key_norm = which == 0 && P.l2;
  const int s_sink = P.s_sink, max_pages = P.max_pages, num_pages = P.num_pages, page_bytes = P.page_bytes;
  const int32_t* ptab = P.page_table + (size_t)b * max_pages;
  uint8_t* const pages = P.pages;
  // this half's row position, advanced by nwarps (token, head) steps per iteration
  int item = i0 + warp + hr * nwarps;
  int nx_h = 0, nx_tok = 0, nx_slot = 0, pid_n = -1;
  uint4 raw_n = make_uint4(0u, 0u, 0u, 0u);
  auto fetch = [&]() {
    const int pidx = (nx_tok - s_sink) >> 4;
    pid_n = (pidx < max_pages) ? ptab[pidx] : -1;
    raw_n = *reinterpret_cast<const uint4*>(
        ring + (((size_t)b * hkv + nx_h) * rcap + nx_slot) * kHeadDim + 8 * hl);
  };
  {
    const int r0 = item >> 1, t = r0 / hkv;
    nx_h = r0 - t * hkv;
    nx_tok = sq + t;
    nx_slot = nx_tok % rcap;
    if (item < i1) fetch();
  }
  for (int base = i0 + warp; base < i1; base += 2 * nwarps, item += 2 * nwarps) {
    const bool live = item < i1;
    const int tok = nx_tok, h = nx_h, pid = pid_n;
    const uint4 raw = raw_n;
    nx_h += nwarps;
    while (nx_h >= hkv) {
      nx_h -= hkv;
      ++nx_tok;
      if (++nx_slot == rcap) nx_slot = 0;
    }
    if (item + 2 * nwarps < i1) fetch();
    const int tp = (tok - s_sink) & (kPage - 1);
    const bool pid_ok = pid >= 0 && pid < num_pages;
    if (live && !pid_ok && hl == 0) set_status(P.status, KVQ_ERR_BOUNDS);
    const bool valid = live && pid_ok;
    uint8_t* chunk = pages + ((size_t)(valid ? pid : 0) * hkv + h) * page_bytes;
    bool bad = false;
    float y[8];
    y[0] = __uint_as_float(raw.x << 16);
    y[1] = __uint_as_float(raw.x & 0xffff0000u);
    y[2] = __uint_as_float(raw.y << 16);
    y[3] = __uint_as_float(raw.y & 0xffff0000u);
    y[4] = __uint_as_float(raw.z << 16);
    y[5] = __uint_as_float(raw.z & 0xffff0000u);
    y[6] = __uint_as_float(raw.w << 16);
    y[7] = __uint_as_float(raw.w & 0xffff0000u);
    if (!valid) {
#pragma unroll
      for (int m = 0; m < 8; ++m) y[m] = 0.0f;
    }
    if (key_norm) {
      double ss = 0.0;
#pragma unroll
      for (int m = 0; m < 8; ++m) ss = __dadd_rn(ss, __dmul_rn((double)y[m], (double)y[m]));
      for (int o = 8; o > 0; o >>= 1) ss = __dadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
      __half s16 = double_to_half_rn(__dsqrt_rn(ss));
      float sf = __half2float(s16);
      if (!isfinite(sf)) bad = true;
      // both halves divide (the division's warp vote needs the whole warp); a zero norm gives
      // a zero row
      const float sdiv = sf == 0.0f ? 1.0f : sf;
      float yn[8];
      div4_by_scale(*reinterpret_cast<const float(*)[4]>(&y[0]), sdiv, *reinterpret_cast<float(*)[4]>(&yn[0]));
      div4_by_scale(*reinterpret_cast<const float(*)[4]>(&y[4]), sdiv, *reinterpret_cast<float(*)[4]>(&yn[4]));
#pragma unroll
      for (int m = 0; m < 8; ++m) y[m] = sf == 0.0f ? 0.0f : yn[m];
      if (valid && hl == 0) reinterpret_cast<__half*>(chunk + norm_off(ng))[tp] = s16;
    }
    __half2 dz;
    uint32_t c[8];
    quant_row8(Q, y, lane, c, dz, bad);
    const int nl = Q.nl;
    if (valid && (hl & (nl - 1)) == 0) {
      const int g = hl / nl;
      if (which == 0) {
        *reinterpret_cast<__half2*>(chunk + k_scale_off() + (tp * ng + g) * 4) = dz;
      } else {
        *reinterpret_cast<__half*>(chunk + v_delta_off(ng, tp, g, P.key_axis)) = __low2half(dz);
        *reinterpret_cast<__half*>(chunk + v_zero_off(ng, tp, g, P.key_axis)) = __high2half(dz);
      }
    }
    // Pack as flush_kernel does: channels 8 hl + 4 j + m are those of the one-row kernel's lane
    // 2 hl + j, whose words land at bits 2 (hl >> 1) and 16 + 2 (hl >> 1); OR over the lanes of
    // equal hl % 2.  Lane hl < 2 then holds the words of class 2 hl + j.
    const int sh = 2 * (hl >> 1);
    uint32_t u[2][2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      u[j][0] = (c[4 * j] << sh) | (c[4 * j + 1] << (16 + sh));
      u[j][1] = (c[4 * j + 2] << sh) | (c[4 * j + 3] << (16 + sh));
    }
#pragma unroll
    for (int o = 2; o < 16; o <<= 1)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        u[j][0] |= __shfl_xor_sync(0xffffffffu, u[j][0], o);
        u[j][1] |= __shfl_xor_sync(0xffffffffu, u[j][1], o);
      }
    if (valid && hl < 2) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int hi = hl, lo = j;
        if (which == 0) {
          uint32_t* kw = reinterpret_cast<uint32_t*>(chunk);
          const int kb = (4 * (tp & 7) + 2 * lo) * 4 + 2 * hi + (tp >> 3);
          kw[kb] = u[j][0];
          kw[kb + 4] = u[j][1];
        } else {
          uint16_t* vw = reinterpret_cast<uint16_t*>(chunk + kCodeBytes);
          const int off = 2 * (((tp & 7) >> 1) * 4 + 2 * (tp >> 3) + hi) + (tp & 1);
          const int rr = 4 * lo;
          vw[2 * (4 * rr) * 4 + off] = (uint16_t)(u[j][0] & 0xffffu);
          vw[2 * (4 * (rr + 1)) * 4 + off] = (uint16_t)(u[j][0] >> 16);
          vw[2 * (4 * (rr + 2)) * 4 + off] = (uint16_t)(u[j][1] & 0xffffu);
          vw[2 * (4 * (rr + 3)) * 4 + off] = (uint16_t)(u[j][1] >> 16);
        }
      }
    }
    if (bad && valid && hl == 0) set_status(P.status, KVQ_ERR_NONFINITE);
  }
  if (threadIdx.x == 0 && ticket == (int)gridDim.x - 1) {
    __threadfence();
    flush_publish(P, b, sq, n_adv, L_new);
    P.counters[b] = 0;
  }
}

// ---- self-check of the scale division ------------------------------------------------------
// div_by_scale against IEEE division for every finite bf16 y and every positive finite
// float16 d (the whole domain of the unscaled quantizer: 65,280 x 31,743 pairs), plus 2^29
// hashed float32 y (the l2-scaled keys); counts bitwise differences (NaN equals NaN).
__device__ __forceinline__ void div_compare(float y, float d, float r, unsigned long long* bad) {
  const float a = div_by_scale(y, d, r), b = __fdiv_rn(y, d);
  if (__float_as_uint(a) != __float_as_uint(b) && !(isnan(a) && isnan(b))) atomicAdd(bad, 1ull);
}
__global__ void div_selftest_exhaustive(unsigned long long* bad) {
  const float d = __half2float(__ushort_as_half((uint16_t)(blockIdx.x + 1)));   // 0x0001 .. 0x7bff
  const float r = __frcp_rn(d);
  for (uint32_t yb = threadIdx.x; yb < 65536u; yb += blockDim.x) {
    if (((yb >> 7) & 0xffu) == 0xffu) continue;                                // bf16 inf / NaN
    div_compare(__uint_as_float(yb << 16), d, r, bad);
  }
}
__device__ __forceinline__ uint32_t mix32(uint32_t x) {
  x ^= x >> 16; x *= 0x7feb352du; x ^= x >> 15; x *= 0x846ca68bu; x ^= x >> 16;
  return x;
}
__global__ void div_selftest_random(unsigned long long* bad) {
  const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
  for (uint32_t k = 0; k < 64; ++k) {
    const uint32_t h1 = mix32(t * 64u + k), h2 = mix32(h1 ^ 0x5bd1e995u);
    const float d = __half2float(__ushort_as_half((uint16_t)(1u + h2 % 0x7bffu)));
    // half of the samples uniform over float32 bit patterns, half with exponents near 1
    const uint32_t yb = (k & 1u) ? h1 : ((h1 & 0x807fffffu) | ((96u + (h1 >> 24) % 64u) << 23));
    if (((yb >> 23) & 0xffu) == 0xffu) continue;
    div_compare(__uint_as_float(yb), d, __frcp_rn(d), bad);
  }
}

}  // namespace kvq

using namespace kvq;

extern "C" int kvq_launch_div_selftest(unsigned long long* d_mismatches, cudaStream_t stream) {
  div_selftest_exhaustive<<<0x7bff, 256, 0, stream>>>(d_mismatches);
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  div_selftest_random<<<kSms * 64, 256, 0, stream>>>(d_mismatches);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

static FlushParams flush_params(const kvq_config* cfg, const kvq_cache* cache, int32_t* d_status) {
  FlushParams P{};
  P.pages = (uint8_t*)cache->pages;
  P.page_table = cache->page_table;
  P.seq_len = cache->seq_len;
  P.s_quant = cache->s_quant;
  P.ring_k = cache->ring_k;
  P.ring_v = cache->ring_v;
  P.counters = cache->counters;
  P.status = d_status;
  P.batch = cfg->batch;
  P.hkv = cfg->n_kv_heads;
  P.s_sink = cfg->s_sink;
  P.s_keep = cfg->s_keep;
  P.s_flush = cfg->s_flush;
  P.ring_cap = cfg->ring_cap;
  P.max_pages = cfg->max_pages_per_seq;
  P.num_pages = cfg->num_pages;
  P.group = cfg->group_size;
  P.quantizer = cfg->quantizer;
  P.l2 = cfg->key_l2norm;
  P.page_bytes = page_head_bytes(cfg->group_size, cfg->key_l2norm, cfg->key_axis);
  P.alpha = cfg->quest_alpha;
  P.key_axis = cfg->key_axis;
  {
    const QuantSpec kc = make_quant_spec(kPage, KVQ_QUANT_AFFINE_KAPPA, cfg->kappa_k, cfg->quest_alpha);
    P.kc_i_lo = kc.i_lo;
    P.kc_i_hi = kc.i_hi;
    P.kc_f_lo = kc.f_lo;
    P.kc_f_hi = kc.f_hi;
  }
  const double kap[2] = {cfg->kappa_k, cfg->kappa_v};
  for (int w = 0; w < 2; ++w) {
    const QuantSpec q = make_quant_spec(cfg->group_size, cfg->quantizer, kap[w], cfg->quest_alpha);
    P.i_hi[w] = q.i_hi;
    P.f_hi[w] = q.f_hi;
    P.i_lo[w] = q.i_lo;
    P.f_lo[w] = q.f_lo;
    P.n_hi[w] = q.n_hi;
    P.n_lo[w] = q.n_lo;
  }
  return P;
}

// Work items are (token, kv head, K|V) rows over `grid_tokens` tokens per sequence.
// Decode-sized flushes: CTAs of 4 warps, one item per warp while that fits one wave of 16 warps
// per SM, spread over many SMs so the flush costs about one row's latency; a grid sized for a
// large S_flush (which flushes on few steps and finds nothing to do on the others) gives each
// warp several items instead, so that the empty launches stay one short wave.  Prefill-sized
// flushes: CTAs of 8 warps, enough items per warp to fill one wave of the GPU, each warp
// prefetching its next row and taking two rows at a time.  The last CTA of a sequence
// publishes s_quant.
static int launch_flush_grid(FlushParams& P, const kvq_config* cfg, int grid_tokens, cudaStream_t stream) {
  const long long items = 2LL * grid_tokens * cfg->n_kv_heads;
  const long long total = items * cfg->batch;
  int threads = 128;
  int ipw = (int)std::max(1LL, (total + kSms * 16LL - 1) / (kSms * 16LL));
  if (total > 4LL * kSms * 16) {
    threads = 256;
    const long long slots = (long long)kSms * 3 * (threads / 32);   // 3 resident CTAs per SM (<= 85 registers)
    ipw = (int)((total + slots - 1) / slots);
  }
  const long long ipc = (long long)ipw * (threads / 32);
  if (ipc > (1LL << 30) || (items + ipc - 1) / ipc > 0x7fffffffLL || cfg->batch > 65535) return KVQ_ERR_UNSUPPORTED;
  P.items_per_cta = (int)ipc;
  const int ctas = (int)std::max(1LL, (items + ipc - 1) / ipc);
  dim3 grid(ctas, cfg->batch);
  return launch_pdl(threads == 256 ? flush_kernel2 : flush_kernel, grid, dim3(threads), 0, stream, P) == cudaSuccess
             ? KVQ_OK
             : KVQ_ERR_CUDA;
}

extern "C" int kvq_launch_flush(const kvq_config* cfg, const kvq_cache* cache, int32_t max_tokens,
                                int32_t* d_status, cudaStream_t stream) {
  FlushParams P = flush_params(cfg, cache, d_status);
  // no call can quantize more than the ring holds beyond S_keep (tokens [s_quant, L) live in
  // the ring), which bounds the launch whatever max_tokens says
  const int ring_limit = cfg->ring_cap - cfg->s_keep;
  if (max_tokens > ring_limit) max_tokens = ring_limit;
  int cap = max_tokens > 0 ? (max_tokens / cfg->s_flush) * cfg->s_flush : 0;
  if (cap <= 0) return KVQ_OK;
  P.max_tokens = cap;
  if (cfg->key_axis == KVQ_KEY_PER_CHANNEL) {
    // key pages first (they read s_quant before the value flush publishes it)
    const long long items = (long long)(cap / kPage) * cfg->n_kv_heads;
    const long long ctas = (items + 3) / 4;
    if (ctas > 0x7fffffffLL || cfg->batch > 65535) return KVQ_ERR_UNSUPPORTED;
    if (ctas > 0 &&
        launch_pdl(flush_keys_channel_kernel, dim3((unsigned)ctas, cfg->batch), dim3(128), 0, stream, P) != cudaSuccess)
      return KVQ_ERR_CUDA;
  }
  return launch_flush_grid(P, cfg, cap, stream);
}

extern "C" int kvq_launch_flush_append(const kvq_config* cfg, const kvq_cache* cache, const int32_t* cu_rows,
                                       int32_t* d_status, cudaStream_t stream) {
  FlushParams P = flush_params(cfg, cache, d_status);
  P.cu_rows = cu_rows;
  // the tokens still in the ring (at most ring_cap); the grid covers what a ring holds between
  // complete steps (fewer than S_keep + S_flush tokens), the last CTA of a sequence the rest
  P.max_tokens = cfg->ring_cap;
  return launch_flush_grid(P, cfg, std::min(cfg->ring_cap, cfg->s_keep + cfg->s_flush), stream);
}
