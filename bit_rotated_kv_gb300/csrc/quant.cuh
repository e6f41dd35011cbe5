// The per-token INT2 quantizer shared by the flush kernels and the fused append path:
// scale division, quantizer constants, and the 8-lanes-per-row ("octet") form that
// quantizes four rows per warp from 16 values per lane.
//
// Source: WUSH-KV digest, inference algorithm (per-group kappa-quantile affine or QuEST
// quantizer on S_flush-aligned spans); OSCAR summary, section 3 "Scale Determination and
// Clipping" (per-token affine scale and zero point, percentile clipping); OScaR reading
// note, "整数量化基础" (Q(x), Delta = (max - min)/(2^b - 1)), KIVI background (z = -min/Delta)
// and step 2 "Omni-Token Scaling" (s = ||k||, k / s quantized, s stored).
//
// Every float operation is an explicit IEEE round-to-nearest intrinsic, so a row gives the
// same Delta16, z16, codes and norm in every layout (one row per warp, two per warp, four per
// warp): only the order of the float64 sum of squares differs, which is exact for rows whose
// squares span fewer than 37 binades and otherwise changes the float16 result only when the
// square root lies within 2^-52 relative of a float16 rounding boundary.
#pragma once
#include "common.cuh"

namespace kvq {

// y / d for a positive float16 scale d, correctly rounded.  With r = RN(1/d) and
// q0 = RN(y r) (within one ulp of y / d), Markstein's theorem gives RN(y / d) =
// RN(q0 + (y - q0 d) r), the remainder exact by FMA -- as long as nothing underflows or
// overflows, which holds for 2^-96 <= |y| <= 2^96 since 2^-24 <= d <= 65504.  Other y (and
// y = 0, NaN or infinity) take the IEEE division.
__device__ __forceinline__ bool div_fast_ok(float y) {
  const float ay = fabsf(y);
  return ay >= 0x1p-96f && ay <= 0x1p96f;
}
__device__ __forceinline__ float div_fast(float y, float d, float r) {
  const float q0 = __fmul_rn(y, r);
  const float rem = __fmaf_rn(-q0, d, y);
  return __fmaf_rn(rem, r, q0);
}
__device__ __forceinline__ float div_by_scale(float y, float d, float r) {
  return div_fast_ok(y) ? div_fast(y, d, r) : __fdiv_rn(y, d);
}
// The four quotients of a lane, branch-free unless some lane of the warp holds a dividend
// outside the fast range (then those quotients are redone by IEEE division).  All 32 lanes
// must call it.
__device__ __forceinline__ void div4_by_scale(const float (&y)[4], float d, float (&q)[4]) {
  const float r = __frcp_rn(d);
  bool ok = true;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    q[m] = div_fast(y[m], d, r);
    ok = ok && div_fast_ok(y[m]);
  }
  if (!__all_sync(0xffffffffu, ok)) {
#pragma unroll
    for (int m = 0; m < 4; ++m)
      if (!div_fast_ok(y[m])) q[m] = __fdiv_rn(y[m], d);
  }
}
// The same for N = 4 k quotients.
template <int N>
__device__ __forceinline__ void divn_by_scale(const float (&y)[N], float d, float (&q)[N]) {
  const float r = __frcp_rn(d);
  bool ok = true;
#pragma unroll
  for (int m = 0; m < N; ++m) {
    q[m] = div_fast(y[m], d, r);
    ok = ok && div_fast_ok(y[m]);
  }
  if (!__all_sync(0xffffffffu, ok)) {
#pragma unroll
    for (int m = 0; m < N; ++m)
      if (!div_fast_ok(y[m])) q[m] = __fdiv_rn(y[m], d);
  }
}

// Quantizer constants of one kind of row (keys or values), held in registers.  nl is the
// number of lanes a group of G channels spans in the layout at hand.  The clipping range
// is hi = a[i_hi] + f_hi (a[i_hi + 1] - a[i_hi]) over the group's ascending values a (and
// lo likewise), which needs the n_hi largest and the n_lo smallest values.
struct QuantConsts {
  int nl, group, affine, n_hi, n_lo, i_hi, i_lo;
  float f_hi, f_lo;
  double alpha;
};

// Host side: the constants of a group size and clipping quantile (kappa = 1: min / max).
struct QuantSpec {
  int group, affine, n_hi, n_lo, i_hi, i_lo;
  float f_hi, f_lo;
  double alpha;
};

inline void kappa_position(int g, double kappa, int& i, float& f) {
  const double pos = (double)(g - 1) * kappa;
  const double fl = floor(pos);
  i = (int)fl;
  f = (float)(pos - fl);
}

inline QuantSpec make_quant_spec(int group, int quantizer, double kappa, double alpha) {
  QuantSpec s{};
  s.group = group;
  s.affine = quantizer == KVQ_QUANT_AFFINE_KAPPA;
  s.alpha = alpha;
  kappa_position(group, kappa, s.i_hi, s.f_hi);
  kappa_position(group, 1.0 - kappa, s.i_lo, s.f_lo);
  s.n_hi = s.i_hi >= group - 1 ? 1 : group - s.i_hi;
  s.n_lo = s.i_lo + 2 > group ? group : s.i_lo + 2;
  return s;
}

__device__ __forceinline__ QuantConsts quant_consts(const QuantSpec& s, int values_per_lane) {
  QuantConsts Q;
  Q.nl = s.group / values_per_lane;
  Q.group = s.group;
  Q.affine = s.affine;
  Q.n_hi = s.n_hi;
  Q.n_lo = s.n_lo;
  Q.i_hi = s.i_hi;
  Q.i_lo = s.i_lo;
  Q.f_hi = s.f_hi;
  Q.f_lo = s.f_lo;
  Q.alpha = s.alpha;
  return Q;
}

__device__ __forceinline__ void cswap(float& a, float& b) {
  const float t = fminf(a, b);
  b = fmaxf(a, b);
  a = t;
}

// ---- octet layout: lane j = lane % 8 of octet lane / 8 owns channels 16 j .. 16 j + 15 ---------

// Ascending sort of 16 values: Batcher's odd-even merge sort (63 comparators), every index a
// compile-time constant after unrolling.
__device__ __forceinline__ void sort16(float (&s)[16]) {
#pragma unroll
  for (int p = 1; p < 16; p <<= 1)
#pragma unroll
    for (int k = p; k >= 1; k >>= 1)
#pragma unroll
      for (int j = k % p; j + k < 16; j += 2 * k)
#pragma unroll
        for (int i = 0; i < k; ++i)
          if (i + j + k < 16 && (i + j) / (2 * p) == (i + j + k) / (2 * p)) cswap(s[i + j], s[i + j + k]);
}

// The K most extreme values of the group (largest when TOP), most extreme first, on every lane
// of the group, from each lane's 16 sorted values: a butterfly merge over the group's nl lanes
// (the k-th most extreme of two sorted lists v, w is ext_{i=0..k} inner(v[i-1], w[k-i]) with
// v[-1] = w[-1] = the most extreme value).
template <int K, bool TOP>
__device__ __forceinline__ void octet_topk(const float (&s)[16], int nl, float (&r)[K]) {
#pragma unroll
  for (int i = 0; i < K; ++i) r[i] = TOP ? s[15 - i] : s[i];
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

// n-th and (n-1)-th most extreme values of the group by repeated extraction (any n up to the
// group size; equal values are extracted one at a time, lowest lane first).
template <bool TOP>
__device__ __forceinline__ void octet_extract(const float (&s)[16], int n, int nl, unsigned gmask, int lane,
                                           float& cur, float& prev) {
  int ptr = TOP ? 15 : 0;
  float cand = TOP ? s[15] : s[0];
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
      for (int q = 0; q < 16; ++q)
        if (ptr == q) next = s[q];
      cand = next;
    }
    prev = cur;
    cur = m;
  }
}

template <bool TOP>
__device__ __forceinline__ void octet_order_stats(const float (&s)[16], int n, int nl, unsigned gmask, int lane,
                                                  float& cur, float& prev) {
  switch (n) {
    case 1: { float r[1]; octet_topk<1, TOP>(s, nl, r); cur = prev = r[0]; break; }
    case 2: { float r[2]; octet_topk<2, TOP>(s, nl, r); cur = r[1]; prev = r[0]; break; }
    case 3: { float r[3]; octet_topk<3, TOP>(s, nl, r); cur = r[2]; prev = r[1]; break; }
    case 4: { float r[4]; octet_topk<4, TOP>(s, nl, r); cur = r[3]; prev = r[2]; break; }
    default: octet_extract<TOP>(s, n, nl, gmask, lane, cur, prev); break;
  }
}

// Quantize the octet's row (16 values per lane, Q.nl = G / 16 lanes per group): the lane's 16
// codes and the group's (Delta16, z16) on every lane of the group.  All 32 lanes call it.
__device__ __forceinline__ void quant_octet(const QuantConsts& Q, const float (&y)[16], int lane,
                                            uint32_t (&code)[16], __half2& dz, bool& bad) {
  const int nl = Q.nl;
  const unsigned gmask = ((1u << nl) - 1u) << (lane & ~(nl - 1));
  __half d16, z16;
  if (Q.affine) {
    float hc, hp, lc, lp;
    if (Q.n_hi == 1 && Q.n_lo == 1) {
      // min / max only (kappa = 1)
      float mx = y[0], mn = y[0];
#pragma unroll
      for (int m = 1; m < 16; ++m) {
        mx = fmaxf(mx, y[m]);
        mn = fminf(mn, y[m]);
      }
      for (int o = nl >> 1; o > 0; o >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      }
      hc = hp = mx;
      lc = lp = mn;
    } else {
      float s[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) s[m] = y[m];
      sort16(s);
      octet_order_stats<true>(s, Q.n_hi, nl, gmask, lane, hc, hp);
      octet_order_stats<false>(s, Q.n_lo, nl, gmask, lane, lc, lp);
    }
    const int g = Q.group;
    const float hi = (Q.i_hi >= g - 1) ? hc : __fadd_rn(hc, __fmul_rn(Q.f_hi, __fsub_rn(hp, hc)));
    const float lo = (Q.i_lo >= g - 1) ? lc : __fadd_rn(lp, __fmul_rn(Q.f_lo, __fsub_rn(lc, lp)));
    const float delta = __fdiv_rn(__fsub_rn(hi, lo), 3.0f);
    d16 = __float2half_rn(delta);
    if (__half2float(d16) == 0.0f) d16 = __float2half_rn(1.0f);
    const float z = -__fdiv_rn(lo, __half2float(d16));
    z16 = __float2half_rn(z);
  } else {
    double ss = 0.0;
#pragma unroll
    for (int m = 0; m < 16; ++m) ss = __dadd_rn(ss, __dmul_rn((double)y[m], (double)y[m]));
    for (int o = nl >> 1; o > 0; o >>= 1) ss = __dadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    const double rms = __dsqrt_rn(__ddiv_rn(ss, (double)Q.group));
    const double delta = __ddiv_rn(__dmul_rn(__dmul_rn(2.0, Q.alpha), rms), 3.0);
    d16 = double_to_half_rn(delta);
    if (__half2float(d16) == 0.0f) d16 = __float2half_rn(1.0f);
    z16 = __float2half_rn(1.5f);
  }
  const float df = __half2float(d16), zf = __half2float(z16);
  if (!isfinite(df) || !isfinite(zf)) bad = true;
  float qv[16];
  divn_by_scale<16>(y, df, qv);
#pragma unroll
  for (int m = 0; m < 16; ++m) {
    const int c = __float2int_rn(__fadd_rn(qv[m], zf));
    code[m] = (uint32_t)min(max(c, 0), 3);
  }
  dz = __halves2half2(d16, z16);
}

// OR over the 8 lanes of an octet of eight words, scattered: lane j returns the OR of word j.
__device__ __forceinline__ uint32_t octet_or_scatter(const uint32_t (&w)[8], int j) {
  uint32_t a[4], b[2];
  {
    const bool up = (j & 4) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t send = up ? w[i] : w[4 + i];
      a[i] = (up ? w[4 + i] : w[i]) | __shfl_xor_sync(0xffffffffu, send, 4);
    }
  }
  {
    const bool up = (j & 2) != 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t send = up ? a[i] : a[2 + i];
      b[i] = (up ? a[2 + i] : a[i]) | __shfl_xor_sync(0xffffffffu, send, 2);
    }
  }
  const bool up = (j & 1) != 0;
  const uint32_t send = up ? b[0] : b[1];
  return (up ? b[1] : b[0]) | __shfl_xor_sync(0xffffffffu, send, 1);
}

// l2-scale (keys with key_l2norm), quantize and store the octet's row as token tp of the
// (page, kv head) chunk (nullptr or !valid: computed, nothing stored; key_axis: the page
// layout's key-scale kind, which places the value scales).  y holds channels
// 16 j .. 16 j + 15 (j = lane % 8) and is overwritten.  All 32 lanes call it.
__device__ __forceinline__ void quantize_store_octet(const QuantConsts& Q, bool is_key, bool key_norm,
                                                     float (&y)[16], uint8_t* chunk, int tp, int ng, bool valid,
                                                     int lane, int32_t* status, int key_axis = 0) {
  const int j = lane & 7;
  bool bad = false;
  if (key_norm) {
    double ss = 0.0;
#pragma unroll
    for (int m = 0; m < 16; ++m) ss = __dadd_rn(ss, __dmul_rn((double)y[m], (double)y[m]));
    for (int o = 4; o > 0; o >>= 1) ss = __dadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    const __half s16 = double_to_half_rn(__dsqrt_rn(ss));
    const float sf = __half2float(s16);
    if (!isfinite(sf)) bad = true;
    // every lane divides (the division's warp vote needs the whole warp); a zero norm gives a
    // zero row
    const float sdiv = sf == 0.0f ? 1.0f : sf;
    float yn[16];
    divn_by_scale<16>(y, sdiv, yn);
#pragma unroll
    for (int m = 0; m < 16; ++m) y[m] = sf == 0.0f ? 0.0f : yn[m];
    if (valid && j == 0) reinterpret_cast<__half*>(chunk + norm_off(ng, key_axis))[tp] = s16;
  }
  uint32_t c[16];
  __half2 dz;
  quant_octet(Q, y, lane, c, dz, bad);
  const int nl = Q.nl;
  if (valid && (j & (nl - 1)) == 0) {
    const int g = j / nl;
    if (is_key) {
      *reinterpret_cast<__half2*>(chunk + k_scale_off() + (tp * ng + g) * 4) = dz;
    } else {
      *reinterpret_cast<__half*>(chunk + v_delta_off(ng, tp, g, key_axis)) = __low2half(dz);
      *reinterpret_cast<__half*>(chunk + v_zero_off(ng, tp, g, key_axis)) = __high2half(dz);
    }
  }
  uint32_t w[8];
  if (is_key) {
    // key word k (channel offset 2k within each 16-channel block s): bits 2s and 16 + 2s
    // hold the codes of channels 16s + 2k and 16s + 2k + 1; this lane is block s = j
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = (c[2 * k] << (2 * j)) | (c[2 * k + 1] << (16 + 2 * j));
  } else {
    // value half-word c16 (channels 16m + c16): bits 2m hold the code of channel 16m + c16;
    // this lane is m = j; half-words 2i and 2i + 1 share word i
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = (c[2 * i] << (2 * j)) | (c[2 * i + 1] << (16 + 2 * j));
  }
  const uint32_t word = octet_or_scatter(w, j);
  if (valid) {
    if (is_key) {
      // key word (k = j) of token tp: u32 index 4 l + r with l = 4 (tp % 8) + k % 4,
      // r = 2 (k / 4) + tp / 8
      uint32_t* kw = reinterpret_cast<uint32_t*>(chunk);
      kw[16 * (tp & 7) + 4 * (j & 3) + 2 * (j >> 2) + (tp >> 3)] = word;
    } else {
      // value half-words c16 = 2j, 2j + 1 of token tp: u16 index 2 (4 l + r) + tp % 2 with
      // l = 4 (c16 % 8) + (tp / 2) % 4, r = 2 (tp / 8) + c16 / 8
      uint16_t* vw = reinterpret_cast<uint16_t*>(chunk + kCodeBytes);
      const int base = 8 * ((tp >> 1) & 3) + 4 * (tp >> 3) + (tp & 1);
      const int c0 = 2 * j, c1 = 2 * j + 1;
      vw[32 * (c0 & 7) + 2 * (c0 >> 3) + base] = (uint16_t)(word & 0xffffu);
      vw[32 * (c1 & 7) + 2 * (c1 >> 3) + base] = (uint16_t)(word >> 16);
    }
  }
  if (bad && valid && j == 0) set_status(status, KVQ_ERR_NONFINITE);
}

}  // namespace kvq
