// Correct rounding of transformed rows when the fast paths cannot decide it.
//
// A transformed row is the exact product rounded once to bf16 (nearest-even; an exact zero is
// +0), so that rows -- and the codes quantized from them -- do not depend on summation order
// (WUSH-KV digest, inference algorithm: keys transformed on write; OScaR reading note, step 1:
// Walsh-Hadamard rows).  The fast paths of kv_rotate_qk decide almost every output from an
// fp32 (or tensor-core digit) sum with an error bound; the outputs they leave undecided come
// here and go through two more tiers:
//   tier 2  double-float (error-free products and two-sums, fp32 hi + lo) with a rigorous
//           bound on every rounding it still makes; it decides unless a rounding midpoint lies
//           within that bound (about 2^-44 of the result, or less with cancellation);
//   tier 3  exact: every term as an integer times a power of two, summed in a 576-bit
//           fixed-point accumulator (products of fp32 and bf16 lie in [2^-282, 2^256)), then
//           rounded from the exact integer.  For a Walsh-Hadamard output S / sqrt(128) the exact
//           S is compared with the rounding midpoints m through S^2 against 128 m^2.
// Tier 3 runs serially in one lane: it is reached only for values within the tier-2 bound of
// a midpoint (constructed inputs, or exact ties reached through cancellation).
#pragma once
#include "common.cuh"

namespace kvq {

constexpr int kBigWords = 18;        // 576-bit two's complement accumulator
constexpr int kBigBase = -282;       // value = integer * 2^kBigBase: lowest fp32 x bf16 product exponent

struct BigInt {
  uint32_t w[kBigWords];
};

__device__ inline void big_zero(BigInt& a) {
#pragma unroll
  for (int i = 0; i < kBigWords; ++i) a.w[i] = 0u;
}

// a += (-1)^neg * m * 2^sh, m < 2^32, 0 <= sh <= 511
__device__ inline void big_add(BigInt& a, uint32_t m, int sh, bool neg) {
  const int k = sh >> 5;
  const uint64_t v = (uint64_t)m << (sh & 31);
  const uint32_t lo = (uint32_t)v, hi = (uint32_t)(v >> 32);
  if (!neg) {
    uint64_t s = (uint64_t)a.w[k] + lo;
    a.w[k] = (uint32_t)s;
    s = (uint64_t)a.w[k + 1] + hi + (s >> 32);
    a.w[k + 1] = (uint32_t)s;
    uint32_t c = (uint32_t)(s >> 32);
    for (int i = k + 2; c != 0u && i < kBigWords; ++i) {
      s = (uint64_t)a.w[i] + c;
      a.w[i] = (uint32_t)s;
      c = (uint32_t)(s >> 32);
    }
  } else {
    uint64_t d = (uint64_t)a.w[k] - lo;
    a.w[k] = (uint32_t)d;
    uint32_t b = (uint32_t)(d >> 63);
    d = (uint64_t)a.w[k + 1] - hi - b;
    a.w[k + 1] = (uint32_t)d;
    b = (uint32_t)(d >> 63);
    for (int i = k + 2; b != 0u && i < kBigWords; ++i) {
      d = (uint64_t)a.w[i] - b;
      a.w[i] = (uint32_t)d;
      b = (uint32_t)(d >> 63);
    }
  }
}

// Two's complement -> (magnitude in a, sign returned).
__device__ inline bool big_abs(BigInt& a) {
  const bool neg = (a.w[kBigWords - 1] >> 31) != 0u;
  if (neg) {
    uint32_t c = 1u;
    for (int i = 0; i < kBigWords; ++i) {
      const uint64_t s = (uint64_t)(~a.w[i]) + c;
      a.w[i] = (uint32_t)s;
      c = (uint32_t)(s >> 32);
    }
  }
  return neg;
}

// index of the highest set bit, -1 for zero
__device__ inline int big_top(const uint32_t* w, int n) {
  for (int i = n - 1; i >= 0; --i)
    if (w[i]) return 32 * i + 31 - __clz(w[i]);
  return -1;
}
// bit p of a kBigWords-word integer (0 outside it)
__device__ inline uint32_t big_bit(const uint32_t* w, int p) {
  return (p < 0 || p >= 32 * kBigWords) ? 0u : (w[p >> 5] >> (p & 31)) & 1u;
}
// any set bit at positions [0, p]
__device__ inline bool big_any_below(const uint32_t* w, int p) {
  if (p < 0) return false;
  for (int i = 0; i < (p >> 5); ++i)
    if (w[i]) return true;
  return (w[p >> 5] & (0xffffffffu >> (31 - (p & 31)))) != 0u;
}

// bf16 bits (nearest-even) of (-1)^neg * mag * 2^kBigBase; +0 for zero, infinity on overflow.
__device__ inline uint32_t big_to_bf16(const BigInt& a, bool neg) {
  const int top = big_top(a.w, kBigWords);
  if (top < 0) return 0u;
  int lsb = max(top - 7, 149);                 // 2^-133 (the bf16 subnormal step) is bit 149
  uint32_t q = 0u;
  for (int b = 0; b < 8; ++b) q |= big_bit(a.w, lsb + b) << b;
  const uint32_t rb = big_bit(a.w, lsb - 1);
  const bool sticky = big_any_below(a.w, lsb - 2);
  if (rb && (sticky || (q & 1u))) q += 1u;
  if (q == 256u) {
    q = 128u;
    lsb += 1;
  }
  const int biased = lsb - 148;                // exponent field of q * 2^(lsb + kBigBase), q in [128, 255]
  uint32_t bits;
  if (q < 128u) bits = q;                      // subnormal (lsb == 149)
  else if (biased >= 255) bits = 0x7f80u;
  else bits = ((uint32_t)biased << 7) | (q & 127u);
  return bits | (neg ? 0x8000u : 0u);
}

// (integer significand, exponent) of a float32 / a bf16 value: v = m * 2^e
__device__ inline void split_f32(float f, uint32_t& m, int& e, bool& neg) {
  const uint32_t u = __float_as_uint(f);
  const uint32_t ex = (u >> 23) & 0xffu;
  neg = (u >> 31) != 0u;
  m = (u & 0x7fffffu) | (ex ? 0x800000u : 0u);
  e = (int)(ex ? ex : 1u) - 150;
}
__device__ inline void split_bf16(uint32_t b16, uint32_t& m, int& e, bool& neg) {
  const uint32_t ex = (b16 >> 7) & 0xffu;
  neg = (b16 & 0x8000u) != 0u;
  m = (b16 & 0x7fu) | (ex ? 0x80u : 0u);
  e = (int)(ex ? ex : 1u) - 134;
}

// ---- tier 2 helpers: double-float with a running bound --------------------------------------
constexpr float kU = 0x1p-24f;

// (hi, lo) += a * b, bnd += the bound of the roundings made (products are error-free: an fp32
// times a bf16 has at most 32 significant bits; below 2^-100 the remainder may be rounded,
// covered by 2^-149 per term)
__device__ __forceinline__ void ffb_mac(float& hi, float& lo, float& bnd, float a, float b) {
  const float p = __fmul_rn(a, b);
  const float pe = __fmaf_rn(a, b, -p);
  float s, e;
  two_sum(hi, p, s, e);
  const float t = __fadd_rn(e, pe);
  const float l2 = __fadd_rn(lo, t);
  bnd = __fadd_rn(bnd, __fmaf_rn(kU, __fadd_rn(fabsf(t), fabsf(l2)), 0x1p-149f));
  hi = s;
  lo = l2;
}
// (sh, sl) = (ah, al) + (bh, bl), normalized exactly; the bound grows by the two roundings
__device__ __forceinline__ void ffb_add(float ah, float al, float ab, float bh, float bl, float bb, float& sh,
                                        float& sl, float& sb) {
  float s, e;
  two_sum(ah, bh, s, e);
  const float t = __fadd_rn(al, bl);
  const float e2 = __fadd_rn(e, t);
  two_sum(s, e2, sh, sl);
  sb = __fadd_rn(__fadd_rn(ab, bb), kU * __fadd_rn(fabsf(t), fabsf(e2)));
}

// bf16 bits of V = hi + lo (|lo| <= ulp(hi) / 2) when every value within B of V rounds alike;
// -1 when that cannot be decided here (B straddles a midpoint, V is zero or rounds to zero, or
// |V| > 2^120).  Non-finite hi gives the bits of ff_to_bf16.
__device__ inline int ffb_decide(float hi, float lo, float B) {
  if (!isfinite(hi)) return (int)ff_to_bf16(hi, lo);
  const bool neg = hi < 0.f;
  const float h = fabsf(hi), l = neg ? -lo : lo;
  if (!(h > 0.f && h <= 0x1p+120f)) return -1;
  const uint32_t b = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(h));
  if (b == 0u) return -1;                                          // below half the smallest bf16
  const float bv = __uint_as_float(b << 16);
  const float m_lo = 0.5f * (bv + __uint_as_float((b - 1u) << 16));   // exact: 9 significant bits
  const float m_hi = 0.5f * (bv + __uint_as_float((b + 1u) << 16));
  const float r1 = __fadd_rn(h - m_lo, l);                          // h - m_lo, m_hi - h exact (Sterbenz)
  const float r2 = __fadd_rn(m_hi - h, -l);
  const float Bs = __fmaf_rn(B, 1.0f + 0x1p-16f, 0x1p-140f);
  // V - m_lo and m_hi - V, each within u |r| + Bs of r1, r2.  h lies in b's cell, |l| is far
  // below a bf16 step, so V is in b's cell or just across one of its two midpoints (h itself
  // on a midpoint, l deciding the side).
  const float s1 = __fmaf_rn(-kU, fabsf(r1), fabsf(r1)), s2 = __fmaf_rn(-kU, fabsf(r2), fabsf(r2));
  uint32_t res;
  if (r1 > 0.f && r2 > 0.f && s1 > Bs && s2 > Bs) res = b;            // inside b's cell
  else if (r1 < 0.f && s1 > Bs) res = b - 1u;                         // below m_lo
  else if (r2 < 0.f && s2 > Bs) res = b + 1u;                         // above m_hi
  else return -1;
  return (int)(res | (neg ? 0x8000u : 0u));
}

// ---- dense outputs --------------------------------------------------------------------------
// Tier 3 of a dense output: lane 0 sums every term exactly (the terms reach it through
// shuffles); every lane returns the bf16 bits.  Out of line: it runs only for outputs within the
// tier-2 bound of a midpoint.
static __device__ __noinline__ uint32_t exact_dot_tier3(float4 t4, float4 x4, int lane) {
  BigInt acc;
  if (lane == 0) big_zero(acc);
#pragma unroll 1
  for (int src = 0; src < 32; ++src) {
    const float tv[4] = {__shfl_sync(0xffffffffu, t4.x, src), __shfl_sync(0xffffffffu, t4.y, src),
                         __shfl_sync(0xffffffffu, t4.z, src), __shfl_sync(0xffffffffu, t4.w, src)};
    const float xv[4] = {__shfl_sync(0xffffffffu, x4.x, src), __shfl_sync(0xffffffffu, x4.y, src),
                         __shfl_sync(0xffffffffu, x4.z, src), __shfl_sync(0xffffffffu, x4.w, src)};
    if (lane == 0) {
#pragma unroll 1
      for (int k = 0; k < 4; ++k) {
        uint32_t ma, mx;
        int ea, ex;
        bool na, nx;
        split_f32(tv[k], ma, ea, na);
        split_bf16(__float_as_uint(xv[k]) >> 16, mx, ex, nx);
        const uint32_t m = ma * mx;                        // < 2^32, exact
        if (m) big_add(acc, m, ea + ex - kBigBase, na != nx);
      }
    }
  }
  uint32_t r = 0u;
  if (lane == 0) {
    const bool neg = big_abs(acc);
    r = big_to_bf16(acc, neg);
  }
  return __shfl_sync(0xffffffffu, r, 0);
}



// Tier 2 alone: the bf16 bits, or -1 when only tier 3 can decide (same value in every lane).
__device__ __forceinline__ int exact_dot_tier2(float4 t4, float4 x4) {
  float hi = 0.f, lo = 0.f, bnd = 0.f;
  ffb_mac(hi, lo, bnd, t4.x, x4.x);
  ffb_mac(hi, lo, bnd, t4.y, x4.y);
  ffb_mac(hi, lo, bnd, t4.z, x4.z);
  ffb_mac(hi, lo, bnd, t4.w, x4.w);
#pragma unroll
  for (int s2 = 16; s2 > 0; s2 >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, hi, s2);
    const float ol = __shfl_xor_sync(0xffffffffu, lo, s2);
    const float ob = __shfl_xor_sync(0xffffffffu, bnd, s2);
    ffb_add(hi, lo, bnd, oh, ol, ob, hi, lo, bnd);       // symmetric: every lane gets the same bits
  }
  return ffb_decide(hi, lo, bnd);
}

// Tier 2 by one thread over a whole row: sum_j t_j x_j for j < 128 with t float32 (16-byte
// aligned) and x bf16 (8-byte aligned), in order, with the same tracked bound (rigorous in any
// order) and an exact renormalization every 16 terms (ffb_decide needs |lo| <= ulp(hi) / 2);
// the bf16 bits, or -1 when only tier 3 can decide.  Lets a warp take 32 outputs at once.
__device__ __forceinline__ int exact_dot_tier2_row(const float* trow, const uint16_t* xrow) {
  float hi = 0.f, lo = 0.f, bnd = 0.f;
#pragma unroll 4
  for (int j = 0; j < 32; ++j) {
    const float4 t4 = __ldg(reinterpret_cast<const float4*>(trow) + j);
    const uint2 xr = __ldg(reinterpret_cast<const uint2*>(xrow) + j);
    ffb_mac(hi, lo, bnd, t4.x, __uint_as_float(xr.x << 16));
    ffb_mac(hi, lo, bnd, t4.y, __uint_as_float(xr.x & 0xffff0000u));
    ffb_mac(hi, lo, bnd, t4.z, __uint_as_float(xr.y << 16));
    ffb_mac(hi, lo, bnd, t4.w, __uint_as_float(xr.y & 0xffff0000u));
    if ((j & 3) == 3) two_sum(hi, lo, hi, lo);           // exact: keeps lo below half an ulp of hi
  }
  return ffb_decide(hi, lo, bnd);
}

// bf16 bits of the exact sum_j t_j x_j over one warp: lane l holds terms 4l .. 4l + 3 (t float32,
// x bf16 values held exactly as floats).  Every lane returns the result.  Tier 2 inline, tier 3
// out of line.
__device__ __forceinline__ uint32_t exact_dot_bf16_warp(float4 t4, float4 x4, int lane) {
  const int d = exact_dot_tier2(t4, x4);
  return d >= 0 ? (uint32_t)d : exact_dot_tier3(t4, x4, lane);
}

// ---- Walsh-Hadamard outputs -----------------------------------------------------------------
// Compare A (n words) with q * 2^sh (q > 0): -1, 0, 1.
__device__ inline int big_cmp_q(const uint32_t* A, int n, uint64_t q, int sh) {
  const int LA = big_top(A, n) + 1;
  const int LQ = 64 - __clzll((long long)q);
  if (LA != LQ + sh) return LA > LQ + sh ? 1 : -1;
  // equal lengths: A's top LQ bits against q, then A's remaining low bits
  uint64_t top = 0;
  for (int b = 0; b < LQ; ++b) top |= (uint64_t)big_bit(A, LA - LQ + b) << b;
  if (top != q) return top > q ? 1 : -1;
  return big_any_below(A, LA - LQ - 1) ? 1 : 0;
}

// bf16 bits of S / sqrt(128) for the exact S = sum_j (-1)^popcount(i & j) x_j (row src, bf16)
// starting from an estimate `guess` (bf16 bits): S is summed exactly, then each rounding
// midpoint m is compared with |S| / sqrt(128) through S^2 against 128 m^2.  Never a tie
// (sqrt(2) is irrational) unless S = 0, which gives +0.
static __device__ __noinline__ uint32_t exact_wht_output(const uint16_t* src, int i, uint32_t guess) {
  BigInt acc;
  big_zero(acc);
  for (int j = 0; j < kHeadDim; ++j) {
    uint32_t m;
    int e;
    bool ng;
    split_bf16(src[j], m, e, ng);
    if (m) big_add(acc, m, e - kBigBase, ng != ((__popc(i & j) & 1) != 0));
  }
  const bool neg = big_abs(acc);
  const int top = big_top(acc.w, kBigWords);
  if (top < 0) return 0u;
  // |S| = S' 2^(tz + kBigBase) with S' odd and at most 288 bits wide (bf16 sums span < 288 bits)
  int tz = 0;
  while (!big_bit(acc.w, tz)) ++tz;
  uint32_t s[9];
  for (int k = 0; k < 9; ++k) {
    uint32_t v = 0u;
    for (int b = 0; b < 32; ++b) v |= big_bit(acc.w, tz + 32 * k + b) << b;
    s[k] = v;
  }
  // S'^2 (18 words)
  uint32_t sq[18];
  for (int k = 0; k < 18; ++k) sq[k] = 0u;
  for (int a = 0; a < 9; ++a) {
    uint64_t carry = 0;
    for (int b = 0; b < 9; ++b) {
      const uint64_t cur = (uint64_t)s[a] * s[b] + sq[a + b] + carry;
      sq[a + b] = (uint32_t)cur;
      carry = cur >> 32;
    }
    for (int k = a + 9; carry != 0u && k < 18; ++k) {
      const uint64_t cur = (uint64_t)sq[k] + carry;
      sq[k] = (uint32_t)cur;
      carry = cur >> 32;
    }
  }
  // |y| > m  <=>  S'^2 2^(2 (tz + kBigBase)) > 128 m^2 = mq^2 2^(2 me + 7), with m = mq 2^me
  auto above = [&](uint32_t mbits_f32) -> int {          // sign of |y| - m for a positive float m
    uint32_t mq;
    int me;
    bool dummy;
    split_f32(__uint_as_float(mbits_f32), mq, me, dummy);
    const int sh = 2 * me + 7 - 2 * (tz + kBigBase);
    const uint64_t q2 = (uint64_t)mq * mq;
    if (sh < 0) {
      // compare S'^2 2^-sh with q2: S'^2 against q2 >> -sh is not exact, so shift S'^2 up instead
      // by comparing lengths (S'^2 has at least one bit; q2 < 2^48)
      const int LS = big_top(sq, 18) + 1 - sh;           // length of S'^2 2^-sh
      const int LQ = 64 - __clzll((long long)q2);
      if (LS != LQ) return LS > LQ ? 1 : -1;
      // same length (< 49 bits): S'^2 fits in 64 bits here
      const uint64_t sv = ((uint64_t)sq[1] << 32 | sq[0]) << (-sh);
      return sv > q2 ? 1 : (sv < q2 ? -1 : 0);
    }
    return big_cmp_q(sq, 18, q2, sh);
  };
  // walk from the estimate to the bf16 value whose rounding cell holds |y|
  uint32_t b = guess & 0x7fffu;
  if (b > 0x7f7fu) b = 0x7f7fu;
  for (int it = 0; it < 64; ++it) {
    const float bv = __uint_as_float(b << 16);
    const float m_hi = 0.5f * (bv + __uint_as_float((b + 1u) << 16));
    if (b < 0x7f7fu && above(__float_as_uint(m_hi)) > 0) { ++b; continue; }
    if (b > 0u) {
      const float m_lo = 0.5f * (bv + __uint_as_float((b - 1u) << 16));
      if (above(__float_as_uint(m_lo)) < 0) { --b; continue; }
    }
    break;
  }
  // beyond the largest finite bf16's cell, 2^127 (2 - 2^-8), the result is infinity
  if (b == 0x7f7fu && above(__float_as_uint(0x1.ffp+127f)) >= 0) b = 0x7f80u;
  return b | (neg ? 0x8000u : 0u);
}

}  // namespace kvq
