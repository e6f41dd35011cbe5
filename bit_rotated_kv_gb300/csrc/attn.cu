// kv_attn_decode: GQA decode attention over the mixed cache (BF16 sink | INT2 pages |
// BF16 recent ring), split over the token axis with an in-kernel online-softmax merge.
//
// Source: OSCAR summary, section 4 "Decoding Attention Kernel" (partition the cache into
// BF16 and INT2 segments, unpack INT2 and accumulate in floating point; existing kernels
// needed two launches plus a merge); OScaR reading note, "系统设计与 CUDA 实现"
// (INT2 tiles dequantized in registers: x Delta, - z, x s_t, inside split attention) and
// Algorithm 1 steps 14-17; WUSH-KV digest, GQA background (n_q/n_kv query heads read
// one kv head); decode attention softmax(q K^T / sqrt(d)) V.
//
// Design (GB300, sm_103a):
//  * grid (splits, kv_head, sequence); splits [0, n_int2) stream INT2 pages, the rest
//    the BF16 windows.  Every warp owns a private ring of STAGES page slots in shared
//    memory filled by 1-D TMA bulk copies (cp.async.bulk + mbarrier complete_tx); lane
//    0 issues, all lanes wait with a bounded try_wait loop.  No cluster, no multicast.
//  * one page (16 tokens) is one m16n8k16 tile: scores S[token][head] = codes x q',
//    all g <= 8 query heads of the kv head share the read (N = 8 columns).
//  * 2-bit codes become fp16 tensor-core operands with one AND each: a code c at bit
//    position 2s of a 16-bit half is the fp16 subnormal c * 4^s * 2^-24, exact; the
//    4^s and 2^-24 factors are folded into q' (keys) or the output rows (values).  The
//    group scale / zero point and the l2 norm are applied to the fp32 scores:
//    s = norm * sum_g Delta_g (q'.c_g - z_g sum(q'_g)).
//  * P V: the fp32 probabilities times Delta_v become the B operand through
//    movmatrix (C-fragment -> B-fragment transpose); the zero point is a per-group
//    correction sum_t W_t z_t.
//  * BF16 windows use bf16 MMA for q'.k (exact inputs) and two bf16 MMAs (hi + lo
//    split of P) for P V.
//  * the last CTA of each (sequence, kv head) merges the split partials (atomic ticket,
//    no spin wait) and writes out = acc / l.
#include "common.cuh"
#include "launch.h"

#include <mutex>

namespace kvq {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 8;
constexpr long long kWaitLimit = 1LL << 22;

struct AttnParams {
  const uint8_t* pages;
  const int32_t* page_table;
  const int32_t* seq_len;
  const int32_t* s_quant;
  const uint16_t* sink_k;
  const uint16_t* sink_v;
  const uint16_t* ring_k;
  const uint16_t* ring_v;
  const uint16_t* q;
  float* out;
  float* part;        // [B][Hkv][n_split][g][2 + d]
  int32_t* count;     // [B][Hkv]
  int32_t* status;
  int batch, hkv, gqa, s_sink, ring_cap, max_pages, num_pages, group, l2, page_bytes;
  int n_int2, n_win, n_split;
  float scale_log2;   // sm_scale * log2(e)
};

// ---- PTX helpers ----------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; false when the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (long long i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf162(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_half2(uint32_t x) {
  __half2 h = *reinterpret_cast<__half2*>(&x);
  return __half22float2(h);
}
__device__ __forceinline__ float2 unpack_bf162(uint32_t x) {
  return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}

// Code slot s (0..7) of a fragment word as an fp16x2 pair of subnormals c * 4^k * 2^-24,
// k = s (s <= 4) or s - 5 (s >= 5, taken from the word shifted right by 10).
__device__ __forceinline__ uint32_t code_pair(uint32_t w, uint32_t w10, int s) {
  return s <= 4 ? (w & (0x00030003u << (2 * s))) : (w10 & (0x00030003u << (2 * (s - 5))));
}
__host__ __device__ __forceinline__ int slot_pow(int s) { return s <= 4 ? s : s - 5; }

// Online-softmax state of one warp for the two head columns 2*(lane%4) + {0, 1}.
struct Softmax {
  float m[2], l[2];
};

// Fold a page / tile of scores s[t][c] (C fragment: t in {lane/4, lane/4 + 8}, c = column
// pair) into the running max; returns the rescale factors and the probabilities.
__device__ __forceinline__ void softmax_step(Softmax& sm, float (&s)[4], float (&p)[4], float (&alpha)[2]) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    float mx = fmaxf(s[c], s[c + 2]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    float mn = fmaxf(sm.m[c], mx);
    alpha[c] = (mn == -INFINITY) ? 1.0f : exp2f(sm.m[c] - mn);
    float mu = (mn == -INFINITY) ? 0.0f : mn;
    p[c] = exp2f(s[c] - mu);
    p[c + 2] = exp2f(s[c + 2] - mu);
    sm.m[c] = mn;
    sm.l[c] = sm.l[c] * alpha[c] + p[c] + p[c + 2];
  }
}

// ---- shared memory layout ---------------------------------------------------------------
struct __align__(16) QShared {
  float mult[kMaxGqa];        // 2^(24 - sigma_h)
  float qsum[kMaxGqa][4];     // sum of q' over each group
};

// Per-warp result in canonical order: for each head (m, l, o[d]); warps `wstride` floats apart.
__device__ __forceinline__ float* warp_result(float* base, int warp, size_t wstride) {
  return base + (size_t)warp * wstride;
}

// ---- INT2 pages ----------------------------------------------------------------------------
template <int NG>
__device__ void int2_split(const AttnParams& P, uint8_t* smem, int b, int h, int split, float* res,
                           size_t wstride) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = P.gqa;
  const int L = P.seq_len[b];
  const int sq = min(P.s_quant[b], L);
  const int n_tok = max(0, sq - P.s_sink);
  const int np = (n_tok + kPage - 1) / kPage;
  const int p0 = (int)((long long)np * split / P.n_int2);
  const int p1 = (int)((long long)np * (split + 1) / P.n_int2);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);                      // [kWarps][kStages]
  int* slot_pid = reinterpret_cast<int*>(smem + kWarps * kStages * 8);     // [kWarps][kStages]
  QShared* qs = reinterpret_cast<QShared*>(smem + kWarps * kStages * 12);
  uint8_t* ring = smem + 1024;                                             // [kWarps][kStages][page_bytes]
  const int pb = P.page_bytes;
  uint8_t* my_ring = ring + (size_t)warp * kStages * pb;
  uint64_t* my_bars = bars + warp * kStages;
  int* my_pid = slot_pid + warp * kStages;

  // ---- queries: B fragments scaled to fp16 range, per-head multipliers and group sums
  const uint16_t* qb = P.q + ((size_t)b * P.hkv * g + (size_t)h * g) * kHeadDim;
  const int hrow = lane >> 2, quad = lane & 3;
  uint32_t bq[8][2];
  {
    float qv[8][4];
    float amax = 0.f;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        int ch = 16 * s + 2 * quad + (e & 1) + 8 * (e >> 1);
        float x = (hrow < g) ? bf16_bits_to_float(qb[(size_t)hrow * kHeadDim + ch]) : 0.f;
        qv[s][e] = x;
        amax = fmaxf(amax, fabsf(x));
      }
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int sigma = 0;
    if (amax > 0.f) {
      int e2;
      frexpf(amax, &e2);       // amax in [2^(e2-1), 2^e2)
      sigma = 14 - e2;         // amax * 2^sigma < 2^14
    }
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      float f = ldexpf(1.0f, sigma - 2 * slot_pow(s));
      bq[s][0] = pack_half2(qv[s][0] * f, qv[s][1] * f);
      bq[s][1] = pack_half2(qv[s][2] * f, qv[s][3] * f);
    }
    // group sums: lanes of one head cover all channels
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      float acc = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s)
        if ((16 * s) / (kHeadDim / NG) == gi) acc += qv[s][0] + qv[s][1] + qv[s][2] + qv[s][3];
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      if (warp == 0 && quad == 0) qs->qsum[hrow][gi] = acc;
    }
    if (warp == 0 && quad == 0) qs->mult[hrow] = ldexpf(1.0f, 24 - sigma);
  }
  if (lane < kStages) mbar_init(my_bars + lane, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();

  const int hA = 2 * quad, hB = 2 * quad + 1;
  const float multA = qs->mult[hA], multB = qs->mult[hB];
  float qsA[NG], qsB[NG];
#pragma unroll
  for (int gi = 0; gi < NG; ++gi) { qsA[gi] = qs->qsum[hA][gi]; qsB[gi] = qs->qsum[hB][gi]; }

  // ---- this warp's pages: p0 + warp + k * kWarps
  const int first = p0 + warp;
  const int nk = first < p1 ? (p1 - first + kWarps - 1) / kWarps : 0;
  const int32_t* ptab = P.page_table + (size_t)b * P.max_pages;
  auto issue = [&](int k) {
    int slot = k % kStages;
    int lp = first + k * kWarps;
    int pid = (lp < P.max_pages) ? ptab[lp] : -1;
    if (pid < 0 || pid >= P.num_pages) {
      set_status(P.status, KVQ_ERR_BOUNDS);
      my_pid[slot] = -1;
      mbar_arrive(my_bars + slot);
    } else {
      my_pid[slot] = pid;
      fence_proxy_async();
      mbar_arrive_tx(my_bars + slot, (uint32_t)pb);
      tma_load_1d(my_ring + (size_t)slot * pb, P.pages + ((size_t)pid * P.hkv + h) * pb, (uint32_t)pb,
                  my_bars + slot);
    }
  };
  if (lane == 0)
    for (int k = 0; k < min(nk, kStages); ++k) issue(k);
  __syncwarp();

  Softmax sm;
  sm.m[0] = sm.m[1] = -INFINITY;
  sm.l[0] = sm.l[1] = 0.f;
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[mt][c] = 0.f;
  float zc[2][NG];
#pragma unroll
  for (int gi = 0; gi < NG; ++gi) zc[0][gi] = zc[1][gi] = 0.f;

  const int tA = lane >> 2, tB = tA + 8;
  const int ng_off_v = v_scale_off(NG);
  bool timed_out = false;
  int k = 0;
  for (; k < nk; ++k) {
    const int slot = k % kStages;
    if (!mbar_wait(my_bars + slot, (uint32_t)((k / kStages) & 1))) {
      timed_out = true;
      break;
    }
    const uint8_t* pg = my_ring + (size_t)slot * pb;
    const int pid = my_pid[slot];
    const int lp = first + k * kWarps;
    const int valid_tok = (pid < 0) ? 0 : min(kPage, n_tok - kPage * lp);
    // fragments and scales
    uint4 wk = *reinterpret_cast<const uint4*>(pg + 16 * lane);
    uint4 wv = *reinterpret_cast<const uint4*>(pg + kCodeBytes + 16 * lane);
    float dkA[NG], zkA[NG], dkB[NG], zkB[NG], dvA[NG], zvA[NG], dvB[NG], zvB[NG];
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      float2 a = unpack_half2(*reinterpret_cast<const uint32_t*>(pg + k_scale_off() + (tA * NG + gi) * 4));
      float2 bb = unpack_half2(*reinterpret_cast<const uint32_t*>(pg + k_scale_off() + (tB * NG + gi) * 4));
      float2 c = unpack_half2(*reinterpret_cast<const uint32_t*>(pg + ng_off_v + (tA * NG + gi) * 4));
      float2 d = unpack_half2(*reinterpret_cast<const uint32_t*>(pg + ng_off_v + (tB * NG + gi) * 4));
      dkA[gi] = a.x; zkA[gi] = a.y; dkB[gi] = bb.x; zkB[gi] = bb.y;
      const bool vA = tA < valid_tok, vB = tB < valid_tok;
      dvA[gi] = vA ? c.x : 0.f; zvA[gi] = vA ? c.y : 0.f;
      dvB[gi] = vB ? d.x : 0.f; zvB[gi] = vB ? d.y : 0.f;
    }
    float nA = 1.f, nB = 1.f;
    if (P.l2) {
      const __half* nrm = reinterpret_cast<const __half*>(pg + norm_off(NG));
      nA = __half2float(nrm[tA]);
      nB = __half2float(nrm[tB]);
    }
    // ---- scores: codes x q' per group
    const uint32_t kw[4] = {wk.x, wk.y, wk.z, wk.w};
    const uint32_t kw10[4] = {wk.x >> 10, wk.y >> 10, wk.z >> 10, wk.w >> 10};
    float acc[NG][4];
#pragma unroll
    for (int gi = 0; gi < NG; ++gi)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[gi][c] = 0.f;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      uint32_t a[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = code_pair(kw[r], kw10[r], s);
      mma_f16(acc[(16 * s) / (kHeadDim / NG)], a, bq[s][0], bq[s][1]);
    }
    float sc[4];
    {
      float sA0 = 0.f, sA1 = 0.f, sB0 = 0.f, sB1 = 0.f;
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        sA0 += dkA[gi] * (acc[gi][0] * multA - zkA[gi] * qsA[gi]);
        sA1 += dkA[gi] * (acc[gi][1] * multB - zkA[gi] * qsB[gi]);
        sB0 += dkB[gi] * (acc[gi][2] * multA - zkB[gi] * qsA[gi]);
        sB1 += dkB[gi] * (acc[gi][3] * multB - zkB[gi] * qsB[gi]);
      }
      const float cA = P.scale_log2 * nA, cB = P.scale_log2 * nB;
      const bool vA = tA < valid_tok, vB = tB < valid_tok;
      sc[0] = vA ? sA0 * cA : -INFINITY;
      sc[1] = vA ? sA1 * cA : -INFINITY;
      sc[2] = vB ? sB0 * cB : -INFINITY;
      sc[3] = vB ? sB1 * cB : -INFINITY;
    }
    float p[4], alpha[2];
    softmax_step(sm, sc, p, alpha);
    if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= alpha[0]; o[mt][2] *= alpha[0];
        o[mt][1] *= alpha[1]; o[mt][3] *= alpha[1];
      }
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) { zc[0][gi] *= alpha[0]; zc[1][gi] *= alpha[1]; }
    }
    // ---- P V: per value group, W = P * Delta_v as the B operand (fp16)
    uint32_t bw[NG][2];
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      uint32_t wa = pack_half2(p[0] * dvA[gi], p[1] * dvA[gi]);   // token tA, heads hA, hB
      uint32_t wb = pack_half2(p[2] * dvB[gi], p[3] * dvB[gi]);   // token tB
      float2 fa = unpack_half2(wa), fb = unpack_half2(wb);
      zc[0][gi] += fa.x * zvA[gi] + fb.x * zvB[gi];
      zc[1][gi] += fa.y * zvA[gi] + fb.y * zvB[gi];
      bw[gi][0] = movmatrix_trans(wa);
      bw[gi][1] = movmatrix_trans(wb);
    }
    const uint32_t vw[4] = {wv.x, wv.y, wv.z, wv.w};
    const uint32_t vw10[4] = {wv.x >> 10, wv.y >> 10, wv.z >> 10, wv.w >> 10};
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t a[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = code_pair(vw[r], vw10[r], mt);
      const int gi = (16 * mt) / (kHeadDim / NG);
      mma_f16(o[mt], a, bw[gi][0], bw[gi][1]);
    }
    // every lane has consumed this slot: refill it with the page kStages ahead
    __syncwarp();
    if (lane == 0 && k + kStages < nk) issue(k + kStages);
  }
  if (timed_out) {
    if (lane == 0) set_status(P.status, KVQ_ERR_TIMEOUT);
    // let copies still in flight land before the CTA can exit (bounded)
    for (int kk = k; kk < min(nk, k + kStages); ++kk)
      (void)mbar_wait(my_bars + kk % kStages, (uint32_t)((kk / kStages) & 1));
  }

  // ---- per-warp result: reduce l and z-corrections over the 8 lanes of a column pair
#pragma unroll
  for (int c = 0; c < 2; ++c) {
#pragma unroll
    for (int o2 = 4; o2 < 32; o2 <<= 1) {
      sm.l[c] += __shfl_xor_sync(0xffffffffu, sm.l[c], o2);
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) zc[c][gi] += __shfl_xor_sync(0xffffffffu, zc[c][gi], o2);
    }
  }
  float* wr = warp_result(res, warp, wstride);
  if (hA < g) {
    if (tA == 0) { wr[hA * (2 + kHeadDim)] = sm.m[0]; wr[hA * (2 + kHeadDim) + 1] = sm.l[0]; }
  }
  if (hB < g) {
    if (tA == 0) { wr[hB * (2 + kHeadDim)] = sm.m[1]; wr[hB * (2 + kHeadDim) + 1] = sm.l[1]; }
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const float f = ldexpf(1.0f, 24 - 2 * slot_pow(mt));
    const int gi = (16 * mt) / (kHeadDim / NG);
    const int ch0 = 16 * mt + tA, ch1 = ch0 + 8;
    if (hA < g) {
      wr[hA * (2 + kHeadDim) + 2 + ch0] = o[mt][0] * f - zc[0][gi];
      wr[hA * (2 + kHeadDim) + 2 + ch1] = o[mt][2] * f - zc[0][gi];
    }
    if (hB < g) {
      wr[hB * (2 + kHeadDim) + 2 + ch0] = o[mt][1] * f - zc[1][gi];
      wr[hB * (2 + kHeadDim) + 2 + ch1] = o[mt][3] * f - zc[1][gi];
    }
  }
}

// ---- BF16 windows --------------------------------------------------------------------------
__device__ void window_split(const AttnParams& P, int b, int h, int wsplit, float* res, size_t wstride) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = P.gqa;
  const int L = P.seq_len[b];
  const int n_sink = min(P.s_sink, max(L, 0));
  const int r0 = max(min(P.s_quant[b], L), P.s_sink);     // first recent token
  const int n_sink_t = (n_sink + kPage - 1) / kPage;
  const int rt0 = r0 / kPage;
  const int n_rec_t = (L > r0) ? ((L - 1) / kPage - rt0 + 1) : 0;
  const int nt = n_sink_t + n_rec_t;
  const int t0 = (int)((long long)nt * wsplit / P.n_win);
  const int t1 = (int)((long long)nt * (wsplit + 1) / P.n_win);

  const int quad = lane & 3, hrow = lane >> 2;
  const int hA = 2 * quad, hB = hA + 1;
  // q' B fragments (bf16, exact): head lane/4, channels 32*(lane%4) + 4s + {0,1} / {2,3}
  uint32_t bq[8][2];
  {
    const uint16_t* qrow = P.q + (((size_t)b * P.hkv + h) * g + hrow) * kHeadDim + 32 * quad;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      if (hrow < g) {
        uint2 v2 = *reinterpret_cast<const uint2*>(qrow + 4 * s);
        bq[s][0] = v2.x;
        bq[s][1] = v2.y;
      } else {
        bq[s][0] = bq[s][1] = 0u;
      }
    }
  }
  Softmax sm;
  sm.m[0] = sm.m[1] = -INFINITY;
  sm.l[0] = sm.l[1] = 0.f;
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[mt][c] = 0.f;

  const int tA = lane >> 2, tB = tA + 8;
  for (int ti = t0 + warp; ti < t1; ti += kWarps) {
    // token range of this tile and where its rows live
    const uint16_t *kbase, *vbase;
    int tok0, lo, hi, rows_avail;
    if (ti < n_sink_t) {
      tok0 = ti * kPage;
      lo = tok0;
      hi = min(tok0 + kPage, n_sink);
      const size_t off = ((size_t)b * P.hkv + h) * P.s_sink * kHeadDim + (size_t)tok0 * kHeadDim;
      kbase = P.sink_k + off;
      vbase = P.sink_v + off;
      rows_avail = hi - tok0;                 // rows beyond the sink buffer are never read
    } else {
      tok0 = (rt0 + ti - n_sink_t) * kPage;
      lo = max(tok0, r0);
      hi = min(tok0 + kPage, L);
      const size_t off = (((size_t)b * P.hkv + h) * P.ring_cap + (tok0 % P.ring_cap)) * kHeadDim;
      kbase = P.ring_k + off;
      vbase = P.ring_v + off;
      rows_avail = kPage;
    }
    auto row_ok = [&](int t) { return tok0 + t >= lo && tok0 + t < hi; };
    auto row_ptr = [&](const uint16_t* base, int t) { return base + (size_t)(t < rows_avail ? t : 0) * kHeadDim; };
    // ---- scores (bf16 MMA): K rows tA, tB, channels 32*quad .. +32
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const uint4* ka = reinterpret_cast<const uint4*>(row_ptr(kbase, tA) + 32 * quad);
      const uint4* kb = reinterpret_cast<const uint4*>(row_ptr(kbase, tB) + 32 * quad);
      uint32_t ra[16], rb[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint4 x = ka[i], y = kb[i];
        ra[4 * i] = x.x; ra[4 * i + 1] = x.y; ra[4 * i + 2] = x.z; ra[4 * i + 3] = x.w;
        rb[4 * i] = y.x; rb[4 * i + 1] = y.y; rb[4 * i + 2] = y.z; rb[4 * i + 3] = y.w;
      }
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t a[4] = {ra[2 * s], rb[2 * s], ra[2 * s + 1], rb[2 * s + 1]};
        mma_bf16(acc, a, bq[s][0], bq[s][1]);
      }
    }
    float sc[4];
    sc[0] = row_ok(tA) ? acc[0] * P.scale_log2 : -INFINITY;
    sc[1] = row_ok(tA) ? acc[1] * P.scale_log2 : -INFINITY;
    sc[2] = row_ok(tB) ? acc[2] * P.scale_log2 : -INFINITY;
    sc[3] = row_ok(tB) ? acc[3] * P.scale_log2 : -INFINITY;
    float p[4], alpha[2];
    softmax_step(sm, sc, p, alpha);
    if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= alpha[0]; o[mt][2] *= alpha[0];
        o[mt][1] *= alpha[1]; o[mt][3] *= alpha[1];
      }
    }
    // ---- P V: P = P_hi + P_lo in bf16, two MMAs per 16 channels
    uint32_t bh[2], bl[2];
    {
      uint32_t h0 = pack_bf162(p[0], p[1]);
      uint32_t h1 = pack_bf162(p[2], p[3]);
      float2 f0 = unpack_bf162(h0), f1 = unpack_bf162(h1);
      uint32_t l0 = pack_bf162(p[0] - f0.x, p[1] - f0.y);
      uint32_t l1 = pack_bf162(p[2] - f1.x, p[3] - f1.y);
      bh[0] = movmatrix_trans(h0); bh[1] = movmatrix_trans(h1);
      bl[0] = movmatrix_trans(l0); bl[1] = movmatrix_trans(l1);
    }
    // V rows 2q, 2q+1, 2q+8, 2q+9, channels 16*(lane/4) .. +16
    uint32_t vr[4][8];
    const int vt[4] = {2 * quad, 2 * quad + 1, 2 * quad + 8, 2 * quad + 9};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4* src = reinterpret_cast<const uint4*>(row_ptr(vbase, vt[i]) + 16 * hrow);
      uint4 x = src[0], y = src[1];
      const bool ok = row_ok(vt[i]);
      vr[i][0] = ok ? x.x : 0u; vr[i][1] = ok ? x.y : 0u; vr[i][2] = ok ? x.z : 0u; vr[i][3] = ok ? x.w : 0u;
      vr[i][4] = ok ? y.x : 0u; vr[i][5] = ok ? y.y : 0u; vr[i][6] = ok ? y.z : 0u; vr[i][7] = ok ? y.w : 0u;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t a[4];
      a[0] = __byte_perm(vr[0][mt], vr[1][mt], 0x5410);   // channel 16*hrow + 2mt, tokens 2q, 2q+1
      a[1] = __byte_perm(vr[0][mt], vr[1][mt], 0x7632);   // channel + 1
      a[2] = __byte_perm(vr[2][mt], vr[3][mt], 0x5410);   // tokens 2q+8, 2q+9
      a[3] = __byte_perm(vr[2][mt], vr[3][mt], 0x7632);
      mma_bf16(o[mt], a, bh[0], bh[1]);
      mma_bf16(o[mt], a, bl[0], bl[1]);
    }
  }
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int o2 = 4; o2 < 32; o2 <<= 1) sm.l[c] += __shfl_xor_sync(0xffffffffu, sm.l[c], o2);
  float* wr = warp_result(res, warp, wstride);
  if (hA < g && tA == 0) { wr[hA * (2 + kHeadDim)] = sm.m[0]; wr[hA * (2 + kHeadDim) + 1] = sm.l[0]; }
  if (hB < g && tA == 0) { wr[hB * (2 + kHeadDim)] = sm.m[1]; wr[hB * (2 + kHeadDim) + 1] = sm.l[1]; }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int ch0 = 16 * hrow + 2 * mt, ch1 = ch0 + 1;
    if (hA < g) { wr[hA * (2 + kHeadDim) + 2 + ch0] = o[mt][0]; wr[hA * (2 + kHeadDim) + 2 + ch1] = o[mt][2]; }
    if (hB < g) { wr[hB * (2 + kHeadDim) + 2 + ch0] = o[mt][1]; wr[hB * (2 + kHeadDim) + 2 + ch1] = o[mt][3]; }
  }
}

// Merge the kWarps per-warp results (m, l, o[d]) in shared memory, `stride` floats apart,
// into one partial (m, l, o[j]) in the workspace.
__device__ __forceinline__ void merge_warps(const float* src, size_t stride, float* dst, int j) {
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) M = fmaxf(M, src[i * stride]);
  float Lsum = 0.f, acc = 0.f;
  if (M != -INFINITY) {
#pragma unroll
    for (int i = 0; i < kWarps; ++i) {
      const float mi = src[i * stride];
      const float f = (mi == -INFINITY) ? 0.f : exp2f(mi - M);
      Lsum += src[i * stride + 1] * f;
      acc += src[i * stride + 2 + j] * f;
    }
  }
  dst[2 + j] = acc;
  if (j == 0) { dst[0] = M; dst[1] = Lsum; }
}

__global__ void __launch_bounds__(kThreads, 2) attn_decode_kernel(const AttnParams Pk, int ng_sel) {
  extern __shared__ __align__(128) uint8_t smem[];
  // shared-memory copy of the parameters (device functions take references to it)
  __shared__ AttnParams Ps;
  if (threadIdx.x == 0) Ps = Pk;
  __syncthreads();
  const AttnParams& P = Ps;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = P.gqa;
  // per-warp results: an INT2 warp writes into its own (drained) page ring, a window warp
  // into a plain array; both start after the 1 KB of barriers and query data.
  float* res = reinterpret_cast<float*>(smem + 1024);
  size_t wstride;
  if (split < P.n_int2) {
    wstride = (size_t)kStages * P.page_bytes / sizeof(float);
    if (ng_sel == 1) int2_split<1>(P, smem, b, h, split, res, wstride);
    else if (ng_sel == 2) int2_split<2>(P, smem, b, h, split, res, wstride);
    else int2_split<4>(P, smem, b, h, split, res, wstride);
  } else {
    wstride = (size_t)g * (2 + kHeadDim);
    window_split(P, b, h, split - P.n_int2, res, wstride);
  }
  __syncthreads();
  // ---- CTA partial: merge the warps, store to the workspace
  float* part = P.part + (((size_t)b * P.hkv + h) * P.n_split + split) * g * (2 + kHeadDim);
  for (int idx = threadIdx.x; idx < g * kHeadDim; idx += kThreads) {
    const int hh = idx / kHeadDim, j = idx % kHeadDim;
    merge_warps(res + hh * (2 + kHeadDim), wstride, part + hh * (2 + kHeadDim), j);
  }
  __threadfence();
  __syncthreads();
  __shared__ int last;
  if (threadIdx.x == 0) {
    const int t = atomicAdd(P.count + b * P.hkv + h, 1);
    last = (t == P.n_split - 1);
    if (last) P.count[b * P.hkv + h] = 0;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  // ---- final merge of the n_split partials of this (sequence, kv head), all loads
  // independent: (1) every (split, head) max and sum into shared memory, (2) one warp per
  // head turns them into rescale factors, (3) every thread sums its outputs over splits.
  const float* base = P.part + ((size_t)b * P.hkv + h) * P.n_split * g * (2 + kHeadDim);
  float* fs = reinterpret_cast<float*>(smem + 1024);             // [n_split][g] factors
  float* ls = fs + (size_t)P.n_split * g;                         // [n_split][g] sums
  float* Ls = ls + (size_t)P.n_split * g;                         // [g] totals
  const int ns = P.n_split;
  for (int idx = threadIdx.x; idx < ns * g; idx += kThreads) {
    const float* pp = base + (size_t)idx * (2 + kHeadDim);        // idx = split * g + head
    fs[idx] = __ldcg(pp);
    ls[idx] = __ldcg(pp + 1);
  }
  __syncthreads();
  {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (warp < g) {
      float M = -INFINITY;
      for (int s2 = lane; s2 < ns; s2 += 32) M = fmaxf(M, fs[s2 * g + warp]);
      for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
      float L = 0.f;
      for (int s2 = lane; s2 < ns; s2 += 32) {
        const float m = fs[s2 * g + warp];
        const float f = (M == -INFINITY || m == -INFINITY) ? 0.f : exp2f(m - M);
        fs[s2 * g + warp] = f;
        L += ls[s2 * g + warp] * f;
      }
      for (int o2 = 16; o2 > 0; o2 >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o2);
      if (lane == 0) Ls[warp] = L;
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < g * kHeadDim; idx += kThreads) {
    const int hh = idx / kHeadDim, j = idx % kHeadDim;
    const float* src = base + (size_t)hh * (2 + kHeadDim) + 2 + j;
    const size_t stride = (size_t)g * (2 + kHeadDim);
    float acc = 0.f;
    int s2 = 0;
    for (; s2 + 16 <= ns; s2 += 16) {
      float v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) v[u] = __ldcg(src + (size_t)(s2 + u) * stride);
#pragma unroll
      for (int u = 0; u < 16; ++u) acc += v[u] * fs[(s2 + u) * g + hh];
    }
    for (; s2 < ns; ++s2) acc += __ldcg(src + (size_t)s2 * stride) * fs[s2 * g + hh];
    const float L = Ls[hh];
    P.out[(((size_t)b * P.hkv + h) * g + hh) * kHeadDim + j] = (L > 0.f) ? acc / L : 0.f;
  }
}

}  // namespace kvq

using namespace kvq;

// Split counts from sizes only (no device query), so the workspace size is a pure
// function of (cfg, max_ctx).  Sized for 152 SMs with two resident CTAs each.
extern "C" void kvq_attn_splits(const kvq_config* cfg, int32_t max_ctx, int* n_int2, int* n_win) {
  const int units = cfg->batch * cfg->n_kv_heads;
  const int pages = max(0, (max_ctx - cfg->s_sink + kPage - 1) / kPage);
  int ni = cfg->attn_splits > 0 ? cfg->attn_splits : (304 + units - 1) / units;
  ni = max(1, min(ni, max(1, pages / 8)));
  const int pb = page_head_bytes(cfg->group_size, cfg->key_l2norm);
  const long long per_cta = (long long)((pages + ni - 1) / ni) * pb;        // INT2 bytes per CTA
  const int wtiles = (cfg->s_sink + kPage - 1) / kPage + cfg->ring_cap / kPage + 1;
  const long long tile_b = kPage * kHeadDim * 2 * 2;
  int nw = (int)((wtiles * tile_b + per_cta - 1) / max(per_cta, tile_b * kWarps));
  nw = max(1, min(nw, wtiles));
  *n_int2 = ni;
  *n_win = nw;
}

extern "C" size_t kvq_attn_ws_bytes(const kvq_config* cfg, int32_t max_ctx) {
  int ni, nw;
  kvq_attn_splits(cfg, max_ctx, &ni, &nw);
  const int g = cfg->n_q_heads / cfg->n_kv_heads;
  const size_t units = (size_t)cfg->batch * cfg->n_kv_heads;
  const size_t counters = (units * 4 + 255) / 256 * 256;
  return counters + units * (ni + nw) * g * (2 + kHeadDim) * sizeof(float);
}

extern "C" int kvq_launch_attn(const kvq_config* cfg, const kvq_cache* cache, const uint16_t* q_rot,
                               float* out, float sm_scale, int32_t max_ctx, void* ws, int32_t* d_status,
                               cudaStream_t stream) {
  AttnParams P{};
  P.pages = (const uint8_t*)cache->pages;
  P.page_table = cache->page_table;
  P.seq_len = cache->seq_len;
  P.s_quant = cache->s_quant;
  P.sink_k = cache->sink_k;
  P.sink_v = cache->sink_v;
  P.ring_k = cache->ring_k;
  P.ring_v = cache->ring_v;
  P.q = q_rot;
  P.out = out;
  P.status = d_status;
  P.batch = cfg->batch;
  P.hkv = cfg->n_kv_heads;
  P.gqa = cfg->n_q_heads / cfg->n_kv_heads;
  P.s_sink = cfg->s_sink;
  P.ring_cap = cfg->ring_cap;
  P.max_pages = cfg->max_pages_per_seq;
  P.num_pages = cfg->num_pages;
  P.group = cfg->group_size;
  P.l2 = cfg->key_l2norm;
  P.page_bytes = page_head_bytes(cfg->group_size, cfg->key_l2norm);
  kvq_attn_splits(cfg, max_ctx, &P.n_int2, &P.n_win);
  P.n_split = P.n_int2 + P.n_win;
  P.scale_log2 = sm_scale * 1.4426950408889634f;
  const size_t units = (size_t)cfg->batch * cfg->n_kv_heads;
  P.count = (int32_t*)ws;
  P.part = (float*)((char*)ws + (units * 4 + 255) / 256 * 256);
  const int ng = kHeadDim / cfg->group_size;
  const size_t ring_bytes = (size_t)kWarps * kStages * P.page_bytes;
  const size_t res_bytes = (size_t)kWarps * P.gqa * (2 + kHeadDim) * sizeof(float);
  const size_t merge_bytes = (size_t)(2 * P.n_split + 1) * P.gqa * sizeof(float);
  size_t body = ring_bytes > res_bytes ? ring_bytes : res_bytes;
  body = body > merge_bytes ? body : merge_bytes;
  const size_t smem = 1024 + body;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  static unsigned long long attr_done = 0ull;
  if (dev < 64 && !(attr_done & (1ull << dev))) {
    if (cudaFuncSetAttribute(attn_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) !=
        cudaSuccess)
      return KVQ_ERR_CUDA;
    attr_done |= 1ull << dev;
  }
  dim3 grid(P.n_split, cfg->n_kv_heads, cfg->batch);
  attn_decode_kernel<<<grid, kThreads, smem, stream>>>(P, ng);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

// ---- allocation-free variant ---------------------------------------------------------------
// The workspace of kv_attn_decode_noalloc lives in this fixed array: 8 MiB of device memory
// that every GPU which loads the library keeps until the process exits.  Host code must not
// use the symbol itself as a pointer (it names a host-side shadow); its device address is
// fetched once per device with cudaGetSymbolAddress while that device is current.
static __device__ __align__(256) uint8_t g_noalloc_workspace[KVQ_NOALLOC_WORKSPACE_BYTES];

extern "C" int kvq_launch_attn_noalloc(const kvq_config* cfg, const kvq_cache* cache, const uint16_t* q_rot,
                                       float* out, float sm_scale, int32_t max_ctx, int32_t* d_status,
                                       cudaStream_t stream) {
  const size_t need = kvq_attn_ws_bytes(cfg, max_ctx);
  if (need > (size_t)KVQ_NOALLOC_WORKSPACE_BYTES) return KVQ_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ERR_CUDA;
  static std::mutex mu;
  static void* addr[64] = {};
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || p == nullptr) return KVQ_ERR_CUDA;
      addr[dev] = p;
    }
    ws = addr[dev];
  }
  // the ticket counters at the head of the workspace must start at zero on every call
  const size_t units = (size_t)cfg->batch * cfg->n_kv_heads;
  if (cudaMemsetAsync(ws, 0, units * sizeof(int32_t), stream) != cudaSuccess) return KVQ_ERR_CUDA;
  return kvq_launch_attn(cfg, cache, q_rot, out, sm_scale, max_ctx, ws, d_status, stream);
}
