// kv_attn_decode: GQA decode attention over the mixed cache (BF16 sink | INT2 pages |
// BF16 recent ring), split over the token axis with an in-kernel online-softmax merge.
//
// Source: OSCAR summary, section 4 "Decoding Attention Kernel" (partition the cache into
// BF16 and INT2 segments, unpack INT2 and accumulate in floating point; existing kernels
// needed two launches plus a merge); OScaR reading note, "系统设计与 CUDA 实现"
// (INT2 tiles dequantized in registers: x Delta, - z, x s_t, inside split attention) and
// the algorithm's attention phase; WUSH-KV digest, GQA background (n_q/n_kv query heads read
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
#include <type_traits>

namespace kvq {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 4;
constexpr long long kWaitLimit = 1LL << 22;
constexpr int kRow = 4 + kHeadDim;      // one (m, l, -, -, o[d]) record; o 16-byte aligned
constexpr int kGroup = 8;               // splits merged together at the first merge level
// partials of one (sequence, kv head) up to this size are merged in one level from shared memory
// (two CTAs still fit on an SM); larger ones go through the two-level tree
constexpr size_t kMerge1Bytes = 96 * 1024;

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
  float* part;        // [B * Hkv][n_split][g][kRow]   per-CTA partials
  float* part2;       // [B * Hkv][n_groups][g][kRow]  merged groups of kGroup splits
  int32_t* count;     // [B * Hkv][n_groups + 1]       tickets of the merge tree
  int32_t* status;
  int batch, hkv, gqa, s_sink, ring_cap, max_pages, num_pages, group, l2, page_bytes;
  int n_int2, n_win, n_split;
  int mp;             // INT2 pages per sequence covered by the splits (host-known bound)
  int merge1;         // 1: the last CTA of a unit merges every split partial from shared memory
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
__device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity) {
  for (int i = 0; i < (int)kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity);
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
// Orders this thread's earlier (acquired) view of global memory before its later bulk copies.
__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// d = a * b (accumulator starts at zero)
__device__ __forceinline__ void mma_f16_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// 2^x (MUFU; about 2 ulp, -inf -> 0): the softmax weights need no more
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
// a * b - c in one rounding (fp16x2)
__device__ __forceinline__ uint32_t hfma2_neg_bits(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b),
                      __hneg2(*reinterpret_cast<__half2*>(&c)));
  return *reinterpret_cast<uint32_t*>(&r);
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
// Scale data of one token for all NG groups: NG (Delta16, z16) pairs in one vector load.
template <int NG>
__device__ __forceinline__ void load_scales(const uint8_t* p, uint32_t (&o)[NG]) {
  if constexpr (NG == 1) {
    o[0] = *reinterpret_cast<const uint32_t*>(p);
  } else if constexpr (NG == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    o[0] = v.x; o[1] = v.y;
  } else {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
}

template <int NG, bool L2>
__device__ void int2_split(const AttnParams& P, uint8_t* smem, int b, int h, int split, float* res,
                           size_t wstride) {
  // accumulators per group; with fewer than 4 groups the k-steps alternate between two
  // accumulators so that consecutive MMAs do not wait on each other
  constexpr int NS = NG == 1 ? 2 : 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = P.gqa;
  // The splits cover the host-known page range [0, mp) so that every warp fetches its first
  // page-table entries without waiting for the sequence length; pages beyond the sequence's
  // INT2 region are then skipped.
  const int p0 = (int)((long long)P.mp * split / P.n_int2);
  const int p1 = (int)((long long)P.mp * (split + 1) / P.n_int2);
  const int first = p0 + warp;
  const int nk_max = first < p1 ? (p1 - first + kWarps - 1) / kWarps : 0;
  const int32_t* ptab = P.page_table + (size_t)b * P.max_pages;
  // page-table entries of this warp's pages, 32 at a time: lane i of chunk c holds page 32c + i
  auto load_pids = [&](int c) -> int {
    const int k = 32 * c + lane;
    const int lp = first + k * kWarps;
    return (k < nk_max && lp < P.max_pages) ? ptab[lp] : -1;
  };
  // Before waiting for the producer kernels (programmatic dependent launch): the page table is
  // not written by them, so its entries are read now, and the first pages of this warp are
  // pulled into L2 (a prefetch only -- the copies that the results use start after the wait).
  int pid_a = load_pids(0), pid_b = load_pids(1);
  {
    const int pid0 = __shfl_sync(0xffffffffu, pid_a, lane & (kStages - 1));
    if (lane < kStages && lane < nk_max && pid0 >= 0 && pid0 < P.num_pages)
      prefetch_l2_bulk(P.pages + ((size_t)pid0 * P.hkv + h) * P.page_bytes, (uint32_t)P.page_bytes);
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);                      // [kWarps][kStages]
  int* slot_pid = reinterpret_cast<int*>(smem + kWarps * kStages * 8);     // [kWarps][kStages]
  QShared* qs = reinterpret_cast<QShared*>(smem + kWarps * kStages * 12);
  constexpr int pb = (2 * kCodeBytes + 2 * kPage * NG * 4 + (L2 ? kPage * 2 : 0) + 31) / 32 * 32;
  uint8_t* my_ring = smem + 1024 + (size_t)warp * kStages * pb;            // [kStages][page_bytes]
  uint64_t* my_bars = bars + warp * kStages;
  int* my_pid = slot_pid + warp * kStages;
  if (lane < kStages) mbar_init(my_bars + lane, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  // copy page k of this warp into its slot (lane 0 only); an entry that is not a page id
  // completes the slot without data and is reported when (if) the page is consumed
  auto issue = [&](int k, int pid) {
    const int slot = k % kStages;
    if (pid < 0 || pid >= P.num_pages) {
      my_pid[slot] = -1;
      mbar_arrive(my_bars + slot);
    } else {
      my_pid[slot] = pid;
      mbar_arrive_tx(my_bars + slot, (uint32_t)pb);
      tma_load_1d(my_ring + (size_t)slot * pb, P.pages + ((size_t)pid * P.hkv + h) * pb, (uint32_t)pb,
                  my_bars + slot);
    }
  };
  __syncwarp();
  pdl_wait();
  // the first kStages pages of the host-known range are copied at once, before the sequence's
  // own extent is known; copies past the extent are waited for and dropped
  const int n_first = min(kStages, nk_max);
#pragma unroll
  for (int k = 0; k < kStages; ++k) {
    const int pid = __shfl_sync(0xffffffffu, pid_a, k);
    if (lane == 0 && k < n_first) issue(k, pid);
  }
  const int Lraw = P.seq_len[b];
  const int sqraw = P.s_quant[b];

  // ---- this warp's pages inside the INT2 region
  const int L = Lraw;
  const int sq = min(sqraw, L);
  const int n_tok = max(0, sq - P.s_sink);
  const int np = (n_tok + kPage - 1) / kPage;
  if (split == 0 && threadIdx.x == 0 && np > P.mp) set_status(P.status, KVQ_ERR_BOUNDS);
  const int pend = min(p1, np);
  const int nk = first < pend ? (pend - first + kWarps - 1) / kWarps : 0;

  // ---- queries (their loads fly while the first pages are copied): B fragments scaled into
  // fp16 range, per-head multipliers and group sums
  const uint16_t* qb = P.q + ((size_t)b * P.hkv * g + (size_t)h * g) * kHeadDim;
  const int hrow = lane >> 2, quad = lane & 3;
  uint32_t qraw[8][2];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint16_t* src = qb + (size_t)hrow * kHeadDim + 16 * s + 2 * quad;
    qraw[s][0] = (hrow < g) ? *reinterpret_cast<const uint32_t*>(src) : 0u;
    qraw[s][1] = (hrow < g) ? *reinterpret_cast<const uint32_t*>(src + 8) : 0u;
  }
  uint32_t bq[8][2];
  {
    float qv[8][4];
    float amax = 0.f;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const float2 lo = unpack_bf162(qraw[s][0]), hi2 = unpack_bf162(qraw[s][1]);
      qv[s][0] = lo.x; qv[s][1] = lo.y; qv[s][2] = hi2.x; qv[s][3] = hi2.y;
#pragma unroll
      for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(qv[s][e]));
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
      const float f = ldexpf(1.0f, sigma - 2 * slot_pow(s));
      bq[s][0] = pack_half2(qv[s][0] * f, qv[s][1] * f);
      bq[s][1] = pack_half2(qv[s][2] * f, qv[s][3] * f);
    }
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
  __syncthreads();

  const int hA = 2 * quad, hB = 2 * quad + 1;
  // Loop constants in registers: the parameter block lives in shared memory and would be
  // re-read after every barrier operation.  Scores are
  //   s = x_t (mult_h sum_g Delta_g acc_g - sum_g Delta_g z_g qsum_g),
  // x_t = scale_log2 * norm_t with key norms, else scale_log2 folded into mult and qsum here.
  const float xs = P.scale_log2;
  const float fx = L2 ? 1.f : xs;
  const float multA = qs->mult[hA] * fx, multB = qs->mult[hB] * fx;
  float qsA[NG], qsB[NG];
#pragma unroll
  for (int gi = 0; gi < NG; ++gi) { qsA[gi] = qs->qsum[hA][gi] * fx; qsB[gi] = qs->qsum[hB][gi] * fx; }
  const int num_pages = P.num_pages;
  const uint8_t* const page_base = P.pages + (size_t)h * pb;
  const int page_stride = P.hkv * pb;
  auto refill = [&](int kk, int pid) {     // lane 0 only: page kk of this warp into its slot
    const int slot = kk & (kStages - 1);
    if ((unsigned)pid >= (unsigned)num_pages) {
      my_pid[slot] = -1;
      mbar_arrive(my_bars + slot);
    } else {
      my_pid[slot] = pid;
      mbar_arrive_tx(my_bars + slot, (uint32_t)pb);
      tma_load_1d(my_ring + slot * pb, page_base + (size_t)pid * page_stride, (uint32_t)pb, my_bars + slot);
    }
  };

  // Online softmax with a lazy reference maximum m: probabilities are p = exp2(s - m), with m
  // moved only when a score exceeds it by more than 8, so p <= 2^8.  The loop keeps
  // mb = m + 8 and works with p' = exp2(s - mb) = p 2^-8 <= 1 (the fp16 B operand of P V);
  // l accumulates p' as well and is scaled back at the end.  mb starts at a finite "minus
  // infinity" so that fully masked pages (scores -inf) give p' = 0 on the lazy path.
  float mb[2] = {-1e30f, -1e30f};
  float lsum[2] = {0.f, 0.f};
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[mt][c] = 0.f;
  // zero-point correction sum_t W_g z_g: row g (group) of one m16n8 accumulator, columns = heads
  float corr[4] = {0.f, 0.f, 0.f, 0.f};

  const int tA = lane >> 2, tB = tA + 8;
  const int off_kw = 16 * lane, off_vw = kCodeBytes + 16 * lane;
  const int off_skA = k_scale_off() + tA * NG * 4, off_skB = k_scale_off() + tB * NG * 4;
  const int off_dv0 = v_delta_off(NG, 2 * quad, 0), off_dv1 = v_delta_off(NG, 2 * quad + 8, 0);
  const int off_zp0 = v_zero_off(NG, 2 * quad, hrow < NG ? hrow : 0);
  const int off_zp1 = v_zero_off(NG, 2 * quad + 8, hrow < NG ? hrow : 0);
  const int off_gd0 = v_delta_off(NG, 2 * quad, hrow < NG ? hrow : 0);
  const int off_gd1 = v_delta_off(NG, 2 * quad + 8, hrow < NG ? hrow : 0);

  // One page: scores, softmax, P V.  MASKED pages (the sequence's last, partial page, or an
  // entry that is not a page id) keep only their first valid_tok tokens.
  auto page = [&](const uint8_t* pg, int valid_tok, auto masked) {
    constexpr bool MASKED = decltype(masked)::value;
    const uint4 wk = *reinterpret_cast<const uint4*>(pg + off_kw);
    uint32_t skA[NG], skB[NG];
    load_scales<NG>(pg + off_skA, skA);
    load_scales<NG>(pg + off_skB, skB);
    float xA = 1.f, xB = 1.f;
    if constexpr (L2) {
      const __half* nrm = reinterpret_cast<const __half*>(pg + norm_off(NG));
      xA = xs * __half2float(nrm[tA]);
      xB = xs * __half2float(nrm[tB]);
    }
    // ---- scores: codes x q' per group
    const uint32_t kw[4] = {wk.x, wk.y, wk.z, wk.w};
    const uint32_t kw10[4] = {wk.x >> 10, wk.y >> 10, wk.z >> 10, wk.w >> 10};
    float acc[NG][NS][4];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      uint32_t a[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = code_pair(kw[r], kw10[r], s);
      const int gi = (16 * s) / (kHeadDim / NG), u = s % NS;
      const int first_of = gi * (8 / NG) + u;            // first k-step feeding acc[gi][u]
      if (s == first_of) mma_f16_z(acc[gi][u], a, bq[s][0], bq[s][1]);
      else mma_f16(acc[gi][u], a, bq[s][0], bq[s][1]);
    }
    float sc[4];
    {
      float sA0 = 0.f, sA1 = 0.f, sB0 = 0.f, sB1 = 0.f, cA0 = 0.f, cA1 = 0.f, cB0 = 0.f, cB1 = 0.f;
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        float a0 = acc[gi][0][0], a1 = acc[gi][0][1], a2 = acc[gi][0][2], a3 = acc[gi][0][3];
        if constexpr (NS == 2) {
          a0 += acc[gi][1][0]; a1 += acc[gi][1][1]; a2 += acc[gi][1][2]; a3 += acc[gi][1][3];
        }
        const float2 dzA = unpack_half2(skA[gi]), dzB = unpack_half2(skB[gi]);
        const float pzA = dzA.x * dzA.y, pzB = dzB.x * dzB.y;      // exact: 11 x 11 bits
        sA0 = fmaf(dzA.x, a0, sA0); sA1 = fmaf(dzA.x, a1, sA1);
        sB0 = fmaf(dzB.x, a2, sB0); sB1 = fmaf(dzB.x, a3, sB1);
        cA0 = fmaf(pzA, qsA[gi], cA0); cA1 = fmaf(pzA, qsB[gi], cA1);
        cB0 = fmaf(pzB, qsA[gi], cB0); cB1 = fmaf(pzB, qsB[gi], cB1);
      }
      sc[0] = fmaf(sA0, multA, -cA0);
      sc[1] = fmaf(sA1, multB, -cA1);
      sc[2] = fmaf(sB0, multA, -cB0);
      sc[3] = fmaf(sB1, multB, -cB1);
      if constexpr (L2) {
        sc[0] *= xA; sc[1] *= xA; sc[2] *= xB; sc[3] *= xB;
      }
      if constexpr (MASKED) {
        if (tA >= valid_tok) sc[0] = sc[1] = -INFINITY;
        if (tB >= valid_tok) sc[2] = sc[3] = -INFINITY;
      }
    }
    float p[4];
    {
      const bool up = (fmaxf(sc[0], sc[2]) > mb[0]) || (fmaxf(sc[1], sc[3]) > mb[1]);
      if (__any_sync(0xffffffffu, up)) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float mx = fmaxf(sc[c], sc[c + 2]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          // the new reference: the running maximum (never below the old reference)
          const float nb = fmaxf(mb[c], mx + 8.f);
          const float alpha = ex2_approx(mb[c] - nb);
          mb[c] = nb;
          p[c] = ex2_approx(sc[c] - nb);
          p[c + 2] = ex2_approx(sc[c + 2] - nb);
          lsum[c] = fmaf(lsum[c], alpha, p[c] + p[c + 2]);
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) { o[mt][c] *= alpha; o[mt][c + 2] *= alpha; }
          corr[c] *= alpha;
        }
      } else {
        p[0] = ex2_approx(sc[0] - mb[0]);
        p[1] = ex2_approx(sc[1] - mb[1]);
        p[2] = ex2_approx(sc[2] - mb[0]);
        p[3] = ex2_approx(sc[3] - mb[1]);
        lsum[0] += p[0] + p[2];
        lsum[1] += p[1] + p[3];
      }
    }
    // ---- P V: per value group, W = P' * Delta_v as the B operand (fp16)
    // P' in the B-fragment layout (tokens 2q, 2q+1 | 2q+8, 2q+9 of head lane/4), then one
    // HMUL2 per group with the Delta_v pairs of the same tokens
    const uint32_t pb0 = movmatrix_trans(pack_half2(p[0], p[1]));
    const uint32_t pb1 = movmatrix_trans(pack_half2(p[2], p[3]));
    const uint4 wv = *reinterpret_cast<const uint4*>(pg + off_vw);
    uint32_t dv0[NG], dv1[NG];
    load_scales<NG>(pg + off_dv0, dv0);
    load_scales<NG>(pg + off_dv1, dv1);
    uint32_t zp0 = 0u, zp1 = 0u;                       // z_v pairs of group lane/4
    uint32_t gd0 = 0u, gd1 = 0u;                       // Delta_v pairs of group lane/4 (NG > 1)
    if (hrow < NG) {
      zp0 = *reinterpret_cast<const uint32_t*>(pg + off_zp0);
      zp1 = *reinterpret_cast<const uint32_t*>(pg + off_zp1);
      if constexpr (NG > 1) {
        gd0 = *reinterpret_cast<const uint32_t*>(pg + off_gd0);
        gd1 = *reinterpret_cast<const uint32_t*>(pg + off_gd1);
      }
    }
    if constexpr (MASKED) {                            // clear the dead tokens' scale data
      const uint32_t m0 = (2 * quad < valid_tok ? 0x0000ffffu : 0u) | (2 * quad + 1 < valid_tok ? 0xffff0000u : 0u);
      const uint32_t m1 = (2 * quad + 8 < valid_tok ? 0x0000ffffu : 0u) | (2 * quad + 9 < valid_tok ? 0xffff0000u : 0u);
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) { dv0[gi] &= m0; dv1[gi] &= m1; }
      zp0 &= m0;
      zp1 &= m1;
    }
    uint32_t bw[NG][2];
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      bw[gi][0] = hmul2_bits(pb0, dv0[gi]);
      bw[gi][1] = hmul2_bits(pb1, dv1[gi]);
    }
    if constexpr (NG == 1) {
      // row 0 of the correction: sum_t z_t W_t with the same W as the P V product
      const uint32_t az[4] = {hrow == 0 ? zp0 : 0u, 0u, hrow == 0 ? zp1 : 0u, 0u};
      mma_f16(corr, az, bw[0][0], bw[0][1]);
    } else {
      // all groups in one product: row g = sum_t (z Delta)_{t,g} P'_t, with z Delta carried as
      // an fp16 hi + lo pair (the product is 22 bits; the lo part is exact by the fused HFMA2)
      const uint32_t hi0 = hmul2_bits(zp0, gd0), hi1 = hmul2_bits(zp1, gd1);
      const uint32_t lo0 = hfma2_neg_bits(zp0, gd0, hi0), lo1 = hfma2_neg_bits(zp1, gd1, hi1);
      const uint32_t ah[4] = {hi0, 0u, hi1, 0u}, al[4] = {lo0, 0u, lo1, 0u};
      mma_f16(corr, ah, pb0, pb1);
      mma_f16(corr, al, pb0, pb1);
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
  };

  bool timed_out = false;
  int chunk_a = 0;               // page-table chunk held in pid_a
  int k = 0;
  for (; k < nk; ++k) {
    const int slot = k & (kStages - 1);
    if (!mbar_wait(my_bars + slot, ((unsigned)k / kStages) & 1u)) {
      timed_out = true;
      break;
    }
    const uint8_t* pg = my_ring + slot * pb;
    const int pid = my_pid[slot];
    const int lp = first + k * kWarps;
    if (pid >= 0 && kPage * (lp + 1) <= n_tok) {
      page(pg, kPage, std::false_type{});
    } else {
      if (pid < 0 && lane == 0) set_status(P.status, KVQ_ERR_BOUNDS);
      page(pg, pid < 0 ? 0 : min(kPage, n_tok - kPage * lp), std::true_type{});
    }
    // every lane has consumed this slot: refill it with the page kStages ahead, whose
    // page-table entry was fetched a chunk earlier
    const int kk = k + kStages;
    if ((kk >> 5) > chunk_a) {
      pid_a = pid_b;
      ++chunk_a;
      pid_b = load_pids(chunk_a + 1);
    }
    const int pid_next = __shfl_sync(0xffffffffu, pid_a, kk & 31);
    __syncwarp();
    if (lane == 0 && kk < nk) refill(kk, pid_next);
  }
  // l was accumulated in units of 2^-8 (see above); m is the reference without the bias
  Softmax sm;
  sm.m[0] = mb[0] - 8.f;
  sm.m[1] = mb[1] - 8.f;
  sm.l[0] = lsum[0] * 256.f;
  sm.l[1] = lsum[1] * 256.f;
  if (timed_out && lane == 0) set_status(P.status, KVQ_ERR_TIMEOUT);
  // copies not consumed (first copies past the extent; after a time-out, everything still in
  // flight) land before the slots are reused or the CTA exits (bounded)
  for (int kk = k; kk < max(min(nk, k + kStages), n_first); ++kk)
    (void)mbar_wait(my_bars + kk % kStages, (uint32_t)((kk / kStages) & 1));

  // ---- per-warp result: reduce l over the 8 lanes of a column pair; the zero-point
  // correction of group gi, heads (hA, hB) sits in lane 4 gi + quad
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int o2 = 4; o2 < 32; o2 <<= 1) sm.l[c] += __shfl_xor_sync(0xffffffffu, sm.l[c], o2);
  float zcA[NG], zcB[NG];
#pragma unroll
  for (int gi = 0; gi < NG; ++gi) {
    zcA[gi] = 256.f * __shfl_sync(0xffffffffu, corr[0], 4 * gi + quad);
    zcB[gi] = 256.f * __shfl_sync(0xffffffffu, corr[1], 4 * gi + quad);
  }
  float* wr = warp_result(res, warp, wstride);
  if (hA < g && tA == 0) { wr[hA * kRow] = sm.m[0]; wr[hA * kRow + 1] = sm.l[0]; }
  if (hB < g && tA == 0) { wr[hB * kRow] = sm.m[1]; wr[hB * kRow + 1] = sm.l[1]; }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    // codes carried 4^slot * 2^-24 and the weights 2^-8
    const float f = ldexpf(1.0f, 32 - 2 * slot_pow(mt));
    const int gi = (16 * mt) / (kHeadDim / NG);
    const int ch0 = 16 * mt + tA, ch1 = ch0 + 8;
    if (hA < g) {
      wr[hA * kRow + 4 + ch0] = o[mt][0] * f - zcA[gi];
      wr[hA * kRow + 4 + ch1] = o[mt][2] * f - zcA[gi];
    }
    if (hB < g) {
      wr[hB * kRow + 4 + ch0] = o[mt][1] * f - zcB[gi];
      wr[hB * kRow + 4 + ch1] = o[mt][3] * f - zcB[gi];
    }
  }
}

// ---- BF16 windows --------------------------------------------------------------------------
__device__ void window_split(const AttnParams& P, int b, int h, int wsplit, float* res, size_t wstride) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = P.gqa;
  pdl_wait();
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
  if (hA < g && tA == 0) { wr[hA * kRow] = sm.m[0]; wr[hA * kRow + 1] = sm.l[0]; }
  if (hB < g && tA == 0) { wr[hB * kRow] = sm.m[1]; wr[hB * kRow + 1] = sm.l[1]; }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int ch0 = 16 * hrow + 2 * mt, ch1 = ch0 + 1;
    if (hA < g) { wr[hA * kRow + 4 + ch0] = o[mt][0]; wr[hA * kRow + 4 + ch1] = o[mt][2]; }
    if (hB < g) { wr[hB * kRow + 4 + ch0] = o[mt][1]; wr[hB * kRow + 4 + ch1] = o[mt][3]; }
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
      acc += src[i * stride + 4 + j] * f;
    }
  }
  dst[4 + j] = acc;
  if (j == 0) { dst[0] = M; dst[1] = Lsum; }
}

// Merge n records (m, l, o[d]) per head from the workspace (other CTAs' writes: read past L1)
// with all loads of a chunk of 8 records in flight: warp w handles head w, lane the channels
// 4*lane .. 4*lane+3.  TO_OUT: dst[head][j] = o / l; otherwise dst holds merged records.
__device__ __noinline__ void merge_global(const float* src, int n, int g, float* dst, bool to_out) {
  const int lane = threadIdx.x & 31, hh = threadIdx.x >> 5;
  if (hh >= g) return;
  const size_t stride = (size_t)g * kRow;
  const float* s0 = src + (size_t)hh * kRow;
  float M = -INFINITY, L = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < n; c0 += 8) {
    float m[8], l[8];
    float4 o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (c0 + i < n) {
        const float* r = s0 + (size_t)(c0 + i) * stride;
        m[i] = __ldcg(r);
        l[i] = __ldcg(r + 1);
        o[i] = __ldcg(reinterpret_cast<const float4*>(r + 4) + lane);
      } else {
        m[i] = -INFINITY;
        l[i] = 0.f;
        o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float Mc = M;
#pragma unroll
    for (int i = 0; i < 8; ++i) Mc = fmaxf(Mc, m[i]);
    const float f0 = (M == -INFINITY) ? 0.f : exp2f(M - Mc);
    L *= f0;
    O.x *= f0; O.y *= f0; O.z *= f0; O.w *= f0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float f = (m[i] == -INFINITY) ? 0.f : exp2f(m[i] - Mc);
      L += l[i] * f;
      O.x += o[i].x * f; O.y += o[i].y * f; O.z += o[i].z * f; O.w += o[i].w * f;
    }
    M = Mc;
  }
  if (to_out) {
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    reinterpret_cast<float4*>(dst + (size_t)hh * kHeadDim)[lane] =
        make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
  } else {
    float* r = dst + (size_t)hh * kRow;
    if (lane == 0) { r[0] = M; r[1] = L; }
    reinterpret_cast<float4*>(r + 4)[lane] = O;
  }
}

// One kernel per (groups per row, key norms) variant, so that each launch's code is only its own
// page loop (a short loop per warp is sensitive to instruction-fetch misses).
template <int NG, bool L2>
__global__ void __launch_bounds__(kThreads, 2) attn_decode_kernel(const AttnParams Pk) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_trigger();
  // shared-memory copy of the parameters (device functions take references to it)
  __shared__ AttnParams Ps;
  if (threadIdx.x == 0) Ps = Pk;
  __syncthreads();
  const AttnParams& P = Ps;
  // (each branch below waits for the producer kernels itself, after its independent loads)
  // split index slowest: every unit's first INT2 split (always full) is dispatched before the
  // later, partly empty ones and the short window splits (longest work first)
  const int split = blockIdx.z, h = blockIdx.x, b = blockIdx.y;
  const int g = P.gqa;
  // per-warp results: an INT2 warp writes into its own (drained) page ring, a window warp
  // into a plain array; both start after the 1 KB of barriers and query data.
  float* res = reinterpret_cast<float*>(smem + 1024);
  size_t wstride;
  if (split < P.n_int2) {
    wstride = (size_t)kStages * P.page_bytes / sizeof(float);
    int2_split<NG, L2>(P, smem, b, h, split, res, wstride);
  } else {
    wstride = (size_t)g * kRow;
    window_split(P, b, h, split - P.n_int2, res, wstride);
  }
  __syncthreads();
  // ---- CTA partial: merge the warps, store to the workspace
  float* part = P.part + (((size_t)b * P.hkv + h) * P.n_split + split) * g * kRow;
  for (int idx = threadIdx.x; idx < g * kHeadDim; idx += kThreads) {
    const int hh = idx / kHeadDim, j = idx % kHeadDim;
    merge_warps(res + hh * kRow, wstride, part + hh * kRow, j);
  }
  __syncthreads();
  __shared__ int role;
  const int unit = b * P.hkv + h;
  if (P.merge1) {
    // ---- one-level merge: the last CTA of this (sequence, kv head) -- an atomic ticket, no
    // waiting -- pulls every split partial into shared memory with one bulk copy and merges.
    int32_t* cnt1 = P.count + (size_t)unit;
    if (threadIdx.x == 0) {
      const int t = atomic_add_acq_rel_gpu(cnt1, 1);   // releases this CTA's partial
      role = (t == P.n_split - 1);                      // ... and acquires the others'
      if (role) *cnt1 = 0;
    }
    __syncthreads();
    if (!role) return;
    __shared__ __align__(8) uint64_t mbar;
    float* buf = reinterpret_cast<float*>(smem + 1024);
    const uint32_t bytes = (uint32_t)((size_t)P.n_split * g * kRow * sizeof(float));
    if (threadIdx.x == 0) {
      fence_proxy_async_all();         // the acquired partials, seen by the bulk copy below
      mbar_init(&mbar, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      mbar_arrive_tx(&mbar, bytes);
      tma_load_1d(buf, P.part + (size_t)unit * P.n_split * g * kRow, bytes, &mbar);
    }
    __syncthreads();
    bool ok = mbar_wait(&mbar, 0u);
    if (!ok) {
      if (threadIdx.x == 0) set_status(P.status, KVQ_ERR_TIMEOUT);
      (void)mbar_wait(&mbar, 0u);      // the copy must land before the CTA can exit (bounded)
      return;
    }
    // warp hh merges head hh, lane the channels 4*lane .. 4*lane + 3
    const int lane = threadIdx.x & 31, hh = threadIdx.x >> 5;
    if (hh >= g) return;
    float M = -INFINITY;
    for (int i = lane; i < P.n_split; i += 32) M = fmaxf(M, buf[((size_t)i * g + hh) * kRow]);
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
    float Ls = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      for (int i = 0; i < P.n_split; ++i) {
        const float* r = buf + ((size_t)i * g + hh) * kRow;
        const float mi = r[0];
        const float f = (mi == -INFINITY) ? 0.f : exp2f(mi - M);
        const float4 oi = reinterpret_cast<const float4*>(r + 4)[lane];
        Ls += r[1] * f;
        O.x += oi.x * f; O.y += oi.y * f; O.z += oi.z * f; O.w += oi.w * f;
      }
    }
    const float inv = (Ls > 0.f) ? 1.f / Ls : 0.f;
    reinterpret_cast<float4*>(P.out + ((size_t)unit * g + hh) * kHeadDim)[lane] =
        make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
    return;
  }
  // ---- two-level merge tree over the splits of this (sequence, kv head): the last CTA of
  // every group of kGroup splits merges the group, the last group merger merges the groups.
  // Tickets are atomic counters (no waiting); every merge issues all its loads at once.
  const int n_grp = (P.n_split + kGroup - 1) / kGroup;
  const int grp = split / kGroup;
  const int gsize = min(kGroup, P.n_split - grp * kGroup);
  int32_t* cnt = P.count + (size_t)unit * (n_grp + 1);
  if (threadIdx.x == 0) {
    const int t = atomic_add_acq_rel_gpu(cnt + grp, 1);
    role = (t == gsize - 1);
    if (role) cnt[grp] = 0;
  }
  __syncthreads();
  if (!role) return;
  float* out_unit = P.out + (size_t)unit * g * kHeadDim;
  const float* gsrc = P.part + ((size_t)unit * P.n_split + (size_t)grp * kGroup) * g * kRow;
  if (n_grp == 1) {
    merge_global(gsrc, gsize, g, out_unit, true);
    return;
  }
  merge_global(gsrc, gsize, g, P.part2 + ((size_t)unit * n_grp + grp) * g * kRow, false);
  __syncthreads();
  if (threadIdx.x == 0) {
    const int t = atomic_add_acq_rel_gpu(cnt + n_grp, 1);
    role = (t == n_grp - 1);
    if (role) cnt[n_grp] = 0;
  }
  __syncthreads();
  if (!role) return;
  merge_global(P.part2 + (size_t)unit * n_grp * g * kRow, n_grp, g, out_unit, true);
}

}  // namespace kvq

using namespace kvq;

// Split counts from sizes only (no device query), so the workspace size is a pure
// function of (cfg, max_ctx): one wave of two CTAs per SM on 152 SMs, shared between INT2
// splits and BF16-window splits by bytes (the window after a flush: S_sink + S_keep +
// S_flush tokens).
// INT2 pages per sequence a call with contexts up to max_ctx can touch.
static int kvq_attn_pages(const kvq_config* cfg, int32_t max_ctx) {
  // 64-bit: max_ctx may be anything up to INT32_MAX
  const long long p = max(0LL, ((long long)max_ctx - cfg->s_sink + kPage - 1) / kPage);
  return (int)min(p, (long long)cfg->max_pages_per_seq);
}

extern "C" void kvq_attn_splits(const kvq_config* cfg, int32_t max_ctx, int* n_int2, int* n_win) {
  const long long units = (long long)cfg->batch * cfg->n_kv_heads;
  const int pages = kvq_attn_pages(cfg, max_ctx);
  const long long pb = page_head_bytes(cfg->group_size, cfg->key_l2norm);
  const long long tile_b = (long long)kPage * kHeadDim * 2 * 2;
  const long long wtiles = (cfg->s_sink + kPage - 1) / kPage + (cfg->s_keep + cfg->s_flush + kPage - 1) / kPage + 1;
  const double wbytes = (double)wtiles * tile_b, ibytes = (double)pages * pb;
  // p = CTAs per unit for one wave of two CTAs per SM.  When the windows are worth at least
  // half a CTA they get their share of the p; otherwise the INT2 splits take all p slots and
  // one short window split per unit comes on top (it fills a slot as the first CTAs retire).
  const int p = (int)max(1LL, 2LL * kSms / max(units, 1LL));
  int nw = (int)(p * wbytes / (wbytes + ibytes) + 0.5);
  int ni;
  if (p == 1 || nw == 0) {
    ni = p;
    nw = 1;
  } else {
    nw = (int)min((long long)min(nw, p - 1), wtiles);     // no more window splits than tiles
    ni = p - nw;
  }
  if (cfg->attn_splits > 0) ni = cfg->attn_splits;
  ni = max(1, min(ni, max(1, pages)));
  *n_int2 = ni;
  *n_win = nw;
}

// Workspace: tickets [units][n_groups + 1] (int32, padded to 256 B), per-CTA partials
// [units][n_split][g][kRow], merged groups [units][n_groups][g][kRow] (float32).
extern "C" size_t kvq_attn_counter_bytes(const kvq_config* cfg, int32_t max_ctx) {
  int ni, nw;
  kvq_attn_splits(cfg, max_ctx, &ni, &nw);
  const size_t units = (size_t)cfg->batch * cfg->n_kv_heads;
  const size_t n_grp = (size_t)(ni + nw + kGroup - 1) / kGroup;
  return (units * (n_grp + 1) * 4 + 255) / 256 * 256;
}

extern "C" size_t kvq_attn_ws_bytes(const kvq_config* cfg, int32_t max_ctx) {
  int ni, nw;
  kvq_attn_splits(cfg, max_ctx, &ni, &nw);
  const int g = cfg->n_q_heads / cfg->n_kv_heads;
  const size_t units = (size_t)cfg->batch * cfg->n_kv_heads;
  const size_t ns = (size_t)(ni + nw), n_grp = (ns + kGroup - 1) / kGroup;
  return kvq_attn_counter_bytes(cfg, max_ctx) + units * (ns + n_grp) * g * kRow * sizeof(float);
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
  P.mp = kvq_attn_pages(cfg, max_ctx);
  P.scale_log2 = sm_scale * 1.4426950408889634f;
  const size_t units = (size_t)cfg->batch * cfg->n_kv_heads;
  P.count = (int32_t*)ws;
  P.part = (float*)((char*)ws + kvq_attn_counter_bytes(cfg, max_ctx));
  P.part2 = P.part + units * (size_t)P.n_split * P.gqa * kRow;
  const int ng = kHeadDim / cfg->group_size;
  const size_t ring_bytes = (size_t)kWarps * kStages * P.page_bytes;
  const size_t res_bytes = (size_t)kWarps * P.gqa * kRow * sizeof(float);
  const size_t merge_bytes = (size_t)P.n_split * P.gqa * kRow * sizeof(float);
  P.merge1 = merge_bytes <= kMerge1Bytes;
  size_t smem = 1024 + (ring_bytes > res_bytes ? ring_bytes : res_bytes);
  if (P.merge1 && 1024 + merge_bytes > smem) smem = 1024 + merge_bytes;
  void (*kern)(const AttnParams) = nullptr;
  int vi = 0;
  if (cfg->key_l2norm) {
    kern = ng == 1 ? attn_decode_kernel<1, true> : ng == 2 ? attn_decode_kernel<2, true> : attn_decode_kernel<4, true>;
    vi = ng == 1 ? 3 : ng == 2 ? 4 : 5;
  } else {
    kern = ng == 1 ? attn_decode_kernel<1, false> : ng == 2 ? attn_decode_kernel<2, false> : attn_decode_kernel<4, false>;
    vi = ng == 1 ? 0 : ng == 2 ? 1 : 2;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ERR_CUDA;
  // the dynamic shared-memory limit is raised once per (device, kernel variant)
  static std::mutex mu;
  static unsigned long long attr_done[6] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!(attr_done[vi] & (1ull << dev))) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) != cudaSuccess)
        return KVQ_ERR_CUDA;
      attr_done[vi] |= 1ull << dev;
    }
  }
  if (cfg->batch > 65535 || P.n_split > 65535) return KVQ_ERR_UNSUPPORTED;   // grid y / z limits
  dim3 grid(cfg->n_kv_heads, cfg->batch, P.n_split);
  return launch_pdl(kern, grid, dim3(kThreads), smem, stream, P) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
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
      // set-up, once per device: the array's device address, and the ticket counters zeroed
      // once -- every completed call leaves the tickets it took at zero again, so later calls
      // need no clearing (and keep their overlap with the previous kernel on the stream)
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || p == nullptr) return KVQ_ERR_CUDA;
      if (cudaMemsetAsync(p, 0, (size_t)KVQ_NOALLOC_WORKSPACE_BYTES, stream) != cudaSuccess) return KVQ_ERR_CUDA;
      addr[dev] = p;
    }
    ws = addr[dev];
  }
  return kvq_launch_attn(cfg, cache, q_rot, out, sm_scale, max_ctx, ws, d_status, stream);
}
