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
//  * grid (kv_head, sequence, splits); splits [0, n_int2) stream INT2 pages, the rest
//    the BF16 windows.  Every warp owns a private ring of kStages page slots in shared
//    memory filled by 1-D TMA bulk copies (cp.async.bulk + mbarrier complete_tx); lane
//    0 issues, all lanes wait with a bounded try_wait loop.  No cluster, no multicast.
//  * one page (16 tokens) is one m16n8k16 tile: scores S[token][head] = codes x q',
//    all g <= 8 query heads of the kv head share the read (N = 8 columns).  A warp takes
//    its pages two at a time: both pages' scores, one softmax maximum test for both, both
//    P V products -- the loop, the waits and the maximum bookkeeping are shared and the two
//    pages' instructions interleave.
//  * 2-bit codes become fp16 tensor-core operands with one AND each: a code c at bit
//    position 2s of a 16-bit half is the fp16 subnormal c * 4^s * 2^-24, exact; the
//    4^s and 2^-24 factors are folded into q' (keys) or the output rows (values).  Scores
//    s = norm * mult_h * sum_g Delta_g (q'.c_g - z_g qsum_g): the group terms by FFMA from
//    the MMA accumulators, the zero-point term sum_g (Delta z)_g qsum_g by one more MMA
//    (Delta z and qsum as exact fp16 hi + lo pairs).
//  * P V: the fp32 probabilities times Delta_v become the B operand through
//    movmatrix (C-fragment -> B-fragment transpose); the zero point is a per-group
//    correction sum_t W_t z_t by MMA, whose row 8 (all ones) also sums P' -- the softmax
//    denominator from the same fp16 weights as the numerator.
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
constexpr int kCtasPerSm = 2;               // resident CTAs per SM the launch shape aims at
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
  void* out;          // [B][Hq][d] float32, or bf16 when out_bf16
  float* part;        // [B * Hkv][n_split][g][kRow]   per-CTA partials
  float* part2;       // [B * Hkv][n_groups][g][kRow]  merged groups of kGroup splits
  int32_t* count;     // [B * Hkv][n_groups + 1]       tickets of the merge tree
  int32_t* status;
  int batch, hkv, gqa, s_sink, ring_cap, max_pages, num_pages, group, l2, page_bytes;
  int n_int2, n_win, n_split;
  int mp;             // INT2 pages per sequence covered by the splits (host-known bound)
  int merge1;         // 1: the last CTA of a unit merges every split partial from shared memory
  int out_bf16;       // 1: the output is rounded once to bf16 (nearest-even)
  float scale_log2;   // sm_scale * log2(e)
  // chunk queries (kv_attn_chunk): grid row b is query row b; its cache sequence is the bc with
  // cu_rows[bc] <= b < cu_rows[bc + 1] (seqs sequences) and it sees tokens [0, p], p its
  // position seq_len[bc] - (cu_rows[bc + 1] - b).  nullptr: one decode query per sequence.
  const int32_t* cu_rows;
  int seqs;
};

// Cache sequence of grid row b (-1: a chunk row outside cu_rows).  cu_rows is a per-call input:
// chunk launches read it only after the dependency wait.
__device__ __forceinline__ int attn_seq(const AttnParams& P, int b) {
  if (!P.cu_rows) return b;
  if (b < __ldg(P.cu_rows) || b >= __ldg(P.cu_rows + P.seqs)) return -1;
  int lo = 0, hi = P.seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(P.cu_rows + mid) <= b) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Length and INT2 edge that grid row b sees (after the dependency wait): a decode query sees
// its sequence's seq_len tokens; a chunk query the tokens up to its own position.
__device__ __forceinline__ void unit_state(const AttnParams& P, int b, int bc, int& L, int& sq) {
  if (bc < 0) {
    L = 0;
    sq = P.s_sink;
    return;
  }
  L = P.seq_len[bc];
  sq = P.s_quant[bc];
  if (P.cu_rows) L = max(0, min(L, L - (__ldg(P.cu_rows + bc + 1) - b) + 1));
}

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

// explicit shared-memory loads (addresses in the shared window; the immediate offsets fold
// into the instruction)
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
template <int NG>
__device__ __forceinline__ void lds_scales(uint32_t a, uint32_t (&o)[NG]) {
  if constexpr (NG == 1) {
    o[0] = lds32(a);
  } else if constexpr (NG == 2) {
    const uint2 v = lds64(a);
    o[0] = v.x; o[1] = v.y;
  } else {
    const uint4 v = lds128(a);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
}

// (Delta z) of one token and group as the fp16 A operand of the key zero-point MMA: (hi, hi)
// for even quads (k = 4g, 4g + 1), (lo, 0) for odd ones (k = 4g + 2, 4g + 3), where
// hi = fp16(Delta16 z16) and lo = Delta16 z16 - hi exactly (fused).
__device__ __forceinline__ uint32_t dz_operand(uint32_t dz, bool odd) {
  const uint32_t zd = __byte_perm(dz, 0u, 0x1032);       // (z, Delta)
  const uint32_t hi = hmul2_bits(dz, zd);                  // (Delta z, z Delta), both rounded alike
  const uint32_t lo = hfma2_neg_bits(dz, zd, hi);          // exact remainders
  return odd ? (lo & 0xffffu) : hi;
}

template <int NG, bool L2, bool KC>
__device__ void int2_split(const AttnParams& P, uint8_t* smem, int b, int bc, int h, int split, float* res,
                           size_t wstride) {
  // accumulators per group; with one group the k-steps alternate between two accumulators so
  // that consecutive MMAs do not wait on each other
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
  const int32_t* ptab = P.page_table + (size_t)(bc < 0 ? 0 : bc) * P.max_pages;
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
  // page bytes: KC (per-channel keys) carries d key Delta16 + d key z16 and the exponent E
  constexpr int pb = (2 * kCodeBytes + (KC ? 4 * kHeadDim : kPage * NG * 4) + kPage * NG * 4 + (L2 ? kPage * 2 : 0) +
                      (KC ? 4 : 0) + 31) / 32 * 32;
  uint8_t* my_ring = smem + 1024 + (size_t)warp * kStages * pb;            // [kStages][page_bytes]
  uint64_t* my_bars = bars + warp * kStages;
  int* my_pid = slot_pid + warp * kStages;
  if (lane < kStages) mbar_init(my_bars + lane, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const uint8_t* const page_base = P.pages + (size_t)h * pb;
  const int page_stride = P.hkv * pb;
  const int num_pages = P.num_pages;
  // copy page k of this warp into its slot (lane 0 only); an entry that is not a page id
  // completes the slot without data and is reported when (if) the page is consumed
  auto refill = [&](int k, int pid) {
    const int slot = k & (kStages - 1);
    if ((unsigned)pid >= (unsigned)num_pages) {
      my_pid[slot] = -1;
      mbar_arrive(my_bars + slot);
    } else {
      my_pid[slot] = pid;
      mbar_arrive_tx(my_bars + slot, (uint32_t)pb);
      tma_load_1d(my_ring + slot * pb, page_base + (size_t)pid * page_stride, (uint32_t)pb, my_bars + slot);
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
    if (lane == 0 && k < n_first) refill(k, pid);
  }
  int Lraw, sqraw;
  unit_state(P, b, bc, Lraw, sqraw);

  // ---- this warp's pages inside the INT2 region
  const int L = Lraw;
  const int sq = min(sqraw, L);
  const int n_tok = max(0, sq - P.s_sink);
  const int np = (n_tok + kPage - 1) / kPage;
  if (split == 0 && threadIdx.x == 0 && np > P.mp) set_status(P.status, KVQ_ERR_BOUNDS);
  const int pend = min(p1, np);
  const int nk = first < pend ? (pend - first + kWarps - 1) / kWarps : 0;

  // ---- queries (their loads fly while the first pages are copied): B fragments scaled into
  // fp16 range (head lane/4: q' 2^(sigma - 2 slot), sigma per head), per-head multipliers, and
  // the B operand of the key zero-point MMA: group sums of q' 2^(sigma - 24) as fp16 hi + lo
  const uint16_t* qb = P.q + ((size_t)b * P.hkv * g + (size_t)h * g) * kHeadDim;
  const int hrow = lane >> 2, quad = lane & 3;
  const bool qodd = (quad & 1) != 0;
  uint32_t qraw[8][2];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint16_t* src = qb + (size_t)hrow * kHeadDim + 16 * s + 2 * quad;
    qraw[s][0] = (hrow < g) ? *reinterpret_cast<const uint32_t*>(src) : 0u;
    qraw[s][1] = (hrow < g) ? *reinterpret_cast<const uint32_t*>(src + 8) : 0u;
  }
  uint32_t bq[8][2];
  uint32_t bz0 = 0u, bz1 = 0u;            // B fragment of the zero-point MMA (k = 2 quad .., + 8 ..)
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
    // group sums in units 2^(sigma - 5) (|qsum| 2^(sigma - 5) < 2^14: hi and lo normal fp16); the
    // product lands in acc units after an exact scaling by 2^-19
    const float fz = ldexpf(1.0f, sigma - 5);
    float qsg[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      float acc = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s)
        if ((16 * s) / (kHeadDim / NG) == gi) acc += qv[s][0] + qv[s][1] + qv[s][2] + qv[s][3];
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      qsg[gi] = acc * fz;
    }
    // zero-point MMA, group q = quad (q < NG): k = 2q, 2q + 1 carry (hi, lo) of (Delta z) against
    // the group sum's hi part twice; k = 8 + 2q carries hi against the sum's lo part
    {
      const float v = quad == 0 ? qsg[0] : quad == 1 ? qsg[1] : quad == 2 ? qsg[2] : qsg[3];
      const __half hh = __float2half_rn(quad < NG ? v : 0.f);
      const __half hl = __float2half_rn(quad < NG ? v - __half2float(hh) : 0.f);
      __half2 r0 = __halves2half2(hh, hh), r1 = __halves2half2(hl, __float2half_rn(0.f));
      bz0 = *reinterpret_cast<uint32_t*>(&r0);
      bz1 = *reinterpret_cast<uint32_t*>(&r1);
    }
    if (warp == 0 && quad == 0) qs->mult[hrow] = ldexpf(1.0f, 24 - sigma);
  }
  __syncthreads();

  const int hA = 2 * quad, hB = 2 * quad + 1;
  // scores s = x_t mult_h (sum_g Delta_g acc_g - C), C the zero-point MMA in acc units;
  // x_t = scale_log2 * norm_t with key norms, else scale_log2 folded into mult here
  const float xs = P.scale_log2;
  const float multA = qs->mult[hA] * xs, multB = qs->mult[hB] * xs;

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
  // value zero-point correction sum_t W_g z_g: row g (group) of one m16n8 accumulator
  float corr[4] = {0.f, 0.f, 0.f, 0.f};

  const int tA = lane >> 2, tB = tA + 8;
  // per-lane offsets inside a page (all loads of a page are base + these)
  const uint32_t off_code = 16u * lane;
  const uint32_t off_sk = (uint32_t)(k_scale_off() + tA * NG * 4);
  const uint32_t off_dv = (uint32_t)v_delta_off(NG, 2 * quad, 0, KC);
  const uint32_t off_zg = (uint32_t)v_delta_off(NG, 2 * quad, hrow < NG ? hrow : 0, KC);
  const uint32_t off_nrm = (uint32_t)(norm_off(NG, KC) + 2 * tA);
  // per-channel keys: this quad's 16 Delta16 / z16 pairs (k-step s, half h at pair 2 s + h)
  const uint32_t off_kd = (uint32_t)(kc_delta_off() + 64 * quad);
  const uint32_t off_kz = (uint32_t)(kc_zero_off() + 64 * quad);
  const uint32_t off_ke = (uint32_t)kc_exp_off(NG, L2);
  const uint32_t ring_s = smem_u32(my_ring);

  // ---- one page, split in three parts so that two pages can share the softmax bookkeeping and
  // the loop overhead: scores (kside), lazy maximum (softmax), P V (vside)
  auto kside = [&](uint32_t sa, float (&sc)[4]) {
    const uint4 wk = lds128(sa + off_code);
    if constexpr (KC) {
      // ---- per-channel keys: s = sum_j q'_j Delta_j (c_j - z_j).  The page's Delta_j, scaled by
      // 2^-E (E the exponent of its largest Delta, so Delta 2^-E < 2), go into the B operand as
      // an exact fp16 pair B_hi + B_lo = q' 2^(sigma - 2p) Delta 2^-E (the product of two fp16
      // values has 22 bits; the fused HFMA2 gives the remainder exactly), so every MMA product
      // is exact as on the per-token path.  The zero-point term takes the same pair times 4^p
      // (exact) against A = z_j, every token row alike, in its own accumulator.
      const uint32_t kw[4] = {wk.x, wk.y, wk.z, wk.w};
      const uint32_t kw10[4] = {wk.x >> 10, wk.y >> 10, wk.z >> 10, wk.w >> 10};
      const int E = (int)lds32(sa + off_ke);
      const uint32_t se = E <= 14 ? (uint32_t)(15 - E) << 10 : 0x0200u;    // 2^-E, E in [-14, 15]
      const uint32_t s2 = se | (se << 16);
      float acc[2][4], accz[4];
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4) {
        const uint4 dq = lds128(sa + off_kd + 16 * s4), zq = lds128(sa + off_kz + 16 * s4);
        const uint32_t dd[4] = {dq.x, dq.y, dq.z, dq.w}, zz[4] = {zq.x, zq.y, zq.z, zq.w};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int s = 2 * s4 + j;
          const uint32_t d0 = hmul2_bits(dd[2 * j], s2), d1 = hmul2_bits(dd[2 * j + 1], s2);
          const uint32_t h0 = hmul2_bits(bq[s][0], d0), h1 = hmul2_bits(bq[s][1], d1);
          const uint32_t l0 = hfma2_neg_bits(bq[s][0], d0, h0), l1 = hfma2_neg_bits(bq[s][1], d1, h1);
          uint32_t a[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) a[r] = code_pair(kw[r], kw10[r], s);
          if (s < 2) mma_f16_z(acc[s & 1], a, h0, h1);
          else mma_f16(acc[s & 1], a, h0, h1);
          mma_f16(acc[s & 1], a, l0, l1);
          const uint32_t p4 = (uint32_t)(15 + 2 * slot_pow(s)) << 10;        // 4^p in fp16
          const uint32_t p4x2 = p4 | (p4 << 16);
          const uint32_t az[4] = {zz[2 * j], zz[2 * j], zz[2 * j + 1], zz[2 * j + 1]};
          if (s == 0) mma_f16_z(accz, az, hmul2_bits(h0, p4x2), hmul2_bits(h1, p4x2));
          else mma_f16(accz, az, hmul2_bits(h0, p4x2), hmul2_bits(h1, p4x2));
          mma_f16(accz, az, hmul2_bits(l0, p4x2), hmul2_bits(l1, p4x2));
        }
      }
      const float mE = __int_as_float((E + 127) << 23);                     // 2^E
      float sum[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sum[i] = __fmaf_rn(accz[i], -0x1p-24f, acc[0][i] + acc[1][i]);
      const float mA = multA * mE, mB = multB * mE;
      if constexpr (L2) {
        const float nA = __half2float(__ushort_as_half((unsigned short)lds16(sa + off_nrm)));
        const float nB = __half2float(__ushort_as_half((unsigned short)lds16(sa + off_nrm + 16)));
        sc[0] = sum[0] * (mA * nA);
        sc[1] = sum[1] * (mB * nA);
        sc[2] = sum[2] * (mA * nB);
        sc[3] = sum[3] * (mB * nB);
      } else {
        sc[0] = sum[0] * mA;
        sc[1] = sum[1] * mB;
        sc[2] = sum[2] * mA;
        sc[3] = sum[3] * mB;
      }
      return;
    }
    uint32_t skA[NG], skB[NG];
    lds_scales<NG>(sa + off_sk, skA);
    lds_scales<NG>(sa + off_sk + 32 * NG, skB);
    // ---- key zero points: C = sum_g (Delta z)_g qsum_g, one MMA; this lane carries group quad
    float cz[4];
    {
      uint32_t a[4] = {0u, 0u, 0u, 0u};
      if (quad < NG) {
        const uint32_t wA = lds32(sa + off_sk + 4 * quad), wB = lds32(sa + off_sk + 32 * NG + 4 * quad);
        const uint32_t zA = __byte_perm(wA, 0u, 0x1032), zB = __byte_perm(wB, 0u, 0x1032);   // (z, Delta)
        const uint32_t hA2 = hmul2_bits(wA, zA), hB2 = hmul2_bits(wB, zB);   // (Delta z, Delta z) rounded
        const uint32_t lA2 = hfma2_neg_bits(wA, zA, hA2), lB2 = hfma2_neg_bits(wB, zB, hB2);   // exact rests
        a[0] = __byte_perm(hA2, lA2, 0x5410);          // (hi, lo)
        a[1] = __byte_perm(hB2, lB2, 0x5410);
        a[2] = hA2 & 0xffffu;                          // (hi, 0)
        a[3] = hB2 & 0xffffu;
      }
      mma_f16_z(cz, a, bz0, bz1);
    }
    // ---- codes x q' per group, combined with Delta as they complete (the zero-point product
    // enters in acc units: an exact scaling by 2^-19)
    const uint32_t kw[4] = {wk.x, wk.y, wk.z, wk.w};
    const uint32_t kw10[4] = {wk.x >> 10, wk.y >> 10, wk.z >> 10, wk.w >> 10};
    float sum[4] = {cz[0] * -0x1p-19f, cz[1] * -0x1p-19f, cz[2] * -0x1p-19f, cz[3] * -0x1p-19f};
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      float acc[NS][4];
#pragma unroll
      for (int ss = 0; ss < 8 / NG; ++ss) {
        const int s = gi * (8 / NG) + ss, u = ss % NS;
        uint32_t a[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) a[r] = code_pair(kw[r], kw10[r], s);
        if (ss < NS) mma_f16_z(acc[u], a, bq[s][0], bq[s][1]);
        else mma_f16(acc[u], a, bq[s][0], bq[s][1]);
      }
      const float dA = __low2float(*reinterpret_cast<const __half2*>(&skA[gi]));
      const float dB = __low2float(*reinterpret_cast<const __half2*>(&skB[gi]));
#pragma unroll
      for (int u = 0; u < NS; ++u) {
        sum[0] = fmaf(dA, acc[u][0], sum[0]);
        sum[1] = fmaf(dA, acc[u][1], sum[1]);
        sum[2] = fmaf(dB, acc[u][2], sum[2]);
        sum[3] = fmaf(dB, acc[u][3], sum[3]);
      }
    }
    if constexpr (L2) {
      const float nA = __half2float(__ushort_as_half((unsigned short)lds16(sa + off_nrm)));
      const float nB = __half2float(__ushort_as_half((unsigned short)lds16(sa + off_nrm + 16)));
      sc[0] = sum[0] * (multA * nA);                   // multA, multB carry scale_log2 here
      sc[1] = sum[1] * (multB * nA);
      sc[2] = sum[2] * (multA * nB);
      sc[3] = sum[3] * (multB * nB);
    } else {
      sc[0] = sum[0] * multA;
      sc[1] = sum[1] * multB;
      sc[2] = sum[2] * multA;
      sc[3] = sum[3] * multB;
    }
  };
  // the reference moves (rarely): scale everything accumulated so far by alpha (heads hA, hB)
  auto rescale = [&](float aA, float aB) {
    const float2 al = make_float2(aA, aB);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      float2 v0 = __fmul2_rn(make_float2(o[mt][0], o[mt][1]), al);
      float2 v1 = __fmul2_rn(make_float2(o[mt][2], o[mt][3]), al);
      o[mt][0] = v0.x; o[mt][1] = v0.y; o[mt][2] = v1.x; o[mt][3] = v1.y;
    }
    const float2 c = __fmul2_rn(make_float2(corr[0], corr[1]), al);
    corr[0] = c.x; corr[1] = c.y;
    if constexpr (NG > 1) {
      const float2 c2 = __fmul2_rn(make_float2(corr[2], corr[3]), al);
      corr[2] = c2.x; corr[3] = c2.y;
    }
    lsum[0] *= aA;
    lsum[1] *= aB;
  };
  // lazy maximum over the scores of NP pages (sc[NP][4]); probabilities p' = exp2(s - mb)
  auto softmax_n = [&](auto& sc, auto& p, auto np_tag) {
    constexpr int NP = decltype(np_tag)::value;
    float mxA = fmaxf(sc[0][0], sc[0][2]), mxB = fmaxf(sc[0][1], sc[0][3]);
#pragma unroll
    for (int j = 1; j < NP; ++j) {
      mxA = fmaxf(mxA, fmaxf(sc[j][0], sc[j][2]));
      mxB = fmaxf(mxB, fmaxf(sc[j][1], sc[j][3]));
    }
    if (__any_sync(0xffffffffu, mxA > mb[0] || mxB > mb[1])) {
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) {
        mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, o2));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, o2));
      }
      // the new reference: the running maximum (never below the old reference)
      const float nA = fmaxf(mb[0], mxA + 8.f), nB = fmaxf(mb[1], mxB + 8.f);
      rescale(ex2_approx(mb[0] - nA), ex2_approx(mb[1] - nB));
      mb[0] = nA;
      mb[1] = nB;
    }
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      p[j][0] = ex2_approx(sc[j][0] - mb[0]);
      p[j][1] = ex2_approx(sc[j][1] - mb[1]);
      p[j][2] = ex2_approx(sc[j][2] - mb[0]);
      p[j][3] = ex2_approx(sc[j][3] - mb[1]);
      if constexpr (NG == 1) {           // (NG > 1: the value zero-point MMA sums P')
        lsum[0] += p[j][0] + p[j][2];
        lsum[1] += p[j][1] + p[j][3];
      }
    }
  };
  // P V of one page (MASKED: only its first valid_tok tokens)
  auto vside = [&](uint32_t sa, const float (&p)[4], int valid_tok, auto masked) {
    constexpr bool MASKED = decltype(masked)::value;
    const uint4 wv = lds128(sa + kCodeBytes + off_code);
    uint32_t dv0[NG], dv1[NG];
    lds_scales<NG>(sa + off_dv, dv0);
    lds_scales<NG>(sa + off_dv + 16 * NG, dv1);
    uint32_t zp0 = 0u, zp1 = 0u, gd0 = 0u, gd1 = 0u;   // z_v, Delta_v pairs of group lane/4
    (void)gd0;
    (void)gd1;
    if (hrow < NG) {
      zp0 = lds32(sa + off_zg + 32 * NG);
      zp1 = lds32(sa + off_zg + 48 * NG);
      if constexpr (NG > 1) {
        gd0 = lds32(sa + off_zg);
        gd1 = lds32(sa + off_zg + 16 * NG);
      }
    }
    // P' in the B-fragment layout (tokens 2q, 2q+1 | 2q+8, 2q+9 of head lane/4), then one
    // HMUL2 per group with the Delta_v pairs of the same tokens
    const uint32_t pb0 = movmatrix_trans(pack_half2(p[0], p[1]));
    const uint32_t pb1 = movmatrix_trans(pack_half2(p[2], p[3]));
    if constexpr (MASKED) {
      // clear the dead tokens' scale data: their bytes are whatever the page held before (the
      // pool need not be initialised), and 0 * Inf or NaN would poison the products
      const uint32_t m0 = (2 * quad < valid_tok ? 0x0000ffffu : 0u) | (2 * quad + 1 < valid_tok ? 0xffff0000u : 0u);
      const uint32_t m1 = (2 * quad + 8 < valid_tok ? 0x0000ffffu : 0u) | (2 * quad + 9 < valid_tok ? 0xffff0000u : 0u);
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) { dv0[gi] &= m0; dv1[gi] &= m1; }
      zp0 &= m0;
      zp1 &= m1;
      gd0 &= m0;
      gd1 &= m1;
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
      // row 8: ones -- C[8][h] = sum_t P'_t (the softmax denominator, from the same fp16 P')
      const uint32_t ones = lane < 4 ? 0x3C003C00u : 0u;
      const uint32_t ah[4] = {hi0, ones, hi1, ones}, al[4] = {lo0, 0u, lo1, 0u};
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
  // one page on its own (partial pages, bad entries, an odd last page)
  auto page1 = [&](uint32_t sa, int valid_tok, auto masked) {
    constexpr bool MASKED = decltype(masked)::value;
    float sc[1][4], p[1][4];
    kside(sa, sc[0]);
    if constexpr (MASKED) {
      if (tA >= valid_tok) sc[0][0] = sc[0][1] = -INFINITY;
      if (tB >= valid_tok) sc[0][2] = sc[0][3] = -INFINITY;
    }
    softmax_n(sc, p, std::integral_constant<int, 1>{});
    vside(sa, p[0], valid_tok, masked);
  };

  bool timed_out = false;
  int chunk_a = 0;               // page-table chunk held in pid_a
  int k = 0;
  // every lane has consumed slots: refill them with the pages kStages ahead, whose page-table
  // entries were fetched a chunk earlier
  auto refill_from = [&](int kk) {
    if ((kk >> 5) > chunk_a) {
      pid_a = pid_b;
      ++chunk_a;
      pid_b = load_pids(chunk_a + 1);
    }
    return __shfl_sync(0xffffffffu, pid_a, kk & 31);
  };
  // pages in pairs (two full pages share the loop, the waits and the softmax maximum)
  for (; k + 1 < nk; k += 2) {
    const int s0 = k & (kStages - 1), s1 = s0 + 1;          // k even: same phase for both
    const uint32_t ph = ((unsigned)k / kStages) & 1u;
    if (!mbar_wait(my_bars + s0, ph) || !mbar_wait(my_bars + s1, ph)) {
      timed_out = true;
      break;
    }
    const uint32_t sa0 = ring_s + (uint32_t)(s0 * pb), sa1 = sa0 + (uint32_t)pb;
    const int pid0 = my_pid[s0], pid1 = my_pid[s1];
    const int lp0 = first + k * kWarps, lp1 = lp0 + kWarps;
    if (pid0 >= 0 && pid1 >= 0 && kPage * (lp1 + 1) <= n_tok) {
      float sc[2][4], p[2][4];
      kside(sa0, sc[0]);
      kside(sa1, sc[1]);
      softmax_n(sc, p, std::integral_constant<int, 2>{});
      vside(sa0, p[0], kPage, std::false_type{});
      vside(sa1, p[1], kPage, std::false_type{});
    } else {
      if ((pid0 < 0 || pid1 < 0) && lane == 0) set_status(P.status, KVQ_ERR_BOUNDS);
      if (pid0 >= 0 && kPage * (lp0 + 1) <= n_tok) page1(sa0, kPage, std::false_type{});
      else page1(sa0, pid0 < 0 ? 0 : max(0, min(kPage, n_tok - kPage * lp0)), std::true_type{});
      page1(sa1, pid1 < 0 ? 0 : max(0, min(kPage, n_tok - kPage * lp1)), std::true_type{});
    }
    const int kk = k + kStages;
    const int pn0 = refill_from(kk);
    const int pn1 = __shfl_sync(0xffffffffu, pid_a, (kk + 1) & 31);
    __syncwarp();
    if (lane == 0) {
      if (kk < nk) refill(kk, pn0);
      if (kk + 1 < nk) refill(kk + 1, pn1);
    }
  }
  if (k < nk && !timed_out) {                                 // an odd last page
    const int slot = k & (kStages - 1);
    if (!mbar_wait(my_bars + slot, ((unsigned)k / kStages) & 1u)) {
      timed_out = true;
    } else {
      const uint32_t sa = ring_s + (uint32_t)(slot * pb);
      const int pid = my_pid[slot];
      const int lp = first + k * kWarps;
      if (pid >= 0 && kPage * (lp + 1) <= n_tok) {
        page1(sa, kPage, std::false_type{});
      } else {
        if (pid < 0 && lane == 0) set_status(P.status, KVQ_ERR_BOUNDS);
        page1(sa, pid < 0 ? 0 : min(kPage, n_tok - kPage * lp), std::true_type{});
      }
      ++k;                                                    // (no refill: nothing follows)
    }
  }
  // l was accumulated in units of 2^-8 (see above); m is the reference without the bias
  Softmax sm;
  sm.m[0] = mb[0] - 8.f;
  sm.m[1] = mb[1] - 8.f;
  if constexpr (NG > 1) {               // row 8 of the value zero-point MMA: lanes 0..3
    lsum[0] = __shfl_sync(0xffffffffu, corr[2], quad);
    lsum[1] = __shfl_sync(0xffffffffu, corr[3], quad);
  }
  sm.l[0] = lsum[0] * 256.f;
  sm.l[1] = lsum[1] * 256.f;
  if (timed_out && lane == 0) set_status(P.status, KVQ_ERR_TIMEOUT);
  // copies not consumed (first copies past the extent; after a time-out, everything still in
  // flight) land before the slots are reused or the CTA exits (bounded)
  for (int kk = k; kk < max(min(nk, k + kStages), n_first); ++kk)
    (void)mbar_wait(my_bars + kk % kStages, (uint32_t)((kk / kStages) & 1));

  // ---- per-warp result: reduce l over the 8 lanes of a column pair; the zero-point
  // correction of group gi, heads (hA, hB) sits in lane 4 gi + quad
  if constexpr (NG == 1) {
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) sm.l[c] += __shfl_xor_sync(0xffffffffu, sm.l[c], o2);
  }
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
__device__ void window_split(const AttnParams& P, int b, int bc, int h, int wsplit, float* res, size_t wstride) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = P.gqa;
  pdl_wait();
  int L, sqw;
  unit_state(P, b, bc, L, sqw);
  const int n_sink = min(P.s_sink, max(L, 0));
  const int r0 = max(min(sqw, L), P.s_sink);              // first recent token
  const int bcc = bc < 0 ? 0 : bc;                        // the cache rows (none read when L = 0)
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
      const size_t off = ((size_t)bcc * P.hkv + h) * P.s_sink * kHeadDim + (size_t)tok0 * kHeadDim;
      kbase = P.sink_k + off;
      vbase = P.sink_v + off;
      rows_avail = hi - tok0;                 // rows beyond the sink buffer are never read
    } else {
      tok0 = (rt0 + ti - n_sink_t) * kPage;
      lo = max(tok0, r0);
      hi = min(tok0 + kPage, L);
      const size_t off = (((size_t)bcc * P.hkv + h) * P.ring_cap + (tok0 % P.ring_cap)) * kHeadDim;
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

// Output row element j = 4 lane .. 4 lane + 3 of (unit row) `row`: float32, or bf16 rounded once.
__device__ __forceinline__ void store_out(void* out, bool bf16, size_t row, int lane, float4 v) {
  if (bf16) {
    uint2 b;
    b.x = pack_bf162(v.x, v.y);
    b.y = pack_bf162(v.z, v.w);
    reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(out) + row * kHeadDim)[lane] = b;
  } else {
    reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + row * kHeadDim)[lane] = v;
  }
}

// Merge n records (m, l, o[d]) per head from the workspace (other CTAs' writes: read past L1)
// with all loads of a chunk of 8 records in flight: warp w handles head w, lane the channels
// 4*lane .. 4*lane+3.  TO_OUT: dst[head][j] = o / l; otherwise dst holds merged records.
__device__ __noinline__ void merge_global(const float* src, int n, int g, void* dst, bool to_out, bool bf16) {
  const int lane = threadIdx.x & 31;
  for (int hh = threadIdx.x >> 5; hh < g; hh += kWarps) {
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
    store_out(dst, bf16, (size_t)hh, lane, make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
  } else {
    float* r = reinterpret_cast<float*>(dst) + (size_t)hh * kRow;
    if (lane == 0) { r[0] = M; r[1] = L; }
    reinterpret_cast<float4*>(r + 4)[lane] = O;
  }
  }
}

// One kernel per (groups per row, key norms, per-channel keys) variant, so that each launch's
// code is only its own page loop (a short loop per warp is sensitive to instruction-fetch misses).
template <int NG, bool L2, bool KC>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) attn_decode_kernel(const __grid_constant__ AttnParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_trigger();
  // (each branch below waits for the producer kernels itself, after its independent loads)
  // split index slowest: every unit's first INT2 split (always full) is dispatched before the
  // later, partly empty ones and the short window splits (longest work first)
  const int split = blockIdx.z, h = blockIdx.x, b = blockIdx.y;
  const int g = P.gqa;
  if (P.cu_rows) pdl_wait();          // (the rows' sequences: see attn_seq)
  const int bc = attn_seq(P, b);
  if (bc < 0 && threadIdx.x == 0 && split == 0 && h == 0) set_status(P.status, KVQ_ERR_BOUNDS);
  // per-warp results: an INT2 warp writes into its own (drained) page ring, a window warp
  // into a plain array; both start after the 1 KB of barriers and query data.
  float* res = reinterpret_cast<float*>(smem + 1024);
  size_t wstride;
  if (split < P.n_int2) {
    wstride = (size_t)kStages * P.page_bytes / sizeof(float);
    int2_split<NG, L2, KC>(P, smem, b, bc, h, split, res, wstride);
  } else {
    wstride = (size_t)g * kRow;
    window_split(P, b, bc, h, split - P.n_int2, res, wstride);
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
    const int lane = threadIdx.x & 31;
    for (int hh = threadIdx.x >> 5; hh < g; hh += kWarps) {
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
    store_out(P.out, P.out_bf16 != 0, (size_t)unit * g + hh, lane, make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
    }
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
  void* out_unit = P.out_bf16 ? (void*)(reinterpret_cast<uint16_t*>(P.out) + (size_t)unit * g * kHeadDim)
                              : (void*)(reinterpret_cast<float*>(P.out) + (size_t)unit * g * kHeadDim);
  const float* gsrc = P.part + ((size_t)unit * P.n_split + (size_t)grp * kGroup) * g * kRow;
  if (n_grp == 1) {
    merge_global(gsrc, gsize, g, out_unit, true, P.out_bf16 != 0);
    return;
  }
  merge_global(gsrc, gsize, g, P.part2 + ((size_t)unit * n_grp + grp) * g * kRow, false, false);
  __syncthreads();
  if (threadIdx.x == 0) {
    const int t = atomic_add_acq_rel_gpu(cnt + n_grp, 1);
    role = (t == n_grp - 1);
    if (role) cnt[n_grp] = 0;
  }
  __syncthreads();
  if (!role) return;
  merge_global(P.part2 + (size_t)unit * n_grp * g * kRow, n_grp, g, out_unit, true, P.out_bf16 != 0);
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
  const long long pb = page_head_bytes(cfg->group_size, cfg->key_l2norm, cfg->key_axis);
  const long long tile_b = (long long)kPage * kHeadDim * 2 * 2;
  const long long wtiles = (cfg->s_sink + kPage - 1) / kPage + (cfg->s_keep + cfg->s_flush + kPage - 1) / kPage + 1;
  const double wbytes = (double)wtiles * tile_b, ibytes = (double)pages * pb;
  // p = CTAs per unit for one wave of two CTAs per SM.  When the windows are worth at least
  // half a CTA they get their share of the p; otherwise the INT2 splits take all p slots and
  // one short window split per unit comes on top (it fills a slot as the first CTAs retire).
  const int p = (int)max(1LL, (long long)kCtasPerSm * kSms / max(units, 1LL));
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

// The decode launch; cfg->batch is the number of grid rows (sequences, or chunk query rows
// with cu_rows over seqs sequences).
static int launch_attn_impl(const kvq_config* cfg, const kvq_cache* cache, const uint16_t* q_rot, void* out,
                            int out_bf16, float sm_scale, int32_t max_ctx, void* ws, int32_t* d_status,
                            cudaStream_t stream, const int32_t* cu_rows, int seqs) {
  AttnParams P{};
  P.cu_rows = cu_rows;
  P.seqs = seqs;
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
  P.out_bf16 = out_bf16 ? 1 : 0;
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
  P.page_bytes = page_head_bytes(cfg->group_size, cfg->key_l2norm, cfg->key_axis);
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
  const int vi = (ng == 1 ? 0 : ng == 2 ? 1 : 2) + (cfg->key_l2norm ? 3 : 0) + (cfg->key_axis ? 6 : 0);
  if (cfg->key_axis == KVQ_KEY_PER_CHANNEL) {
    if (cfg->key_l2norm)
      kern = ng == 1 ? attn_decode_kernel<1, true, true> : ng == 2 ? attn_decode_kernel<2, true, true>
                                                                  : attn_decode_kernel<4, true, true>;
    else
      kern = ng == 1 ? attn_decode_kernel<1, false, true> : ng == 2 ? attn_decode_kernel<2, false, true>
                                                                   : attn_decode_kernel<4, false, true>;
  } else if (cfg->key_l2norm) {
    kern = ng == 1 ? attn_decode_kernel<1, true, false> : ng == 2 ? attn_decode_kernel<2, true, false>
                                                                 : attn_decode_kernel<4, true, false>;
  } else {
    kern = ng == 1 ? attn_decode_kernel<1, false, false> : ng == 2 ? attn_decode_kernel<2, false, false>
                                                                  : attn_decode_kernel<4, false, false>;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ERR_CUDA;
  // the dynamic shared-memory limit is raised once per (device, kernel variant)
  static std::mutex mu;
  static unsigned long long attr_done[12] = {};
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

extern "C" int kvq_launch_attn(const kvq_config* cfg, const kvq_cache* cache, const uint16_t* q_rot,
                               void* out, int out_bf16, float sm_scale, int32_t max_ctx, void* ws, int32_t* d_status,
                               cudaStream_t stream) {
  return launch_attn_impl(cfg, cache, q_rot, out, out_bf16, sm_scale, max_ctx, ws, d_status, stream, nullptr,
                          cfg->batch);
}

// Chunk queries: one grid row per query row (the sizes follow from a config whose batch is
// the number of rows).
extern "C" size_t kvq_attn_chunk_ws_bytes(const kvq_config* cfg, int32_t n_rows, int32_t max_ctx) {
  kvq_config c = *cfg;
  c.batch = n_rows;
  return kvq_attn_ws_bytes(&c, max_ctx);
}

extern "C" int kvq_launch_attn_chunk(const kvq_config* cfg, const kvq_cache* cache, const uint16_t* q_rot,
                                     const int32_t* cu_rows, int32_t n_rows, float* out, float sm_scale,
                                     int32_t max_ctx, void* ws, int32_t* d_status, cudaStream_t stream) {
  if (n_rows == 0) return KVQ_OK;
  kvq_config c = *cfg;
  c.batch = n_rows;
  return launch_attn_impl(&c, cache, q_rot, out, 0, sm_scale, max_ctx, ws, d_status, stream, cu_rows, cfg->batch);
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
  return kvq_launch_attn(cfg, cache, q_rot, out, 0, sm_scale, max_ctx, ws, d_status, stream);
}
