// kv_rotate_qk for prefill-sized calls: the dense per-head products on the 5th-generation
// tensor cores (tcgen05), every output still the exact product rounded once to bf16.
//
// Source: WUSH-KV digest, core method and inference algorithm (keys transformed by T_K on
// write, queries by T_K^{-T}); OSCAR summary, section 3 "Online Deployment" (fixed
// transforms applied while serving).  The pages fix what is computed; this file fixes how.
//
// Exactness without an accumulation model.  The tensor cores' fp32 accumulation order and
// rounding are not documented, so no output may depend on them.  Each operand is written as
// fixed-point digits on a grid common to the whole dot product:
//   * T row i (float32, 24-bit significands) in units U_i = 2^(e_i - 133), e_i the largest
//     exponent field of the row: |T_ij| / U_i < 128, kept to 2^-24 units as four balanced
//     base-256 digits t_0 + t_1/2^8 + t_2/2^16 + t_3/2^24, each an integer in [-128, 128];
//   * x row r (bf16, 8-bit significands) in units V_r = 2^(f_r - 133), likewise three digits
//     kept to 2^-16 units (exact unless an element lies 16 or more binades below the row's
//     largest).
// A digit is an integer of at most 8 significant bits, so it is an exact bf16, every product
// of two digits is an integer below 2^14, and every sum the tensor cores form over K = 128
// stays an integer below 2^23 -- exact in fp32 whatever the order or alignment of the
// additions (kvq_selftest_tc_integer_sums checks this on the device).  The nine digit
// products with a + b <= 3 go to four fp32 accumulators by level L = a + b:
//   y = U_i V_r sum_L 2^(-8 L) D_L + (dropped digits and truncation, bounded below),
// and the CUDA cores combine the four levels, bound the remainder, and decide the correctly
// rounded bf16 whenever no rounding midpoint lies within that bound; the rest (about 0.01%
// of outputs on the pages' workloads) are recomputed exactly in double-float.
//
// Layout (one CTA of 8 warps per SM, it holds all 512 TMEM columns):
//   TMEM columns   0..255  the four T digit matrices, A operand (lane = output i, K packed
//                          two bf16 per column), written once per tile;
//   TMEM columns 256..511  the four level accumulators D_L for a chunk of 64 rows
//                          (lane = output i, column = row);
//   shared memory          the three x digit matrices of a chunk (B operand, K-major,
//                          128-byte swizzle), double-buffered; per-row metadata.
// One thread issues the 72 MMAs of a chunk (M = 128, N = 64, K = 16 each) while the other
// warps slice the next chunk's rows; the accumulators are read into registers at once, so the
// next chunk's MMAs overlap this chunk's rounding decisions and stores.
#include "rotate.cuh"

#include <mutex>

namespace kvq {
namespace {

constexpr int kUmRows = 64;                          // rows of a chunk (N of every MMA)
constexpr int kXSlice = kUmRows * kHeadDim * 2;      // one x digit matrix: 16 KB
constexpr int kXBuf = 3 * kXSlice;                   // three digit matrices per chunk buffer
constexpr int kList = 256;                           // queued undecided outputs per warp

// per-row metadata of a chunk (three buffers: chunk n, n + 1 being sliced, n + 2)
struct UmRow {
  uint16_t* dst;         // destination row (nullptr: nothing to write)
  const uint16_t* src;   // the source row (for exact recomputation)
  float c;               // bound terms of the row, units of U_i V_r
  int fr;                // exponent field f_r of the row's units
  int flags;             // kRowZero | kRowBad | kRowLossy
  int pad;
};
static_assert(sizeof(UmRow) == 32, "UmRow layout");
constexpr int kRowZero = 1, kRowBad = 2, kRowLossy = 4;

constexpr int kMetaOff = 2 * kXBuf;
constexpr int kListOff = kMetaOff + 3 * kUmRows * (int)sizeof(UmRow);
constexpr int kExchOff = kListOff + 8 * kList * 2;
constexpr int kUmUsed = kExchOff + 3 * 1024;   // exponent exchange [2][128] int, sums [2][128] u64
// more than half of an SM's shared memory: never two CTAs on one SM (each holds all of TMEM)
constexpr int kUmSmem = 118 * 1024;
static_assert(kUmUsed + 1024 <= kUmSmem, "shared memory layout");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 256;
// instruction descriptor, kind::f16: D f32, A and B bf16, both K-major, N = 64, M = 128
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kUmRows >> 3) << 17) |
                            ((128u >> 4) << 24);
constexpr long long kSpinLimit = 1LL << 22;      // try_wait rounds before a wait gives up

// ---- tcgen05 / mbarrier primitives ---------------------------------------------------------
__device__ __forceinline__ uint32_t um_saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void um_mbar_init(uint64_t* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(um_saddr(bar)) : "memory");
}
__device__ __forceinline__ bool um_mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(um_saddr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded wait for phase `parity` of an mbarrier; false when the limit ran out
__device__ __noinline__ bool um_mbar_wait(uint64_t* bar, uint32_t parity) {
  for (long long it = 0; it < kSpinLimit; ++it)
    if (um_mbar_try(bar, parity)) return true;
  return false;
}

// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// D (TMEM) [+]= A (TMEM) x B (shared, descriptor)^T
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(um_saddr(bar))
               : "memory");
}

// 8 consecutive TMEM columns of this warp's 32 lanes <- registers
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
// 32 consecutive TMEM columns of this warp's 32 lanes -> registers (not yet waited for)
#define UM_O8(b)                                                                                            \
  "=r"(v[b]), "=r"(v[b + 1]), "=r"(v[b + 2]), "=r"(v[b + 3]), "=r"(v[b + 4]), "=r"(v[b + 5]), "=r"(v[b + 6]), \
      "=r"(v[b + 7])
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : UM_O8(0), UM_O8(8), UM_O8(16), UM_O8(24)
      : "r"(taddr));
}
#undef UM_O8
// wait for this thread's TMEM loads; the registers pass through so no use moves above it
#define UM_IO8(b)                                                                                           \
  "+r"(v[b]), "+r"(v[b + 1]), "+r"(v[b + 2]), "+r"(v[b + 3]), "+r"(v[b + 4]), "+r"(v[b + 5]), "+r"(v[b + 6]), \
      "+r"(v[b + 7])
__device__ __forceinline__ void tmem_wait_ld32(uint32_t* v) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : UM_IO8(0), UM_IO8(8), UM_IO8(16), UM_IO8(24)::"memory");
}
#undef UM_IO8

// ---- digits ---------------------------------------------------------------------------------
// bf16 bits of an integer d with |d| <= 128 (exact: at most 8 significant bits)
__device__ __forceinline__ uint32_t digit_bf16(int d) {
  const float f = __int_as_float(0x4B400000 + d) - 12582912.0f;    // float(d) for |d| < 2^22
  return __float_as_uint(f) >> 16;
}
// lowest balanced base-256 digit (in [-128, 127]) of M, and M advanced past it
__device__ __forceinline__ int take_digit(uint32_t& M) {
  const int d = (int)((M + 128u) & 255u) - 128;
  M = (M - (uint32_t)d) >> 8;
  return d;
}

// byte offset of x element (row n < 64, k < 128) in a digit matrix: two 8 KB K halves of
// 8-row groups (1024 B), rows 128 B apart, 16-byte chunks XOR-swizzled by row
__device__ __forceinline__ int xs_offset(int n, int k) {
  return (k >> 6) * 8192 + (n >> 3) * 1024 + (n & 7) * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) + (k & 7) * 2;
}


// The 72 MMAs of a chunk: x digit matrix a (shared memory, buffer at xbuf) against T digit
// matrix b (TMEM), into the accumulator of level a + b, K = 128 in eight steps of 16.
__device__ __forceinline__ void issue_chunk(uint32_t tb, uint32_t xbuf) {
  constexpr int kA[9] = {0, 0, 1, 0, 1, 2, 0, 1, 2};
  constexpr int kB[9] = {0, 1, 0, 2, 1, 0, 3, 2, 1};
  constexpr int kFirst[9] = {1, 1, 0, 1, 0, 0, 1, 0, 0};
#pragma unroll
  for (int c = 0; c < 9; ++c) {
    const uint32_t d = tb + kAccCol + 64u * (uint32_t)(kA[c] + kB[c]);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint64_t bd = sw128_desc(xbuf + (uint32_t)(kA[c] * kXSlice + (kk >> 2) * 8192 + (kk & 3) * 32));
      umma_ts(d, tb + 64u * (uint32_t)kB[c] + 8u * (uint32_t)kk, bd, (kFirst[c] && kk == 0) ? 0u : 1u);
    }
  }
}

// T row i, K half `half` (64 entries, global) -> the four digit matrices in TMEM columns
// 64 b + 32 half + ..., this warp's lanes.  e_i is the row's exponent field (both halves);
// returns sum_j M_j of this half (M_j = |T_ij| / U_i in units of 2^-24, truncated).
__device__ __forceinline__ unsigned long long slice_t_half(const float* trow, int e_i, uint32_t taddr) {
  unsigned long long msum = 0;
#pragma unroll 1
  for (int blk = 0; blk < 4; ++blk) {
    uint32_t out[4][8];
#pragma unroll
    for (int j4 = 0; j4 < 4; ++j4) {
      const float4 t4 = reinterpret_cast<const float4*>(trow)[4 * blk + j4];
      const float tv[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
      for (int m2 = 0; m2 < 4; ++m2) {
        const uint32_t u = __float_as_uint(tv[m2]);
        const int E = (int)((u >> 23) & 0xffu);
        const uint32_t m = E ? ((u & 0x7fffffu) | 0x800000u) : (u & 0x7fffffu);
        const int sh = e_i - max(E, 1);
        uint32_t M = sh < 31 ? (m << 7) >> sh : 0u;
        msum += M;
        int d[4];
        d[3] = take_digit(M);
        d[2] = take_digit(M);
        d[1] = take_digit(M);
        d[0] = (int)M;
        const bool neg = (u >> 31) != 0u;
        const int col = 2 * j4 + (m2 >> 1), hi = m2 & 1;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const uint32_t bits = digit_bf16(neg ? -d[b] : d[b]);
          out[b][col] = hi ? (out[b][col] | (bits << 16)) : bits;
        }
      }
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) tmem_st8(taddr + 64u * (uint32_t)b + 8u * (uint32_t)blk, out[b]);
  }
  return msum;
}

// One warp's 8 rows of a chunk, loaded ahead of slicing.
struct XPre {
  uint2 x[8];             // this lane's 4 bf16 (k = 4 lane .. 4 lane + 3) of rows 8 w + j
  int row, head, b, p;    // lanes 0..7: indices of row 8 w + lane (b, p for cache rows)
  int valid;              // lanes 0..7: the row exists
};

__device__ __forceinline__ void x_prefetch(const RotParams& P, const RotTensor& T, int mh, int chunk, int pairs,
                                           int warp, int lane, XPre& pre) {
  const int p0 = chunk * kUmRows, np = min(kUmRows, pairs - p0);
  const int r = 8 * warp + (lane & 7);
  pre.valid = (lane < 8 && r < np) ? 1 : 0;
  int row = 0, head = 0;
  if (r < np) tile_row(T, mh, p0 + r, row, head);
  pre.row = row;
  pre.head = head;
  pre.b = pre.p = 0;
  if (pre.valid && !T.is_query) {
    pre.b = __ldg(P.seq_idx + row);
    pre.p = __ldg(P.pos + row);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int rj = __shfl_sync(0xffffffffu, row, j), hj = __shfl_sync(0xffffffffu, head, j);
    pre.x[j] = make_uint2(0u, 0u);
    if (8 * warp + j < np)
      pre.x[j] = __ldg(reinterpret_cast<const uint2*>(T.src + ((size_t)rj * T.heads + hj) * kHeadDim) + lane);
  }
}

// Digits of the prefetched rows -> x digit matrices (buffer xb) and row metadata.  Runs after
// the dependency wait (destinations read s_quant).
__device__ __forceinline__ void x_slice(const RotParams& P, const RotTensor& T, const XPre& pre, uint8_t* xb,
                                        UmRow* meta, int warp, int lane) {
  uint16_t* dst = nullptr;
  const uint16_t* src = nullptr;
  if (pre.valid) {
    src = T.src + ((size_t)pre.row * T.heads + pre.head) * kHeadDim;
    dst = rot_dst(P, T, pre.row, pre.head, pre.b, pre.p, true);
  }
#pragma unroll 2
  for (int j = 0; j < 8; ++j) {
    const int r = 8 * warp + j;
    const uint32_t h[4] = {pre.x[j].x & 0xffffu, pre.x[j].x >> 16, pre.x[j].y & 0xffffu, pre.x[j].y >> 16};
    int ef = 1;
    bool bad_l = false, nz_l = false;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int E = (int)((h[k] >> 7) & 0xffu);
      ef = max(ef, max(E, 1));
      bad_l |= E == 255;
      nz_l |= (h[k] & 0x7fffu) != 0u;
    }
    const int fr = __reduce_max_sync(0xffffffffu, ef);
    const bool bad = __any_sync(0xffffffffu, bad_l), nz = __any_sync(0xffffffffu, nz_l);
    uint32_t lo[3] = {0u, 0u, 0u}, hi[3] = {0u, 0u, 0u};
    uint32_t nsum = 0;
    bool lost_l = false;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int E = (int)((h[k] >> 7) & 0xffu);
      const uint32_t m = E ? ((h[k] & 0x7fu) | 0x80u) : (h[k] & 0x7fu);
      const int sh = fr - max(E, 1);
      const uint32_t full = m << 15;
      uint32_t N = sh < 32 ? full >> sh : 0u;
      const bool lost = sh < 32 ? ((N << sh) != full) : (full != 0u);
      lost_l |= lost;
      nsum += N + (lost ? 1u : 0u);
      int d[3];
      d[2] = take_digit(N);
      d[1] = take_digit(N);
      d[0] = (int)N;
      const bool neg = (h[k] >> 15) != 0u;
#pragma unroll
      for (int a = 0; a < 3; ++a) {
        const uint32_t bits = digit_bf16(neg ? -d[a] : d[a]);
        if (k < 2) lo[a] |= bits << (16 * k);
        else hi[a] |= bits << (16 * (k - 2));
      }
    }
    const bool lossy = __any_sync(0xffffffffu, lost_l);
    const uint32_t sx = __reduce_add_sync(0xffffffffu, nsum);
    const int off = xs_offset(r, 4 * lane);
#pragma unroll
    for (int a = 0; a < 3; ++a) *reinterpret_cast<uint2*>(xb + a * kXSlice + off) = make_uint2(lo[a], hi[a]);
    uint16_t* dj = (uint16_t*)__shfl_sync(0xffffffffu, (unsigned long long)dst, j);
    const uint16_t* sj = (const uint16_t*)__shfl_sync(0xffffffffu, (unsigned long long)src, j);
    if (lane == 0) {
      UmRow m;
      m.dst = dj;
      m.src = sj;
      // dropped digit products and the fp32 combination (2^-10, 2^-17) and T's truncation,
      // 2^-24 per unit of sum |x| (sx / 2^16 bounds sum |x| in units)
      m.c = 0x1.01p-10f + 0x1p-17f + (float)sx * 0x1.01p-40f;
      m.fr = fr;
      m.flags = (nz ? 0 : kRowZero) | (bad ? kRowBad : 0) | (lossy ? kRowLossy : 0);
      m.pad = 0;
      meta[r] = m;
    }
  }
}

// The queued undecided outputs of a warp ((row << 7) | output), recomputed exactly; returns 0.
__device__ __noinline__ int exact_list(const uint16_t* list, int count, const UmRow* mrow, const float* tmat,
                                       int lane) {
  __syncwarp();
  for (int f = 0; f < count; ++f) {
    const int r = list[f] >> 7, o = list[f] & 127;
    exact_output_warp(tmat + (size_t)o * kHeadDim, mrow[r].src, mrow[r].dst, o, lane);
  }
  __syncwarp();
  return 0;
}

// One CTA per tile: P.rpc chunks of 64 (row, head) pairs that share one matrix.
__global__ void __launch_bounds__(256, 1) rotate_tc_kernel(const RotParams Pk) {
  pdl_trigger();
  __shared__ RotParams Ps;
  __shared__ uint32_t tbase_sh;
  __shared__ __align__(8) uint64_t mbar[2];
  __shared__ int tile_bad, abort_sh;
  extern __shared__ uint8_t um_smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(um_smem_raw) + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q = warp & 3, half = warp >> 2, i = 32 * q + lane;
  if (tid == 0) {
    Ps = Pk;
    tile_bad = 0;
    abort_sh = 0;
    um_mbar_init(&mbar[0]);
    um_mbar_init(&mbar[1]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(um_saddr(&tbase_sh)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const RotParams& P = Ps;
  const uint32_t tb = tbase_sh;
  const uint32_t tlane = (uint32_t)(32 * q) << 16;     // this warp's TMEM lane quadrant
  int tt, tile;
  find_item(P.n_dense, blockIdx.x, tt, tile);
  const RotTensor& T = P.t[tt];
  const int pairs = T.rows * T.head_div;
  const int cpm = (pairs + kUmRows - 1) / kUmRows;
  const int tiles_per_mat = (cpm + P.rpc - 1) / P.rpc;
  const int mh = tile / tiles_per_mat;
  const int c0 = (tile % tiles_per_mat) * P.rpc, nch = min(cpm, c0 + P.rpc) - c0;
  const float* tmat = T.mat + (size_t)mh * kHeadDim * kHeadDim;
  UmRow* meta = reinterpret_cast<UmRow*>(sm + kMetaOff);
  uint16_t* list = reinterpret_cast<uint16_t*>(sm + kListOff) + warp * kList;
  int* ex_e = reinterpret_cast<int*>(sm + kExchOff);                        // [2][128]
  unsigned long long* ex_m = reinterpret_cast<unsigned long long*>(sm + kExchOff + 1024);   // [2][128]

  // ---- the matrix (a caller input: before the dependency wait) ----
  XPre pre;
  x_prefetch(P, T, mh, c0, pairs, warp, lane, pre);
  const float* trow = tmat + (size_t)i * kHeadDim + 64 * half;
  int e_i, tnz;
  {
    int e = 1, nz = 0, bad = 0;
#pragma unroll 4
    for (int j4 = 0; j4 < 16; ++j4) {
      const float4 t4 = reinterpret_cast<const float4*>(trow)[j4];
      const uint32_t u[4] = {__float_as_uint(t4.x), __float_as_uint(t4.y), __float_as_uint(t4.z), __float_as_uint(t4.w)};
#pragma unroll
      for (int m2 = 0; m2 < 4; ++m2) {
        const int E = (int)((u[m2] >> 23) & 0xffu);
        e = max(e, max(E, 1));
        bad |= E == 255;
        nz |= (u[m2] & 0x7fffffffu) != 0u;
      }
    }
    ex_e[half * 128 + i] = e | (nz << 16);
    if (bad) tile_bad = 1;
    __syncthreads();
    const int a0 = ex_e[i], a1 = ex_e[128 + i];
    e_i = max(a0 & 0xffff, a1 & 0xffff);
    tnz = (a0 | a1) >> 16;
  }
  ex_m[half * 128 + i] = slice_t_half(trow, e_i, tb + tlane + 32u * (uint32_t)half);
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  __syncthreads();
  // 2^-16 sum_j |T_ij| / U_i (rounded up): X's truncation bound for lossy rows
  const float st16 = (float)(ex_m[i] + ex_m[128 + i] + 128ull) * 0x1.01p-40f;
  const bool force = tile_bad != 0;

  pdl_wait();
  // ---- pipeline: slice chunk n + 2 while the tensor cores run chunk n + 1 ----
  auto xbuf = [&](int n) { return sm + (n & 1) * kXBuf; };
  x_slice(P, T, pre, xbuf(0), meta, warp, lane);
  if (nch > 1) x_prefetch(P, T, mh, c0 + 1, pairs, warp, lane, pre);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    tc_fence_after();
    issue_chunk(tb, um_saddr(xbuf(0)));
    umma_commit(&mbar[0]);
  }
  if (nch > 1) {
    x_slice(P, T, pre, xbuf(1), meta + kUmRows, warp, lane);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (nch > 2) x_prefetch(P, T, mh, c0 + 2, pairs, warp, lane, pre);
  }
  int count = 0, stuck = -1;
  for (int n = 0; n < nch; ++n) {
    const int timed_out = um_mbar_wait(&mbar[n & 1], (uint32_t)((n >> 1) & 1)) ? 0 : 1;
    stuck = n;
    tc_fence_after();
    uint32_t acc[4][32];
#pragma unroll
    for (int L = 0; L < 4; ++L) tmem_ld32(tb + tlane + kAccCol + 64u * (uint32_t)L + 32u * (uint32_t)half, acc[L]);
#pragma unroll
    for (int L = 0; L < 4; ++L) tmem_wait_ld32(acc[L]);
    tc_fence_before();
    // accumulators free; chunk n + 1's digits written; every thread takes the same exit
    if (__syncthreads_or(timed_out)) {
      abort_sh = 1;
      break;
    }
    if (tid == 0 && n + 1 < nch) {
      tc_fence_after();
      issue_chunk(tb, um_saddr(xbuf(n + 1)));
      umma_commit(&mbar[(n + 1) & 1]);
    }
    // ---- rounding decisions of chunk n: this thread's output i, rows 32 half + c ----
    const UmRow* mrow = meta + (n % 3) * kUmRows;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const int r = 32 * half + c;
      uint16_t* dst = mrow[r].dst;
      const float cr = mrow[r].c;
      const int fr = mrow[r].fr, flags = mrow[r].flags;
      const float L0 = __uint_as_float(acc[0][c]), L1 = __uint_as_float(acc[1][c]);
      const float L2 = __uint_as_float(acc[2][c]), L3 = __uint_as_float(acc[3][c]);
      const float v = fmaf(L3, 0x1p-24f, fmaf(L2, 0x1p-16f, fmaf(L1, 0x1p-8f, L0)));
      // |y / (U_i V_r) - v| <= 3u|v| + the row's terms (+ X's truncation for lossy rows)
      const float bnd = fmaf(fabsf(v), 0x1.81p-23f, (flags & kRowLossy) ? cr + st16 : cr);
      int b = bf16_if_decided(v, bnd);
      if (b >= 0) {
        const int Eu = (b >> 7) & 0xff, S = e_i + fr - 266, Ey = Eu + S;
        b = (Eu != 0 && Ey >= 1 && Ey <= 254) ? b + (S << 7) : -1;
      }
      if ((flags & kRowZero) || !tnz) b = 0;             // an exact zero is +0
      if (force || (flags & kRowBad)) b = -1;
      if (dst != nullptr && b >= 0) dst[i] = (uint16_t)b;
      const bool und = dst != nullptr && b < 0;
      const unsigned mk = __ballot_sync(0xffffffffu, und);
      if (und) list[count + __popc(mk & ((1u << lane) - 1u))] = (uint16_t)((r << 7) | i);
      count += __popc(mk);
      if (count > kList - 32) count = exact_list(list, count, mrow, tmat, lane);
    }
    count = exact_list(list, count, mrow, tmat, lane);
    // ---- digits of chunk n + 2 into chunk n's buffer (its MMAs have completed) ----
    if (n + 2 < nch) {
      x_slice(P, T, pre, xbuf(n), meta + ((n + 2) % 3) * kUmRows, warp, lane);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      if (n + 3 < nch) x_prefetch(P, T, mh, c0 + n + 3, pairs, warp, lane, pre);
    }
  }
  if (abort_sh) {
    // chunk `stuck` is the only one committed and not seen complete: give it one more bounded
    // wait before TMEM is released
    if (tid == 0) {
      set_status(P.status, KVQ_ERR_TIMEOUT);
      (void)um_mbar_wait(&mbar[stuck & 1], (uint32_t)((stuck >> 1) & 1));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tb), "r"(kTmemCols) : "memory");
}

// ---- device check: the tensor cores' integer sums are exact ----------------------------------
// Digit matrices (integers in [-128, 128]) for T and x, hashed or extreme (all +128, all -128,
// alternating), run through issue_chunk exactly as in the rotation; every level accumulator
// must equal the integer sum formed on the CUDA cores.
__device__ __forceinline__ int st_digit(uint32_t seed, int mode, int kind, int idx) {
  if (mode == 1) return 128;
  if (mode == 2) return -128;
  if (mode == 3) return ((idx ^ kind) & 1) ? -128 : 128;
  uint32_t h = seed * 0x9E3779B9u ^ (uint32_t)kind * 0x85EBCA6Bu ^ (uint32_t)idx * 0xC2B2AE35u;
  h ^= h >> 16;
  h *= 0x7feb352du;
  h ^= h >> 15;
  h *= 0x846ca68bu;
  h ^= h >> 16;
  return (int)(h % 257u) - 128;
}

constexpr int kStTd = kXBuf;                          // T digits int8 [4][128][128]
constexpr int kStXd = kStTd + 4 * 128 * 128;          // x digits int8 [3][64][128]
constexpr int kStSmem = kStXd + 3 * 64 * 128 + 1024;

__global__ void __launch_bounds__(256, 1) tc_selftest_kernel(unsigned long long* bad, uint32_t seed) {
  __shared__ uint32_t tbase_sh;
  __shared__ __align__(8) uint64_t mbar;
  extern __shared__ uint8_t um_smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(um_smem_raw) + 1023) & ~(uintptr_t)1023);
  int8_t* td = reinterpret_cast<int8_t*>(sm + kStTd);
  int8_t* xd = reinterpret_cast<int8_t*>(sm + kStXd);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q = warp & 3, half = warp >> 2, i = 32 * q + lane;
  const int mode = (int)(blockIdx.x & 3u);
  if (tid == 0) {
    um_mbar_init(&mbar);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(um_saddr(&tbase_sh)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  const uint32_t sd = seed * 1000003u + blockIdx.x;
  for (int e = tid; e < 4 * 128 * 128; e += blockDim.x) {
    const int d = st_digit(sd, mode, e >> 14, e & 16383);
    td[e] = (int8_t)(d == 128 ? 127 : d);             // 127 stands for 127 or 128 (see tdig)
  }
  for (int e = tid; e < 3 * 64 * 128; e += blockDim.x) {
    const int a = e >> 13, rk = e & 8191;
    const int d = st_digit(sd, mode, 4 + a, rk);
    xd[e] = (int8_t)(d == 128 ? 127 : d);
    *reinterpret_cast<uint16_t*>(sm + a * kXSlice + xs_offset(rk >> 7, rk & 127)) = (uint16_t)digit_bf16(d);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tbase_sh, tlane = (uint32_t)(32 * q) << 16;
  // T digits of row i, this half, into TMEM in the rotation's packing
  for (int b = 0; b < 4; ++b)
    for (int blk = 0; blk < 4; ++blk) {
      uint32_t out[8];
      for (int col = 0; col < 8; ++col) {
        const int k = 64 * half + 16 * blk + 2 * col;
        out[col] = digit_bf16(st_digit(sd, mode, b, i * 128 + k)) | (digit_bf16(st_digit(sd, mode, b, i * 128 + k + 1)) << 16);
      }
      tmem_st8(tb + tlane + 64u * (uint32_t)b + 32u * (uint32_t)half + 8u * (uint32_t)blk, out);
    }
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    tc_fence_after();
    issue_chunk(tb, um_saddr(sm));
    umma_commit(&mbar);
  }
  const bool ok = um_mbar_wait(&mbar, 0u);
  tc_fence_after();
  uint32_t acc[4][32];
  for (int L = 0; L < 4; ++L) tmem_ld32(tb + tlane + kAccCol + 64u * (uint32_t)L + 32u * (uint32_t)half, acc[L]);
  for (int L = 0; L < 4; ++L) tmem_wait_ld32(acc[L]);
  // digits as stored (+128 kept as 127 in the int8 tables: recover it from the hash)
  auto tdig = [&](int b, int k) { const int v = td[(b << 14) + i * 128 + k]; return v == 127 ? st_digit(sd, mode, b, i * 128 + k) : v; };
  auto xdig = [&](int a, int r, int k) { const int v = xd[(a << 13) + r * 128 + k]; return v == 127 ? st_digit(sd, mode, 4 + a, r * 128 + k) : v; };
  constexpr int kA[9] = {0, 0, 1, 0, 1, 2, 0, 1, 2};
  constexpr int kB[9] = {0, 1, 0, 2, 1, 0, 3, 2, 1};
  unsigned long long wrong = ok ? 0ull : 1ull << 20;
  for (int c = 0; c < 32 && ok; ++c) {
    const int r = 32 * half + c;
    long long lev[4] = {0, 0, 0, 0};
    for (int cb = 0; cb < 9; ++cb) {
      long long sum = 0;
      for (int k = 0; k < 128; ++k) sum += (long long)xdig(kA[cb], r, k) * tdig(kB[cb], k);
      lev[kA[cb] + kB[cb]] += sum;
    }
    for (int L = 0; L < 4; ++L)
      if ((double)__uint_as_float(acc[L][c]) != (double)lev[L]) ++wrong;
  }
  if (wrong) atomicAdd(bad, wrong);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tb), "r"(kTmemCols) : "memory");
}

}  // namespace

int launch_rotate_tc(RotParams P, cudaStream_t stream) {
  // chunks of 64 pairs per matrix; chunks per tile chosen so that the slowest SM's work,
  // ceil(tiles / SMs) x (chunks per tile + one chunk's worth of matrix set-up), is least
  long long chunks_total = 0;
  long long cpm[3] = {0, 0, 0};
  for (int t = 0; t < 3; ++t)
    if (P.t[t].mode == ROT_DENSE) {
      cpm[t] = ((long long)P.t[t].rows * P.t[t].head_div + kUmRows - 1) / kUmRows;
      chunks_total += (long long)(P.t[t].heads / P.t[t].head_div) * cpm[t];
    }
  auto tiles_for = [&](long long rpc) {
    long long tiles = 0;
    for (int t = 0; t < 3; ++t)
      if (P.t[t].mode == ROT_DENSE) tiles += (long long)(P.t[t].heads / P.t[t].head_div) * ((cpm[t] + rpc - 1) / rpc);
    return tiles;
  };
  long long best = 1;
  double best_cost = 1e300;
  for (int waves = 1; waves <= 16; ++waves) {
    const long long rpc = std::max(1LL, (chunks_total + (long long)kSms * waves - 1) / ((long long)kSms * waves));
    const double cost = (double)((tiles_for(rpc) + kSms - 1) / kSms) * ((double)rpc + 1.0);
    if (cost < best_cost) {
      best_cost = cost;
      best = rpc;
    }
  }
  P.rpc = (int)std::min(best, (long long)(1 << 20));
  long long dense_total = 0;
  for (int t = 0; t < 3; ++t) {
    const long long tiles =
        P.t[t].mode == ROT_DENSE ? (long long)(P.t[t].heads / P.t[t].head_div) * ((cpm[t] + P.rpc - 1) / P.rpc) : 0;
    if (tiles > 0x3fffffffLL) return KVQ_ERR_UNSUPPORTED;
    P.n_dense[t] = (int)tiles;
    dense_total += tiles;
  }
  if (dense_total == 0) return KVQ_OK;
  if (dense_total > 0x7fffffffLL) return KVQ_ERR_UNSUPPORTED;
  P.dense_total = (int)dense_total;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ERR_CUDA;
  static std::mutex mu;
  static unsigned long long attr_done = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!(attr_done & (1ull << dev))) {
      if (cudaFuncSetAttribute(rotate_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kUmSmem) != cudaSuccess)
        return KVQ_ERR_CUDA;
      attr_done |= 1ull << dev;
    }
  }
  return launch_pdl(rotate_tc_kernel, dim3((unsigned)dense_total), dim3(256), (size_t)kUmSmem, stream, P) ==
                 cudaSuccess
             ? KVQ_OK
             : KVQ_ERR_CUDA;
}

}  // namespace kvq

extern "C" int kvq_launch_tc_selftest(unsigned long long* d_mismatches, cudaStream_t stream) {
  using namespace kvq;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ERR_CUDA;
  static std::mutex mu;
  static unsigned long long attr_done = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!(attr_done & (1ull << dev))) {
      if (cudaFuncSetAttribute(tc_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStSmem) != cudaSuccess)
        return KVQ_ERR_CUDA;
      attr_done |= 1ull << dev;
    }
  }
  for (uint32_t s = 0; s < 4; ++s) {
    tc_selftest_kernel<<<kSms, 256, kStSmem, stream>>>(d_mismatches, s);
    if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  }
  return KVQ_OK;
}
