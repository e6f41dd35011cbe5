// Shared pieces of the tensor-core rotation kernels (kv_rotate_qk at prefill size and
// kv_append_chunk): shared-memory layout, tcgen05 / TMEM / mbarrier primitives, the integer
// digits of T and x, the 72 MMAs of a chunk, and the bounded waits.  The exactness argument
// and the layout are described in rotate_tc.cu.
#pragma once
#include "rotate.cuh"

namespace kvq {
namespace {


constexpr int kUmRows = 64;                          // rows of a chunk (N of every MMA)
constexpr int kXSlice = kUmRows * kHeadDim * 2;      // one x digit matrix: 16 KB
constexpr int kXBuf = 3 * kXSlice;                   // three digit matrices per chunk buffer
constexpr int kList = 256;                           // queued undecided outputs per warp

// per-row metadata of a chunk (four buffers: warps run up to three chunks apart)
struct UmRow {
  void* dst;             // BF16 destination row, or the (page, kv head) chunk (kRowPage)
  const uint16_t* src;   // the source row (for exact recomputation)
  int fr;                // exponent field f_r of the row's units
  int flags;             // kRowZero | kRowBad | kRowLossy | kRowLive | kRowPage
  int tp;                // token slot in the page (kRowPage)
  int pad;
};
static_assert(sizeof(UmRow) == 32, "UmRow layout");
constexpr int kRowZero = 1, kRowBad = 2, kRowLossy = 4, kRowLive = 8, kRowPage = 16;

constexpr int kWorkers = 16;                         // warps that slice rows and decide outputs
constexpr int kThreads = 32 * (kWorkers + 1);        // + one warp that issues the MMAs
constexpr int kRowsPerWarp = kUmRows / kWorkers;     // rows a worker warp slices per chunk
constexpr int kParts = kWorkers / 4;                 // worker warps per TMEM lane quadrant
constexpr int kEpiRows = kUmRows / kParts;           // rows (accumulator columns) per thread
constexpr int kTSpan = kHeadDim / kParts;            // entries of a T row per thread

constexpr int kMetaOff = 2 * kXBuf;
constexpr int kListOff = kMetaOff + 4 * kUmRows * (int)sizeof(UmRow);
constexpr int kExchOff = kListOff + kWorkers * kList * 2;
constexpr int kStgOff = kExchOff + 2 * kParts * 128 * 4;   // after the exponent and |T| sum exchange
// decided rows of a chunk, row-major (128 bf16 + 16 bytes per row: an octet's 16-byte loads
// of one row fall in distinct banks), double-buffered
constexpr int kStgStride = 272;
constexpr int kStgBuf = kUmRows * kStgStride;
constexpr int kUmUsed = kStgOff + 2 * kStgBuf;
// more than half of an SM's shared memory: never two CTAs on one SM (each holds all of TMEM);
// without staging (kv_rotate_qk) the kernel asks only for what it uses, which leaves the rest
// of the SM's 256 KB to L1
constexpr int kUmSmem = 156 * 1024;
constexpr int kUmSmemPlain = 120 * 1024;
static_assert(kStgOff + 1024 <= kUmSmemPlain, "shared memory layout without staging");
static_assert(kUmUsed + 1024 <= kUmSmem, "shared memory layout");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 256;
// instruction descriptor, kind::f16: D f32, A and B bf16, both K-major, N = 64, M = 128
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kUmRows >> 3) << 17) |
                            ((128u >> 4) << 24);
constexpr long long kSpinLimit = 1LL << 22;      // try_wait rounds before a wait gives up

// ---- tcgen05 / mbarrier primitives ---------------------------------------------------------
__device__ __forceinline__ uint32_t um_saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
// explicit shared-memory accesses (the buffers are reached through a re-aligned pointer, which
// the compiler would otherwise treat as generic)
__device__ __forceinline__ void sts_v2(uint32_t a, uint32_t x, uint32_t y) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(a), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void sts_u64(uint32_t a, unsigned long long x) {
  asm volatile("st.shared.u64 [%0], %1;" ::"r"(a), "l"(x) : "memory");
}
__device__ __forceinline__ unsigned long long lds_u64(uint32_t a) {
  unsigned long long x;
  asm volatile("ld.shared.u64 %0, [%1];" : "=l"(x) : "r"(a) : "memory");
  return x;
}
__device__ __forceinline__ uint2 lds_v2(uint32_t a) {
  uint2 x;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(x.x), "=r"(x.y) : "r"(a) : "memory");
  return x;
}
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 x;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w) : "r"(a)
               : "memory");
  return x;
}
__device__ __forceinline__ void sts_u16(uint32_t a, uint32_t x) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"((unsigned short)x) : "memory");
}
// barrier 1 + part: the four worker warps of one part (rows 16 part .. 16 part + 15 of a
// chunk, all 128 outputs); the MMA warp never takes part
__device__ __forceinline__ void part_sync(int part) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + part) : "memory");
}
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
#define UM_O8(b)                                                                                            \
  "=r"(v[b]), "=r"(v[b + 1]), "=r"(v[b + 2]), "=r"(v[b + 3]), "=r"(v[b + 4]), "=r"(v[b + 5]), "=r"(v[b + 6]), \
      "=r"(v[b + 7])
// 16 consecutive TMEM columns of this warp's 32 lanes -> registers (not yet waited for)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : UM_O8(0), UM_O8(8)
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
__device__ __forceinline__ void tmem_wait_ld16(uint32_t* v) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : UM_IO8(0), UM_IO8(8)::"memory");
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

// v * 2^k, exact whenever the result is a normal float (k in [-126, 254])
__device__ __forceinline__ float scale_pow2(float v, int k) {
  if (k > 127) {
    v *= 0x1p64f;
    k -= 64;
  }
  return v * __int_as_float((k + 127) << 23);
}

// bf16 bits of two integer-valued floats of at most 8 significant bits (exact), low = a
__device__ __forceinline__ uint32_t pack_digits(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Balanced base-256 digits of X (|X| < 128): X = d0 + d1/2^8 + d2/2^16 (+ d3/2^24) + rest,
// each digit an integer in [-128, 128] (round to nearest, so the rest is at most half a unit
// of the last digit).  Every step is exact in fp32.
__device__ __forceinline__ float next_digit(float& r) {
  const float d = rintf(r);
  r = (r - d) * 256.0f;
  return d;
}

// T row i, entries kTSpan part .. (global) -> the four digit matrices in TMEM columns
// 64 b + kTSpan / 2 part + ..., this warp's lanes.  Returns sum_j |T_ij| / U_i over them.
__device__ __forceinline__ float slice_t_part(const float* trow, int e_i, uint32_t taddr) {
  const int k = 133 - e_i;
  float asum = 0.f;
#pragma unroll 1
  for (int blk = 0; blk < kTSpan / 16; ++blk) {
    uint32_t out[4][8];
#pragma unroll
    for (int j4 = 0; j4 < 4; ++j4) {
      const float4 t4 = reinterpret_cast<const float4*>(trow)[4 * blk + j4];
      float d[2][2][4];                                 // [pair element][column][digit]
      const float tv[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
      for (int m2 = 0; m2 < 4; ++m2) {
        float r = scale_pow2(tv[m2], k);
        asum += fabsf(r);
#pragma unroll
        for (int b = 0; b < 4; ++b) d[m2 & 1][m2 >> 1][b] = next_digit(r);
      }
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
        for (int b = 0; b < 4; ++b) out[b][2 * j4 + c2] = pack_digits(d[0][c2][b], d[1][c2][b]);
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) tmem_st8(taddr + 64u * (uint32_t)b + 8u * (uint32_t)blk, out[b]);
  }
  return asum;
}

// One worker warp's rows of a chunk, loaded ahead of slicing.
struct XPre {
  uint2 x[kRowsPerWarp];  // this lane's 4 bf16 (k = 4 lane .. 4 lane + 3) of rows R w + j
  int row, head, b, p;    // lanes 0..R-1: indices of row R w + lane (b, p for cache rows;
                          // appended rows: b from cu_rows, p found after the dependency wait)
  int sq;                 // lanes 0..R-1: s_quant[b] (cache rows, loaded after the dependency wait)
  int valid;              // lanes 0..R-1: the row exists
};

// Bounded wait that also gives up when another warp has given up.
__device__ __noinline__ bool um_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  for (long long it = 0; it < kSpinLimit; ++it) {
    if (um_mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}
// The same, decided by lane 0 for the whole warp (so the warp stays converged).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int lane) {
  int ok = 0;
  if (lane == 0) ok = um_wait(bar, parity, abort_flag) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}
__device__ __forceinline__ void um_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(um_saddr(bar)) : "memory");
}

// Constant part of the bound, units of U_i V_r: T's digits kept to 2^-25 (2^-25 sum |x| <=
// 2^-11), the digit products dropped ((1,3), (2,2): 2^-11 each; (2,3): 2^-19) and the fp32
// combination of the levels beyond 3u|v| (2^-17).
constexpr float kBoundConst = 0x1.9p-10f;

}  // namespace
}  // namespace kvq
