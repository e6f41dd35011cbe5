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
//     exponent field of the row: |T_ij| / U_i < 128, kept to 2^-25 units as four balanced
//     base-256 digits t_0 + t_1/2^8 + t_2/2^16 + t_3/2^24, each an integer in [-128, 128]
//     (round-to-nearest extraction in fp32, every step exact);
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
// rounded bf16 whenever no rounding midpoint lies within that bound; the rest (about 0.2% of
// the outputs on the chunk workload's keys: near a midpoint, tiny after cancellation, or on
// rows with an element 16 or more binades below the row's largest; non-finite and subnormal
// results always) are recomputed by the exact tiers of exact.cuh -- queued for the whole tile
// and shared out over the worker warps after its last chunk, so no chunk waits for them.
//
// Layout (one CTA of 17 warps per SM, it holds all 512 TMEM columns):
//   TMEM columns   0..255  the four T digit matrices, A operand (lane = output i, K packed
//                          two bf16 per column), written once per tile;
//   TMEM columns 256..511  the four level accumulators D_L for a chunk of 64 rows
//                          (lane = output i, column = row);
//   shared memory          the three x digit matrices of a chunk (B operand, K-major,
//                          128-byte swizzle), double-buffered; per-row metadata; the
//                          tile's queue of undecided outputs.
// Warp 16 issues the 72 MMAs of a chunk (M = 128, N = 64, K = 16 each) as soon as the
// chunk's digits are written and the previous chunk's sums were read; warps 0-15 read the
// accumulators into registers at once (so the next chunk's MMAs overlap this chunk's rounding
// decisions and stores), then slice the rows of the chunk after next.
#include "tc.cuh"

#include <mutex>

namespace kvq {
namespace {

// after_wait: s_quant may be read (it is written by the previous kernel of a step)
__device__ __forceinline__ void x_prefetch(const RotParams& P, const RotTensor& T, int mh, int chunk, int pairs,
                                           int warp, int lane, bool after_wait, XPre& pre) {
  const int p0 = chunk * kUmRows, np = min(kUmRows, pairs - p0);
  const int r = kRowsPerWarp * warp + (lane % kRowsPerWarp);
  pre.valid = (lane < kRowsPerWarp && r < np) ? 1 : 0;
  int row = 0, head = 0;
  if (r < np) tile_row(T, mh, p0 + r, row, head);
  pre.row = row;
  pre.head = head;
  pre.b = pre.p = 0;
  pre.sq = -1;
  if (pre.valid && !T.is_query) {
    pre.b = __ldg(P.seq_idx + row);
    pre.p = __ldg(P.pos + row);
    if (after_wait && pre.b >= 0 && pre.b < P.batch) pre.sq = P.s_quant[pre.b];
  }
#pragma unroll
  for (int j = 0; j < kRowsPerWarp; ++j) {
    const int rj = __shfl_sync(0xffffffffu, row, j), hj = __shfl_sync(0xffffffffu, head, j);
    pre.x[j] = make_uint2(0u, 0u);
    if (kRowsPerWarp * warp + j < np)
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
    dst = rot_dst(P, T, pre.row, pre.head, pre.b, pre.p, true, pre.sq);
  }
#pragma unroll
  for (int j = 0; j < kRowsPerWarp; ++j) {
    const float xf[4] = {__uint_as_float(pre.x[j].x << 16), __uint_as_float(pre.x[j].x & 0xffff0000u),
                         __uint_as_float(pre.x[j].y << 16), __uint_as_float(pre.x[j].y & 0xffff0000u)};
    const uint32_t am = max(max(__float_as_uint(fabsf(xf[0])), __float_as_uint(fabsf(xf[1]))),
                            max(__float_as_uint(fabsf(xf[2])), __float_as_uint(fabsf(xf[3]))));
    const uint32_t amax = __reduce_max_sync(0xffffffffu, am);     // non-negative floats order as integers
    const int fr = max(1, (int)(amax >> 23));                        // (a NaN is caught by `bad`)
    const bool bad = amax >= 0x7f800000u, zero = amax == 0u;
    const int k = 133 - fr;
    float d[3][4];
    bool lost_l = false;
#pragma unroll
    for (int m2 = 0; m2 < 4; ++m2) {
      float r = scale_pow2(xf[m2], k);
      lost_l |= (r == 0.f) && (xf[m2] != 0.f);
#pragma unroll
      for (int a = 0; a < 3; ++a) d[a][m2] = next_digit(r);
      lost_l |= r != 0.f;
    }
    const bool lossy = __any_sync(0xffffffffu, lost_l);
    const int offj = xs_offset(kRowsPerWarp * warp + j, 4 * lane);
#pragma unroll
    for (int a = 0; a < 3; ++a)
      sts_v2(um_saddr(xb) + (uint32_t)(a * kXSlice + offj), pack_digits(d[a][0], d[a][1]),
             pack_digits(d[a][2], d[a][3]));
    uint16_t* dj = (uint16_t*)__shfl_sync(0xffffffffu, (unsigned long long)dst, j);
    const uint16_t* sj = (const uint16_t*)__shfl_sync(0xffffffffu, (unsigned long long)src, j);
    if (lane == 0) {
      const uint32_t ma = um_saddr(meta + kRowsPerWarp * warp + j);
      sts_u64(ma, (unsigned long long)dj);
      sts_u64(ma + 8, (unsigned long long)sj);
      sts_v2(ma + 16, (uint32_t)fr, (uint32_t)((zero ? kRowZero : 0) | (bad ? kRowBad : 0) | (lossy ? kRowLossy : 0)));
    }
  }
}

// Undecided outputs of a tile, queued in the shared memory the staging of appends would use
// and recomputed exactly (exact.cuh) after the tile's last chunk by all worker warps at once:
// recomputing them within each chunk made every chunk wait for the warp that drew the most.
struct XqEntry {
  uint16_t* dst;         // destination row
  uint32_t src_row;      // source row (row * heads + head) of the tensor
  uint32_t o;            // output index
};
static_assert(sizeof(XqEntry) == 16, "XqEntry layout");
constexpr int kUmSmemTile = 152 * 1024;                     // dynamic shared memory of this kernel
constexpr int kXqCap = (kUmSmemTile - 1024 - kStgOff) / (int)sizeof(XqEntry);


// One CTA per tile: P.rpc chunks of 64 (row, head) pairs that share one matrix.  Warps
// 0 .. kWorkers - 1 slice rows and decide outputs; the last warp issues the MMAs.
__global__ void __launch_bounds__(kThreads, 1) rotate_tc_kernel(const RotParams Pk) {
  pdl_trigger();
  __shared__ RotParams Ps;
  __shared__ uint32_t tbase_sh;
  __shared__ __align__(8) uint64_t bar_x[2], bar_acc, bar_mma[2];
  __shared__ int tile_bad;
  __shared__ volatile int abort_sh;
  __shared__ int xq_count;
  extern __shared__ uint8_t um_smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(um_smem_raw) + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool worker = warp < kWorkers;
  const int q = warp & 3, part = (warp >> 2) % kParts, i = 32 * q + lane;
  if (tid == 0) {
    Ps = Pk;
    tile_bad = 0;
    abort_sh = 0;
    xq_count = 0;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(um_saddr(&bar_x[0])), "r"(kWorkers) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(um_saddr(&bar_x[1])), "r"(kWorkers) : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(um_saddr(&bar_acc)), "r"(kWorkers) : "memory");
    um_mbar_init(&bar_mma[0]);
    um_mbar_init(&bar_mma[1]);
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
  XqEntry* xq = reinterpret_cast<XqEntry*>(sm + kStgOff);
  int* ex_e = reinterpret_cast<int*>(sm + kExchOff);                           // [kParts][128]
  float* ex_s = reinterpret_cast<float*>(sm + kExchOff + kParts * 128 * 4);    // [kParts][128]
  auto xbuf = [&](int n) { return sm + (n & 1) * kXBuf; };

  // ---- the matrix (configuration: before the dependency wait; the call's rows, sequences and
  // positions only after it, as the caller's last kernel may still be writing them) ----
  XPre pre;
  int e_i = 1, tnz = 0;
  float st16 = 0.f;
  const float* trow = tmat + (size_t)i * kHeadDim + kTSpan * part;
  if (worker) {
    int e = 1, nz = 0, bad = 0;
#pragma unroll 4
    for (int j4 = 0; j4 < kTSpan / 4; ++j4) {
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
    ex_e[part * 128 + i] = e | (nz << 16);
    if (bad) tile_bad = 1;
  }
  __syncthreads();
  if (worker) {
#pragma unroll
    for (int pp = 0; pp < kParts; ++pp) {
      const int a = ex_e[pp * 128 + i];
      e_i = max(e_i, a & 0xffff);
      tnz |= a >> 16;
    }
    ex_s[part * 128 + i] =
        slice_t_part(trow, e_i, tb + tlane + (uint32_t)(kTSpan / 2) * (uint32_t)part);
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // X's truncation (lossy rows): 2^-16 sum_j |T_ij| / U_i, rounded up
  if (worker) {
    float ssum = 0.f;
#pragma unroll
    for (int pp = 0; pp < kParts; ++pp) ssum += ex_s[pp * 128 + i];
    st16 = ssum * 0x1.01p-16f;
  }
  const bool force = tile_bad != 0;

  pdl_wait();
  if (!worker) {
    // ---- MMA warp: chunk n once its digits are written and chunk n - 1's sums were read ----
    if (lane == 0) {
      int last = -1;
      for (int n = 0; n < nch; ++n) {
        if (!um_wait(&bar_x[n & 1], (uint32_t)((n >> 1) & 1), &abort_sh)) break;
        if (n > 0 && !um_wait(&bar_acc, (uint32_t)((n - 1) & 1), &abort_sh)) break;
        tc_fence_after();
        issue_chunk(tb, um_saddr(xbuf(n)));
        umma_commit(&bar_mma[n & 1]);
        last = n;
      }
      if (abort_sh && last >= 0) {
        // the last committed chunk must finish before TMEM is released (bounded)
        for (long long it = 0; it < kSpinLimit; ++it)
          if (um_mbar_try(&bar_mma[last & 1], (uint32_t)((last >> 1) & 1))) break;
      }
    }
  } else {
    // ---- worker warps ----
    auto publish = [&](int n) {             // chunk n's digits (buffer n & 1) -> the MMA warp
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) um_arrive(&bar_x[n & 1]);
    };
    x_prefetch(P, T, mh, c0, pairs, warp, lane, true, pre);
    x_slice(P, T, pre, xbuf(0), meta, warp, lane);
    publish(0);
    if (nch > 1) {
      x_prefetch(P, T, mh, c0 + 1, pairs, warp, lane, true, pre);
      x_slice(P, T, pre, xbuf(1), meta + kUmRows, warp, lane);
      publish(1);
      if (nch > 2) x_prefetch(P, T, mh, c0 + 2, pairs, warp, lane, true, pre);
    }
    for (int n = 0; n < nch; ++n) {
      if (!warp_wait(&bar_mma[n & 1], (uint32_t)((n >> 1) & 1), &abort_sh, lane)) break;
      tc_fence_after();
      uint32_t acc[4][kEpiRows];
#pragma unroll
      for (int L = 0; L < 4; ++L)
        tmem_ld16(tb + tlane + kAccCol + 64u * (uint32_t)L + (uint32_t)(kEpiRows * part), acc[L]);
#pragma unroll
      for (int L = 0; L < 4; ++L) tmem_wait_ld16(acc[L]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) um_arrive(&bar_acc);
      // ---- rounding decisions of chunk n: output i, rows kEpiRows part + c ----
      // All rows first, without control flow (independent chains the scheduler interleaves);
      // undecided outputs are queued afterwards, only when the warp has any.
      const UmRow* mrow = meta + (n & 3) * kUmRows;
      const uint32_t mrow_s = um_saddr(mrow);
      uint32_t und_bits = 0;
#pragma unroll
      for (int c = 0; c < kEpiRows; ++c) {
        const int r = kEpiRows * part + c;
        const uint32_t ma = mrow_s + (uint32_t)r * (uint32_t)sizeof(UmRow);
        uint16_t* dst = (uint16_t*)lds_u64(ma);
        const uint2 ff = lds_v2(ma + 16);
        const int fr = (int)ff.x, flags = (int)ff.y;
        const float v = fmaf(__uint_as_float(acc[3][c]), 0x1p-24f,
                             fmaf(__uint_as_float(acc[2][c]), 0x1p-16f,
                                  fmaf(__uint_as_float(acc[1][c]), 0x1p-8f, __uint_as_float(acc[0][c]))));
        const float bnd = fmaf(fabsf(v), 0x1.81p-23f, (flags & kRowLossy) ? kBoundConst + st16 : kBoundConst);
        // the midpoint above v's bf16 truncation; with bound < |v| / 1024 no other midpoint is
        // as close (the decision is the same after the exact scaling by 2^S below)
        const float mid = __uint_as_float((__float_as_uint(v) & 0xffff0000u) | 0x8000u);
        const bool decided = fabsf(v - mid) > bnd && bnd * 1024.0f < fabsf(v);
        const int bu = (int)__bfloat16_as_ushort(__float2bfloat16_rn(v));
        // y = v 2^S, S = e_i + f_r - 266: shift the exponent field; the result must stay normal
        const int ey = ((bu >> 7) & 0xff) + e_i + fr;
        int b = (decided && (unsigned)(ey - 267) < 254u) ? bu + (ey - 266 - ((bu >> 7) & 0xff)) * 128 : -1;
        b = ((flags & kRowZero) || !tnz) ? 0 : b;           // an exact zero is +0
        b = (force || (flags & kRowBad)) ? -1 : b;
        if (dst != nullptr && b >= 0) __stcg(reinterpret_cast<unsigned short*>(dst + i), (unsigned short)b);
        und_bits |= (dst != nullptr && b < 0) ? (1u << c) : 0u;
      }
      if (__any_sync(0xffffffffu, und_bits != 0u)) {
#pragma unroll 1
        for (int c = 0; c < kEpiRows; ++c) {
          const bool und = (und_bits >> c) & 1u;
          const unsigned mk = __ballot_sync(0xffffffffu, und);
          if (!mk) continue;
          int base = 0;
          if (lane == 0) base = atomicAdd(&xq_count, __popc(mk));
          base = __shfl_sync(0xffffffffu, base, 0);
          const int r = kEpiRows * part + c;
          const int pos = base + __popc(mk & ((1u << lane) - 1u));
          if (und && pos < kXqCap)
            xq[pos] = XqEntry{static_cast<uint16_t*>(mrow[r].dst),
                              (uint32_t)((mrow[r].src - T.src) / kHeadDim), (uint32_t)i};
          // beyond the queue's capacity: recomputed at once (the whole warp, one output at a time)
          unsigned over = __ballot_sync(0xffffffffu, und && pos >= kXqCap);
          while (over) {
            const int l = __ffs(over) - 1;
            over &= over - 1;
            const int o = __shfl_sync(0xffffffffu, i, l);
            exact_output_warp(tmat + (size_t)o * kHeadDim, mrow[r].src, static_cast<uint16_t*>(mrow[r].dst), o,
                              lane);
          }
        }
      }
      // ---- digits of chunk n + 2 into chunk n's buffer (its MMAs have completed) ----
      if (n + 2 < nch) {
        x_slice(P, T, pre, xbuf(n), meta + ((n + 2) & 3) * kUmRows, warp, lane);
        publish(n + 2);
        if (n + 3 < nch) x_prefetch(P, T, mh, c0 + n + 3, pairs, warp, lane, true, pre);
      }
    }
    // ---- the tile's queued undecided outputs, spread over the worker warps (every worker warp
    // meets this barrier once, also after a timeout) ----
    asm volatile("bar.sync 1, %0;" ::"r"(kWorkers * 32) : "memory");
    // one output per lane (tier 2 by one thread), the few it leaves undecided by the whole warp
    const int nq = min(xq_count, kXqCap);
    for (int e0 = 32 * warp; e0 < nq; e0 += 32 * kWorkers) {
      const int e = e0 + lane;
      XqEntry x{nullptr, 0u, 0u};
      int r = 0;
      if (e < nq) {
        x = xq[e];
        r = exact_dot_tier2_row(tmat + (size_t)x.o * kHeadDim, T.src + (size_t)x.src_row * kHeadDim);
        if (r >= 0) x.dst[x.o] = (uint16_t)r;
      }
      unsigned und = __ballot_sync(0xffffffffu, e < nq && r < 0);
      while (und) {
        const int l = __ffs(und) - 1;
        und &= und - 1;
        uint16_t* dst = (uint16_t*)__shfl_sync(0xffffffffu, (unsigned long long)x.dst, l);
        const uint32_t srow = __shfl_sync(0xffffffffu, x.src_row, l), o = __shfl_sync(0xffffffffu, x.o, l);
        exact_output_warp(tmat + (size_t)o * kHeadDim, T.src + (size_t)srow * kHeadDim, dst, (int)o, lane);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && abort_sh) set_status(P.status, KVQ_ERR_TIMEOUT);   // whichever warp gave up
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

int plan_rotate_tc(RotParams& P) {
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
  if (dense_total > 0x7fffffffLL) return KVQ_ERR_UNSUPPORTED;
  P.dense_total = (int)dense_total;
  return KVQ_OK;
}

int launch_rotate_tc(RotParams P, cudaStream_t stream) {
  const int rc = plan_rotate_tc(P);
  if (rc != KVQ_OK || P.dense_total == 0) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ERR_CUDA;
  static std::mutex mu;
  static unsigned long long attr_done = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!(attr_done & (1ull << dev))) {
      if (cudaFuncSetAttribute(rotate_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kUmSmemTile) !=
          cudaSuccess)
        return KVQ_ERR_CUDA;
      attr_done |= 1ull << dev;
    }
  }
  return launch_pdl(rotate_tc_kernel, dim3((unsigned)P.dense_total), dim3(kThreads), (size_t)kUmSmemTile, stream,
                    P) ==
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
