// kv_append_chunk: a prefill chunk appended to each sequence in one pass -- transform on write
// and quantize-on-write fused, so rows that fall into the INT2 region never pass through the
// BF16 ring.
//
// Source: OScaR reading note, "系统设计与 CUDA 实现" (the key-quant kernel keeps the transform,
// the scaling and the INT2 packing on chip: the input is read once and the codes written once);
// OSCAR summary, section 4 "KV Cache Update" (prefill clip and quantize fused into one kernel);
// WUSH-KV digest, inference algorithm (keys transformed by T_K on write, S_flush-aligned spans
// beyond S_sink / S_keep quantized).
//
// The call is defined as the two-call path on the same rows: kv_rotate_qk at positions
// seq_len[b] .. seq_len[b] + n_b - 1, then kv_quant_flush -- every byte of the cache it
// writes is the same.  Three launches, each waiting for the previous one:
//   1. the flush of the tokens already in the ring that the advanced length pushes out of the
//      window; it publishes the new seq_len and s_quant (flush.cu, append mode);
//   2. the rows whose transform is the identity (values with T_V folded): read once, written
//      to their window row or quantized into their page (this file);
//   3. the dense transforms on the tensor cores (the exact digit scheme of rotate_tc.cu, from
//      tc.cuh); the decided rows of each 64-row chunk are staged in shared memory, then copied
//      to their window row or quantized into their page by the same octet quantizer.
#include "tc.cuh"

#include <algorithm>
#include <mutex>

namespace kvq {
namespace {

// The rows of chunk `chunk` of this warp, loaded ahead of slicing, with their sequence (from
// cu_rows; called after the dependency wait: the caller's last kernel may be writing them).
__device__ __forceinline__ void x_prefetch_append(const RotParams& P, const RotTensor& T, int mh, int chunk,
                                                  int pairs, int warp, int lane, XPre& pre) {
  const int p0 = chunk * kUmRows, np = min(kUmRows, pairs - p0);
  const int r = kRowsPerWarp * warp + (lane % kRowsPerWarp);
  pre.valid = (lane < kRowsPerWarp && r < np) ? 1 : 0;
  int row = 0, head = 0;
  if (r < np) tile_row(T, mh, p0 + r, row, head);
  pre.row = row;
  pre.head = head;
  pre.b = pre.p = 0;
  pre.sq = -1;
  if (pre.valid) pre.b = append_seq(P.cu_rows, P.batch, row);
#pragma unroll
  for (int j = 0; j < kRowsPerWarp; ++j) {
    const int rj = __shfl_sync(0xffffffffu, row, j), hj = __shfl_sync(0xffffffffu, head, j);
    pre.x[j] = make_uint2(0u, 0u);
    if (kRowsPerWarp * warp + j < np)
      pre.x[j] = __ldg(reinterpret_cast<const uint2*>(T.src + ((size_t)rj * T.heads + hj) * kHeadDim) + lane);
  }
}

// Digits of the prefetched rows -> x digit matrices (buffer xb) and row metadata.  Runs after
// the dependency wait (destinations read seq_len and s_quant).
__device__ __forceinline__ void x_slice_append(const RotParams& P, const RotTensor& T, const XPre& pre,
                                               uint8_t* xb, UmRow* meta, int warp, int lane) {
  void* dst = nullptr;
  const uint16_t* src = nullptr;
  int dflags = 0, tp = 0;
  if (pre.valid) {
    src = T.src + ((size_t)pre.row * T.heads + pre.head) * kHeadDim;
    const int kind = append_dst(P, T, pre.row, pre.head, pre.b, true, dst, tp);
    dflags = kind == kDstPage ? (kRowLive | kRowPage) : kind == kDstRow ? kRowLive : 0;
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
    const unsigned long long dj = __shfl_sync(0xffffffffu, (unsigned long long)dst, j);
    const unsigned long long sj = __shfl_sync(0xffffffffu, (unsigned long long)src, j);
    const int ftj = __shfl_sync(0xffffffffu, dflags | (tp << 8), j);
    const int fj = ftj & 0xff, tj = ftj >> 8;
    if (lane == 0) {
      const uint32_t ma = um_saddr(meta + kRowsPerWarp * warp + j);
      sts_u64(ma, dj);
      sts_u64(ma + 8, sj);
      sts_v2(ma + 16, (uint32_t)fr,
             (uint32_t)(fj | (zero ? kRowZero : 0) | (bad ? kRowBad : 0) | (lossy ? kRowLossy : 0)));
      sts_v2(ma + 24, (uint32_t)tj, 0u);
    }
  }
}

// The queued undecided outputs of a warp ((row << 7) | output), recomputed exactly (exact.cuh)
// into the chunk's staged rows; returns 0.
__device__ __noinline__ int exact_list_staged(const uint16_t* list, int count, const UmRow* mrow,
                                              const float* tmat, uint8_t* stg, int lane) {
  __syncwarp();
  for (int f = 0; f < count; ++f) {
    const int r = list[f] >> 7, o = list[f] & 127;
    exact_output_warp(tmat + (size_t)o * kHeadDim, mrow[r].src, reinterpret_cast<uint16_t*>(stg + r * kStgStride), o,
                      lane);
  }
  __syncwarp();
  return 0;
}

// Row phase of a chunk: the octet (lane / 8) of warp w takes staged row 4 w + lane / 8 (a row
// of the warp's own part), lane j = lane % 8 its channels 16 j .. 16 j + 15.  BF16
// destinations get the row with 16-byte stores (8-byte ones when the destination is only
// 8-byte aligned); page destinations get the quantized token.  The whole warp calls it.
__device__ __forceinline__ void row_phase(const UmRow* mrow, uint32_t stg_s, const QuantConsts& Qc, bool is_key,
                                          bool key_norm, int ng, int32_t* status, int warp, int lane) {
  const int r = 4 * warp + (lane >> 3), j = lane & 7;
  const uint32_t ma = um_saddr(mrow + r);
  void* dst = (void*)lds_u64(ma);
  const int flags = (int)lds_v2(ma + 16).y;
  const int tp = (int)lds_v2(ma + 24).x;
  const bool live = (flags & kRowLive) != 0, page = (flags & kRowPage) != 0;
  // lanes 4..7 of the octet read their upper 16 bytes first, so each quarter-warp's loads
  // cover the 32 banks once
  const int first = (j >> 2) & 1;
  const uint32_t rs = stg_s + (uint32_t)(r * kStgStride + 32 * j);
  const uint4 a = lds_v4(rs + 16u * (uint32_t)first), c = lds_v4(rs + 16u * (uint32_t)(1 - first));
  const uint4 lo = first ? c : a, hi = first ? a : c;          // channels 16j..16j+7, 16j+8..16j+15
  if (live && !page) {
    uint16_t* d = static_cast<uint16_t*>(dst) + 16 * j;
    if (((uintptr_t)d & 15u) == 0) {
      reinterpret_cast<uint4*>(d)[0] = lo;
      reinterpret_cast<uint4*>(d)[1] = hi;
    } else {
      uint2* d2 = reinterpret_cast<uint2*>(d);
      d2[0] = make_uint2(lo.x, lo.y);
      d2[1] = make_uint2(lo.z, lo.w);
      d2[2] = make_uint2(hi.x, hi.y);
      d2[3] = make_uint2(hi.z, hi.w);
    }
  }
  if (__any_sync(0xffffffffu, page)) {
    const uint32_t u[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    float y[16];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      y[2 * m] = __uint_as_float(u[m] << 16);
      y[2 * m + 1] = __uint_as_float(u[m] & 0xffff0000u);
    }
    quantize_store_octet(Qc, is_key, key_norm, y, page ? static_cast<uint8_t*>(dst) : nullptr, tp, ng, page, lane,
                         status);
  }
}


// The tensor-core rotation of rotate_tc.cu for appended rows: one CTA per tile of P.rpc chunks
// of 64 (row, head) pairs that share one matrix; warps 0 .. kWorkers - 1 slice rows and decide
// outputs, the last warp issues the MMAs.  Decided outputs go to the staged rows of the chunk;
// once the four warps of a part have decided theirs, the part's rows go out row by row (BF16
// window rows copied with 16-byte stores, page rows quantized by the octet quantizer).
__global__ void __launch_bounds__(kThreads, 1) append_tc_kernel(const RotParams Pk) {
  pdl_trigger();
  __shared__ RotParams Ps;
  __shared__ uint32_t tbase_sh;
  __shared__ __align__(8) uint64_t bar_x[2], bar_acc, bar_mma[2];
  __shared__ int tile_bad;
  __shared__ volatile int abort_sh;
  extern __shared__ uint8_t um_smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(um_smem_raw) + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool worker = warp < kWorkers;
  const int q = warp & 3, part = (warp >> 2) % kParts, i = 32 * q + lane;
  if (tid == 0) {
    Ps = Pk;
    tile_bad = 0;
    abort_sh = 0;
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
  uint16_t* list = reinterpret_cast<uint16_t*>(sm + kListOff) + (warp % kWorkers) * kList;
  int* ex_e = reinterpret_cast<int*>(sm + kExchOff);                           // [kParts][128]
  float* ex_s = reinterpret_cast<float*>(sm + kExchOff + kParts * 128 * 4);    // [kParts][128]
  auto xbuf = [&](int n) { return sm + (n & 1) * kXBuf; };

  // ---- the matrix (configuration: before the dependency wait) ----
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
    x_prefetch_append(P, T, mh, c0, pairs, warp, lane, pre);
    x_slice_append(P, T, pre, xbuf(0), meta, warp, lane);
    publish(0);
    if (nch > 1) {
      x_prefetch_append(P, T, mh, c0 + 1, pairs, warp, lane, pre);
      x_slice_append(P, T, pre, xbuf(1), meta + kUmRows, warp, lane);
      publish(1);
      if (nch > 2) x_prefetch_append(P, T, mh, c0 + 2, pairs, warp, lane, pre);
    }
    const QuantConsts Qc = quant_consts(P.qs[T.which], 16);
    const bool is_key = T.which == 0, key_norm = T.which == 0 && P.l2 != 0;
    int count = 0;
    bool dead = false;      // a bounded wait ran out: the warp only keeps meeting the barrier
    for (int n = 0; n < nch; ++n) {
      uint8_t* stg = sm + kStgOff + (n & 1) * kStgBuf;
      const uint32_t stg_s = um_saddr(stg);
      const UmRow* mrow = meta + (n & 3) * kUmRows;
      if (!dead && !warp_wait(&bar_mma[n & 1], (uint32_t)((n >> 1) & 1), &abort_sh, lane)) dead = true;
      if (!dead) {
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
      // ---- rounding decisions of chunk n: output i, rows kEpiRows part + c, into the staged
      // rows.  All rows first, without control flow (independent chains the scheduler
      // interleaves); undecided outputs are queued afterwards, only when the warp has any.
      const uint32_t mrow_s = um_saddr(mrow);
      uint32_t und_bits = 0;
#pragma unroll
      for (int c = 0; c < kEpiRows; ++c) {
        const int r = kEpiRows * part + c;
        const uint32_t ma = mrow_s + (uint32_t)r * (uint32_t)sizeof(UmRow);
        const uint2 ff = lds_v2(ma + 16);
        const int fr = (int)ff.x, flags = (int)ff.y;
        const bool live = (flags & kRowLive) != 0;
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
        if (live && b >= 0) sts_u16(stg_s + (uint32_t)(r * kStgStride + 2 * i), (uint32_t)b);
        und_bits |= (live && b < 0) ? (1u << c) : 0u;
      }
      if (__any_sync(0xffffffffu, und_bits != 0u)) {
#pragma unroll 1
        for (int c = 0; c < kEpiRows; ++c) {
          const bool und = (und_bits >> c) & 1u;
          const unsigned mk = __ballot_sync(0xffffffffu, und);
          if (und) list[count + __popc(mk & ((1u << lane) - 1u))] = (uint16_t)(((kEpiRows * part + c) << 7) | i);
          count += __popc(mk);
          if (count > kList - 32) count = exact_list_staged(list, count, mrow, tmat, stg, lane);
        }
      }
      count = exact_list_staged(list, count, mrow, tmat, stg, lane);
      }
      // ---- the four warps of a part meet here once per chunk (also after a timeout); then the
      // part's rows of chunk n go out: BF16 rows copied, page rows quantized ----
      part_sync(part);
      const int stop = __shfl_sync(0xffffffffu, abort_sh, 0);
      if (!stop) row_phase(mrow, stg_s, Qc, is_key, key_norm, P.ng, P.status, warp, lane);
      // ---- digits of chunk n + 2 into chunk n's buffer (its MMAs have completed) ----
      if (!dead && n + 2 < nch) {
        x_slice_append(P, T, pre, xbuf(n), meta + ((n + 2) & 3) * kUmRows, warp, lane);
        publish(n + 2);
        if (n + 3 < nch) x_prefetch_append(P, T, mh, c0 + n + 3, pairs, warp, lane, pre);
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

// One octet (8 lanes) per appended (row, head) of the copied tensor, four per warp.
__global__ void __launch_bounds__(256) append_copy_kernel(const RotParams Pk) {
  pdl_trigger();
  __shared__ RotParams Ps;
  if (threadIdx.x == 0) Ps = Pk;
  __syncthreads();
  const RotParams& P = Ps;
  const RotTensor& T = P.t[2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, j = lane & 7;
  const long long total = (long long)T.rows * T.heads;
  const QuantConsts Qc = quant_consts(P.qs[T.which], 16);
  const bool is_key = T.which == 0, key_norm = is_key && P.l2 != 0;
  const int heads = T.heads, batch = P.batch, ng = P.ng;
  // seq_len / s_quant come from the flush step, and its ring reads must be done before any
  // ring row is overwritten
  pdl_wait();
  for (long long base = ((long long)blockIdx.x * 8 + warp) * 4; base < total; base += (long long)gridDim.x * 32) {
    const long long item = base + (lane >> 3);
    const bool valid = item < total;
    const int row = valid ? (int)(item / heads) : 0, h = valid ? (int)(item % heads) : 0;
    uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
    if (valid) {
      const uint4* src = reinterpret_cast<const uint4*>(T.src + ((size_t)row * heads + h) * kHeadDim + 16 * j);
      lo = __ldg(src);
      hi = __ldg(src + 1);
    }
    void* dst = nullptr;
    int tp = 0, kind = kDstNone;
    if (valid) kind = append_dst(P, T, row, h, append_seq(P.cu_rows, batch, row), j == 0, dst, tp);
    if (kind == kDstRow) {
      uint4* d = reinterpret_cast<uint4*>(static_cast<uint16_t*>(dst) + 16 * j);
      d[0] = lo;
      d[1] = hi;
    }
    const bool page = kind == kDstPage;
    if (__any_sync(0xffffffffu, page)) {
      const uint32_t u[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
      float y[16];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        y[2 * m] = __uint_as_float(u[m] << 16);
        y[2 * m + 1] = __uint_as_float(u[m] & 0xffff0000u);
      }
      quantize_store_octet(Qc, is_key, key_norm, y, page ? static_cast<uint8_t*>(dst) : nullptr, tp, ng, page, lane,
                           P.status);
    }
  }
}

}  // namespace

static int launch_append_tc(RotParams P, cudaStream_t stream) {
  const int rc = plan_rotate_tc(P);
  if (rc != KVQ_OK || P.dense_total == 0) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ERR_CUDA;
  static std::mutex mu;
  static unsigned long long attr_done = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!(attr_done & (1ull << dev))) {
      if (cudaFuncSetAttribute(append_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kUmSmem) != cudaSuccess)
        return KVQ_ERR_CUDA;
      attr_done |= 1ull << dev;
    }
  }
  return launch_pdl(append_tc_kernel, dim3((unsigned)P.dense_total), dim3(kThreads), (size_t)kUmSmem, stream, P) ==
                 cudaSuccess
             ? KVQ_OK
             : KVQ_ERR_CUDA;
}

static int launch_append_copy(const RotParams& P, cudaStream_t stream) {
  const long long items = (long long)P.t[2].rows * P.t[2].heads;
  if (items == 0) return KVQ_OK;
  const long long ctas = std::min((items + 31) / 32, (long long)kSms * 6);
  return launch_pdl(append_copy_kernel, dim3((unsigned)ctas), dim3(256), 0, stream, P) == cudaSuccess ? KVQ_OK
                                                                                                        : KVQ_ERR_CUDA;
}

}  // namespace kvq

using namespace kvq;

extern "C" int kvq_launch_append(const kvq_config* cfg, const kvq_transform* tr, const uint16_t* k, const uint16_t* v,
                                 const int32_t* cu_rows, int32_t n_rows, const kvq_cache* cache, int32_t* d_status,
                                 cudaStream_t stream) {
  int rc = kvq_launch_flush_append(cfg, cache, cu_rows, d_status, stream);
  if (rc != KVQ_OK || n_rows == 0) return rc;
  RotParams P{};
  const int gqa = cfg->n_q_heads / cfg->n_kv_heads;
  P.t[0] = RotTensor{nullptr, 0, cfg->n_q_heads, ROT_DENSE, tr->t_k_inv_t, gqa, 1, nullptr, nullptr, nullptr, 0, 0};
  P.t[1] = RotTensor{k, n_rows, cfg->n_kv_heads, ROT_DENSE, tr->t_k, 1, 0, nullptr, cache->sink_k, cache->ring_k, 0, 0};
  P.t[2] = RotTensor{v, n_rows, cfg->n_kv_heads, tr->t_v ? ROT_DENSE : ROT_COPY, tr->t_v, 1, 0, nullptr,
                     cache->sink_v, cache->ring_v, 0, 1};
  P.seq_len = cache->seq_len;
  P.s_quant = cache->s_quant;
  P.s_sink = cfg->s_sink;
  P.ring_cap = cfg->ring_cap;
  P.batch = cfg->batch;
  P.hkv = cfg->n_kv_heads;
  P.status = d_status;
  P.cu_rows = cu_rows;
  P.pages = (uint8_t*)cache->pages;
  P.page_table = cache->page_table;
  P.max_pages = cfg->max_pages_per_seq;
  P.num_pages = cfg->num_pages;
  P.page_bytes = page_head_bytes(cfg->group_size, cfg->key_l2norm, cfg->key_axis);
  P.ng = kHeadDim / cfg->group_size;
  P.l2 = cfg->key_l2norm;
  P.qs[0] = make_quant_spec(cfg->group_size, cfg->quantizer, cfg->kappa_k, cfg->quest_alpha);
  P.qs[1] = make_quant_spec(cfg->group_size, cfg->quantizer, cfg->kappa_v, cfg->quest_alpha);
  for (int i = 1; i < 3; ++i)
    if ((long long)P.t[i].rows * P.t[i].heads > 0x3fffffffLL) return KVQ_ERR_UNSUPPORTED;
  if (P.t[2].mode == ROT_COPY) {
    rc = launch_append_copy(P, stream);
    if (rc != KVQ_OK) return rc;
  }
  return launch_append_tc(P, stream);
}
