// kv_rotate_qk: per-head transform of new keys / values on write and compensation of
// queries, every output the exact product rounded once to bf16.
//
// Source: WUSH-KV digest, core method and inference algorithm (online key transform
// after RoPE, queries compensated with T^{-T}); OScaR reading note, step 1 "Canalized
// Rotation" (online FHT of K and Q, H H^T = I, inner products preserved); OSCAR
// summary, section 3 "Online Deployment" (fixed transforms applied while serving).
//
// Design (GB300): one launch covers queries, keys and values.  A dense row is a
// 128x128 float32 matrix times a bf16 vector; every output must be the correctly rounded
// bf16 of the exact value -- the flush quantizes these rows, so they must not depend on
// summation order.  The fp32 FMA sum plus a rigorous error bound decides the rounding for
// almost every output; the rest go to exact.cuh (double-float with its own bound, then, only
// within that bound of a midpoint, an exact fixed-point sum).  The matrices stay L2-resident
// across decode steps.
// The Hadamard transform is a warp-wide butterfly (two in-thread stages, five shuffle
// stages): in exact int64 arithmetic when the row's elements span fewer than 32 binades (the
// usual case), else in double-float with an error bound; then one scaling by 1/sqrt(d) with a
// bound, and outputs the bound leaves undecided are recomputed exactly (exact.cuh).
#include "rotate.cuh"
#include "exact.cuh"

namespace kvq {


// One dense tile per CTA of 256 threads: chunks of up to RT rows that share matrix mh, the
// matrix loaded once per tile.  Thread 2i + half
// keeps its 64 matrix entries T[mh][i][64 half .. 64 half + 63] in registers and forms, for
// every row, four fp32 FMA chains v_k = RN(v_{k-1} + T_ik x_k) of 16 terms each, which three
// additions inside the thread and one with the partner thread combine.  Every rounding r adds
// an error of at most u |r| (u = 2^-24), so with A = the sum of |r| over all partial results
// (chains, combining sums and the final v), |v - y| <= u A for y = sum_j T_ij x_j (plus at most
// 2^-142 from underflow; the fp32 evaluation of A is covered by a factor 1 + 2^-16).  bf16(v)
// is then the correctly rounded result unless a rounding midpoint lies within that distance;
// those few outputs are recomputed by a warp each after the tile (exact_dot_bf16_warp).
// Loads are issued in the order that overlaps them: the destination's sequence index and
// position, the matrix, the rows, and only then the dependent s_quant check.
constexpr int kMaxRT = 16;
constexpr int kXPad = 4;
constexpr int kMaxRPW = 8;
template <bool kMulti>
__device__ void dense_tile(const RotParams& P, int tt, int tile) {
  const RotTensor& T = P.t[tt];
  const int pairs = T.rows * T.head_div;                 // (row, head) pairs per matrix
  const int chunks_per_mat = (pairs + P.rt - 1) / P.rt;
  const int tiles_per_mat = (chunks_per_mat + P.rpc - 1) / P.rpc;
  const int mh = tile / tiles_per_mat;
  const int c0 = (tile % tiles_per_mat) * P.rpc;         // first chunk of this tile
  const int c1 = kMulti ? min(chunks_per_mat, c0 + P.rpc) : c0 + 1;
  // rows as floats; the second half of a row starts 4 floats later (kXPad) so that the two
  // half-row broadcasts of one load fall in different banks
  __shared__ __align__(16) float xs[kMaxRT][kHeadDim + kXPad];
  __shared__ uint16_t* dst_sh[kMaxRT];
  __shared__ uint16_t fallback[kMaxRT * kHeadDim];      // (row << 7) | output, undecided outputs
  __shared__ int n_fallback;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int i = tid >> 1, half = tid & 1;
  const int xrow = tid >> 4, xpart = tid & 15;
  // the chunk's destinations and rows: one 16-byte piece (8 bf16) of a row per thread
  int d_row = 0, d_head = 0, d_b = 0, d_p = 0;
  uint4 xr = make_uint4(0u, 0u, 0u, 0u);
  auto load_chunk = [&](int c) {
    const int p0 = c * P.rt, np = min(P.rt, pairs - p0);
    if (tid < np) {
      tile_row(T, mh, p0 + tid, d_row, d_head);
      if (!T.is_query) {
        d_b = P.seq_idx[d_row];
        d_p = P.pos[d_row];
      }
    }
    if (xrow < np) {
      int row, head;
      tile_row(T, mh, p0 + xrow, row, head);
      xr = reinterpret_cast<const uint4*>(T.src + ((size_t)row * T.heads + head) * kHeadDim)[xpart];
    }
  };
  // the matrix, once per tile: thread 2i + half keeps T[mh][i][64 half .. 64 half + 63].  A
  // transform is configuration, read before the dependency wait (it overlaps the kernel before
  // this one on the stream); the call's rows, sequences and positions come after it -- the
  // caller's last kernel may still be writing them -- and so does the cache state
  const float* mrow = T.mat + ((size_t)mh * kHeadDim + i) * kHeadDim;
  const float4* m4 = reinterpret_cast<const float4*>(mrow + 64 * half);
  float4 m[16];
#pragma unroll
  for (int j4 = 0; j4 < 16; ++j4) m[j4] = m4[j4];
  pdl_wait();
  load_chunk(c0);
  for (int c = c0; c < c1; ++c) {
    const int np = min(P.rt, pairs - c * P.rt);
    if (tid < np) dst_sh[tid] = rot_dst(P, T, d_row, d_head, d_b, d_p, true);
    if (xrow < np) {
      float4* xd = reinterpret_cast<float4*>(&xs[xrow][8 * xpart + (xpart >= 8 ? kXPad : 0)]);
      xd[0] = make_float4(__uint_as_float(xr.x << 16), __uint_as_float(xr.x & 0xffff0000u),
                          __uint_as_float(xr.y << 16), __uint_as_float(xr.y & 0xffff0000u));
      xd[1] = make_float4(__uint_as_float(xr.z << 16), __uint_as_float(xr.z & 0xffff0000u),
                          __uint_as_float(xr.w << 16), __uint_as_float(xr.w & 0xffff0000u));
    }
    if (tid == 0) n_fallback = 0;
    __syncthreads();
    if (kMulti && c + 1 < c1) load_chunk(c + 1);        // the next chunk's loads fly meanwhile
    for (int r = 0; r < np; ++r) {
      uint16_t* dst = dst_sh[r];
      if (dst == nullptr) continue;
      const float* x = xs[r] + (64 + kXPad) * half;
      // four independent FMA chains of 16 terms (float4 j4 feeds chain j4 % 4), each with its
      // running sum of |partial|; then two adds inside the thread and one with the partner
      float vc[4] = {0.f, 0.f, 0.f, 0.f}, ac[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j4 = 0; j4 < 16; ++j4) {
        const float4 xv = *reinterpret_cast<const float4*>(x + 4 * j4);
        float& v = vc[j4 & 3];
        float& a = ac[j4 & 3];
        v = fmaf(m[j4].x, xv.x, v); a += fabsf(v);
        v = fmaf(m[j4].y, xv.y, v); a += fabsf(v);
        v = fmaf(m[j4].z, xv.z, v); a += fabsf(v);
        v = fmaf(m[j4].w, xv.w, v); a += fabsf(v);
      }
      const float s01 = vc[0] + vc[1], s23 = vc[2] + vc[3];
      float v = s01 + s23;
      float a = ((ac[0] + ac[1]) + (ac[2] + ac[3])) + ((fabsf(s01) + fabsf(s23)) + fabsf(v));
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      a += __shfl_xor_sync(0xffffffffu, a, 1);
      if (half == 0) {
        const float e = fmaf(a + fabsf(v), 0x1.0001p-24f, 0x1p-140f);   // A includes the final v
        const int b = bf16_if_decided(v, e);
        if (b >= 0) dst[i] = (uint16_t)b;
        else fallback[atomicAdd(&n_fallback, 1)] = (uint16_t)((r << 7) | i);
      }
    }
    __syncthreads();
    // exact recomputation of the undecided outputs: one warp per output, 4 terms per lane
    for (int f = warp; f < n_fallback; f += (int)(blockDim.x >> 5)) {
      const int r = fallback[f] >> 7, o = fallback[f] & 127;
      const float4 t4 = reinterpret_cast<const float4*>(T.mat + ((size_t)mh * kHeadDim + o) * kHeadDim)[lane];
      const float4 x4 = reinterpret_cast<const float4*>(xs[r])[lane + (lane >= 16 ? kXPad / 4 : 0)];
      const uint32_t res = exact_dot_bf16_warp(t4, x4, lane);
      if (lane == 0) dst_sh[r][o] = (uint16_t)res;
    }
    __syncthreads();                                    // xs, dst_sh and the list are reused
  }
}

// Exact copies (identity transform): one warp per P.rpw consecutive (row, head) items, all of
// their loads in flight before the first store.  Lane k < rpw resolves item k's indices and
// destination (one division per warp, no per-lane repetition); the rows are then moved 8
// bytes per lane with the destination taken from lane k.
__device__ void warp_copies(const RotParams& P, int tt, int witem, int lane) {
  const RotTensor& T = P.t[tt];
  const int item0 = witem * P.rpw;
  const int n = min(P.rpw, T.rows * T.heads - item0);
  const int row0 = item0 / T.heads, h0 = item0 - row0 * T.heads;
  // item k = (row0 + (h0 + k) / heads, (h0 + k) % heads), k < rpw <= kMaxRPW <= heads or not
  int krow = row0, kh = h0 + (lane < n ? lane : 0);
  while (kh >= T.heads) {
    kh -= T.heads;
    ++krow;
  }
  pdl_wait();                           // the call's rows and positions: after the wait
  int kb = 0, kp = 0;
  if (lane < n && !T.is_query) {
    kb = P.seq_idx[krow];
    kp = P.pos[krow];
  }
  uint2 raw[kMaxRPW];
#pragma unroll
  for (int k = 0; k < kMaxRPW; ++k) {
    raw[k] = make_uint2(0u, 0u);
    if (k < n) {
      const int rk = __shfl_sync(0xffffffffu, krow, k), hk = __shfl_sync(0xffffffffu, kh, k);
      raw[k] = reinterpret_cast<const uint2*>(T.src + ((size_t)rk * T.heads + hk) * kHeadDim)[lane];
    }
  }
  uint16_t* dst = lane < n ? rot_dst(P, T, krow, kh, kb, kp, true) : nullptr;
#pragma unroll
  for (int k = 0; k < kMaxRPW; ++k) {
    if (k < n) {
      uint16_t* d = (uint16_t*)__shfl_sync(0xffffffffu, (unsigned long long)dst, k);
      if (d != nullptr) reinterpret_cast<uint2*>(d)[lane] = raw[k];
    }
  }
}

// One warp per (row, head): normalised Walsh-Hadamard transform.
__device__ void warp_item(const RotParams& P, int tt, int item, int lane) {
  const RotTensor& T = P.t[tt];
  int row = item / T.heads, h = item % T.heads;
  pdl_wait();                           // the call's rows and positions: after the wait
  int b = 0, p = 0;
  if (!T.is_query) {
    b = P.seq_idx[row];
    p = P.pos[row];
  }
  const uint16_t* src = T.src + ((size_t)row * T.heads + h) * kHeadDim;
  uint2 raw = *reinterpret_cast<const uint2*>(src + 4 * lane);
  uint16_t* dst = rot_dst(P, T, row, h, b, p, lane == 0);
  if (dst == nullptr) return;
  // S = H x.  Two ways, both ending in (hi, lo) with |S - (hi + lo)| <= bd (times the scale sc):
  // * every nonzero element a finite normal bf16 of exponent E >= 9 and the row spanning fewer
  //   than 32 binades: x_j = I_j 2^(emin - 134) with the integer I_j = +-M_j << (E_j - emin) (M the 8-bit
  //   significand), |I_j| < 2^39, so every partial sum of the butterflies is an integer below
  //   2^46 and exact in int64; then hi = RN(S), lo = S - hi exactly (at most 22 bits remain), bd
  //   = 0, and the scale sc = 2^(emin - 134) is applied after the product with 1/sqrt(128);
  // * otherwise double-float butterflies, each a sum or difference of two such values with its
  //   bound (ffb_add), at the row's own scale (sc = 1).
  float hi[4], lo[4], bd[4];
  hi[0] = __uint_as_float(raw.x << 16);
  hi[1] = __uint_as_float(raw.x & 0xffff0000u);
  hi[2] = __uint_as_float(raw.y << 16);
  hi[3] = __uint_as_float(raw.y & 0xffff0000u);
#pragma unroll
  for (int m = 0; m < 4; ++m) lo[m] = bd[m] = 0.f;
  uint32_t emax = 0u, emin = 255u;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t e = (__float_as_uint(hi[m]) >> 23) & 0xffu;
    if ((__float_as_uint(hi[m]) & 0x7fffffffu) != 0u) {
      emax = max(emax, max(e, 1u));
      emin = min(emin, max(e, 1u));
    }
  }
  emax = __reduce_max_sync(0xffffffffu, emax);
  emin = __reduce_min_sync(0xffffffffu, emin);
  const bool int_path = emax < emin + 32u && emin >= 9u && emax < 255u;   // (255: Inf / NaN)
  float sc = 1.0f;
  if (int_path) {
    long long I[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint32_t b16 = __float_as_uint(hi[m]) >> 16;
      const uint32_t E = (b16 >> 7) & 0xffu;
      const long long mag = (b16 & 0x7fffu) ? (long long)((b16 & 0x7fu) | 0x80u) << (E - emin) : 0LL;
      I[m] = (b16 & 0x8000u) ? -mag : mag;
    }
#pragma unroll
    for (int st = 1; st <= 2; st <<= 1) {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        if (m & st) continue;
        const long long u = I[m], v = I[m + st];
        I[m] = u + v;
        I[m + st] = u - v;
      }
    }
#pragma unroll
    for (int ls = 1; ls < 32; ls <<= 1) {
      const bool upper = (lane & ls) != 0;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const long long pv = __shfl_xor_sync(0xffffffffu, I[m], ls);
        I[m] = upper ? pv - I[m] : I[m] + pv;                 // a - b (b is mine) / a + b (a is mine)
      }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      hi[m] = __ll2float_rn(I[m]);
      lo[m] = __ll2float_rn(I[m] - __float2ll_rn(hi[m]));       // hi is an integer: exact
    }
    sc = __uint_as_float((emin - 7u) << 23);                  // 2^(emin - 134), a normal float
  } else {
  // in-thread stages: stride 1 then stride 2
#pragma unroll
  for (int st = 1; st <= 2; st <<= 1) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      if (m & st) continue;
      const float ah = hi[m], al = lo[m], ab = bd[m], bh = hi[m + st], bl = lo[m + st], bb = bd[m + st];
      ffb_add(ah, al, ab, bh, bl, bb, hi[m], lo[m], bd[m]);
      ffb_add(ah, al, ab, -bh, -bl, bb, hi[m + st], lo[m + st], bd[m + st]);
    }
  }
  // cross-lane stages: element stride 4 .. 64 = lane stride 1 .. 16
#pragma unroll
  for (int ls = 1; ls < 32; ls <<= 1) {
    const bool upper = (lane & ls) != 0;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float ph = __shfl_xor_sync(0xffffffffu, hi[m], ls);
      const float pl = __shfl_xor_sync(0xffffffffu, lo[m], ls);
      const float pb = __shfl_xor_sync(0xffffffffu, bd[m], ls);
      if (upper) ffb_add(ph, pl, pb, -hi[m], -lo[m], bd[m], hi[m], lo[m], bd[m]);   // a - b, b is mine
      else       ffb_add(hi[m], lo[m], bd[m], ph, pl, pb, hi[m], lo[m], bd[m]);     // a + b, a is mine
    }
  }
  }
  // y = S / sqrt(128) = S (ch + cl) + S eps, |eps| <= 2^-48 / sqrt(128): the product in
  // double-float with every rounding bounded, then the bf16 decision (exact.cuh); outputs it
  // leaves undecided are recomputed exactly from the row
  const double c = 0.088388347648318440550;  // 1/sqrt(128)
  const float ch = (float)c;
  const float cl = (float)(c - (double)ch);
  uint16_t o[4];
  uint32_t undecided = 0u;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const float p = __fmul_rn(hi[m], ch);
    const float e0 = __fmaf_rn(hi[m], ch, -p);
    const float e1 = __fmul_rn(hi[m], cl), e2 = __fmul_rn(lo[m], ch);
    const float e3 = __fadd_rn(e1, e2);
    const float e4 = __fadd_rn(e0, e3);
    float yh, yl;
    two_sum(p, e4, yh, yl);
    float by = bd[m] * 0.08838835f + (fabsf(hi[m]) + fabsf(lo[m])) * 0x1p-51f + fabsf(lo[m] * cl) +
               kU * (fabsf(e1) + fabsf(e2) + fabsf(e3) + fabsf(e4));
    // the row's scale (a power of two: exact unless the result is a float subnormal, whose
    // rounding the decision's absolute margin covers; beyond the float range it is infinite,
    // as is the bf16 result)
    yh *= sc;
    yl *= sc;
    by *= sc;
    int r;
    if (hi[m] == 0.f && lo[m] == 0.f && bd[m] == 0.f) r = 0;             // S exactly zero: +0
    else r = ffb_decide(yh, yl, by);
    if (r < 0) {
      undecided |= 1u << m;
      r = ff_to_bf16(yh, yl);                                           // the exact path's start
    }
    o[m] = (uint16_t)r;
  }
  // exact recomputation, one output at a time by its lane (rare: within the bound of a midpoint)
#pragma unroll 1
  for (int m = 0; m < 4; ++m)
    if (undecided & (1u << m)) o[m] = (uint16_t)exact_wht_output(src, 4 * lane + m, o[m]);
  uint2 outv;
  outv.x = (uint32_t)o[0] | ((uint32_t)o[1] << 16);
  outv.y = (uint32_t)o[2] | ((uint32_t)o[3] << 16);
  *reinterpret_cast<uint2*>(dst + 4 * lane) = outv;
}

// kMulti: dense tiles span several row chunks (prefill-sized calls); decode-sized calls use
// the single-chunk instantiation, whose smaller register footprint leaves room on the SMs for
// the next kernels of the step to start early.
// The parameter block is a grid constant: device functions take references to it and index
// its arrays at run time, reading the launch's parameter space directly (no per-CTA copy and no
// barrier before the first load).
template <bool kMulti>
__global__ void __launch_bounds__(256) rotate_kernel(const __grid_constant__ RotParams P) {
  pdl_trigger();
  int blk = blockIdx.x;
  // each path waits for the kernel before it itself (a dense tile after loading its matrix)
  if (blk < P.dense_total) {
    int tt, item;
    find_item(P.n_dense, blk, tt, item);
    dense_tile<kMulti>(P, tt, item);
    return;
  }
  int w = (blk - P.dense_total) * 8 + (threadIdx.x >> 5);
  if (w >= P.warp_total) {
    pdl_wait();
    return;
  }
  int tt, item;
  find_item(P.n_warp, w, tt, item);
  if (P.t[tt].mode == ROT_COPY) warp_copies(P, tt, item, threadIdx.x & 31);
  else warp_item(P, tt, item, threadIdx.x & 31);
}


// Warp items only (exact copies, Hadamard rows): the launch that accompanies the tensor-core
// kernel.  Without the dense path's register footprint it runs at full occupancy; the
// copies-only instantiation (kWht = false: no Walsh-Hadamard rows in the call) leaves out the
// Hadamard path's bounds and exact recomputation as well.
template <bool kWht>
__global__ void __launch_bounds__(256, kWht ? 4 : 6) rotate_items_kernel(const __grid_constant__ RotParams P) {
  pdl_trigger();
  const int w = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (w >= P.warp_total) {
    pdl_wait();
    return;
  }
  int tt, item;
  find_item(P.n_warp, w, tt, item);
  if (!kWht || P.t[tt].mode == ROT_COPY) warp_copies(P, tt, item, threadIdx.x & 31);
  else warp_item(P, tt, item, threadIdx.x & 31);
}

}  // namespace kvq

using namespace kvq;

extern "C" int kvq_launch_rotate(const kvq_config* cfg, const kvq_transform* tr, const uint16_t* q,
                                 uint16_t* q_out, int32_t n_q_rows, const uint16_t* k,
                                 const uint16_t* v, const int32_t* seq_idx, const int32_t* pos,
                                 int32_t n_kv_rows, const kvq_cache* cache, int32_t* d_status,
                                 cudaStream_t stream) {
  RotParams P{};
  int gqa = cfg->n_q_heads / cfg->n_kv_heads;
  bool had = tr->kind == KVQ_TRANSFORM_HADAMARD;
  // queries
  P.t[0] = RotTensor{q, n_q_rows, cfg->n_q_heads, had ? ROT_WHT : ROT_DENSE, tr->t_k_inv_t, gqa, 1,
                     q_out, nullptr, nullptr, 0, 0};
  // keys
  P.t[1] = RotTensor{k, n_kv_rows, cfg->n_kv_heads, had ? ROT_WHT : ROT_DENSE, tr->t_k, 1, 0,
                     nullptr, cache->sink_k, cache->ring_k, 1, 0};
  // values
  P.t[2] = RotTensor{v, n_kv_rows, cfg->n_kv_heads, tr->t_v ? ROT_DENSE : ROT_COPY, tr->t_v, 1, 0,
                     nullptr, cache->sink_v, cache->ring_v, 0, 1};
  P.seq_idx = seq_idx;
  P.pos = pos;
  P.seq_len = cache->seq_len;
  P.s_quant = cache->s_quant;
  P.s_sink = cfg->s_sink;
  P.ring_cap = cfg->ring_cap;
  P.batch = cfg->batch;
  P.hkv = cfg->n_kv_heads;
  P.status = d_status;
  long long dense_pairs = 0, copies = 0;
  for (int i = 0; i < 3; ++i) {
    if (P.t[i].mode == ROT_DENSE) dense_pairs += (long long)P.t[i].rows * P.t[i].heads;
    if (P.t[i].mode == ROT_COPY) copies += (long long)P.t[i].rows * P.t[i].heads;
  }
  // copies per warp: one while the copies fit two waves of 16 warps per SM, up to kMaxRPW
  const long long cslots = 2LL * kSms * 16;
  P.rpw = (int)(copies > cslots ? min((copies + cslots - 1) / cslots, (long long)kMaxRPW) : 1);
  for (int i = 0; i < 3; ++i) {
    const long long items = (long long)P.t[i].rows * P.t[i].heads;
    if (items > 0x3fffffffLL) return KVQ_ERR_UNSUPPORTED;
    P.n_warp[i] = P.t[i].mode == ROT_DENSE ? 0
                  : P.t[i].mode == ROT_COPY  ? (int)((items + P.rpw - 1) / P.rpw)
                                             : (int)items;
  }
  const long long warp_total = (long long)P.n_warp[0] + P.n_warp[1] + P.n_warp[2];
  if (warp_total > 0x3fffffffLL) return KVQ_ERR_UNSUPPORTED;
  P.warp_total = (int)warp_total;
  if (dense_pairs >= kTcMinPairs) {
    // prefill-sized: the warp items (copies, Hadamard rows) on their own, then every dense
    // tensor on the tensor cores
    if (P.warp_total > 0) {
      RotParams W = P;
      W.dense_total = 0;
      W.n_dense[0] = W.n_dense[1] = W.n_dense[2] = 0;
      W.rt = W.rpc = 1;
      const bool wht = P.t[0].mode == ROT_WHT || P.t[1].mode == ROT_WHT || P.t[2].mode == ROT_WHT;
      if (launch_pdl(wht ? rotate_items_kernel<true> : rotate_items_kernel<false>,
                     dim3((unsigned)((P.warp_total + 7) / 8)), dim3(256), 0, stream, W) != cudaSuccess)
        return KVQ_ERR_CUDA;
    }
    return launch_rotate_tc(P, stream);
  }
  // rows per tile: at most one tile per SM while that is enough (no SM runs two of a handful
  // of tiles), else about two tiles per SM
  const long long slots = dense_pairs <= 2 * kSms ? kSms : 2 * kSms;
  long long rt = (dense_pairs + slots - 1) / slots;
  P.rt = (int)(rt < 1 ? 1 : (rt > kMaxRT ? kMaxRT : rt));
  // chunks per tile: one for decode-sized calls; for larger ones enough that the grid is
  // about four waves of two tiles per SM, so each 64 KB matrix is read once per many rows
  long long chunks = 0;
  for (int i = 0; i < 3; ++i)
    if (P.t[i].mode == ROT_DENSE)
      chunks += (long long)(P.t[i].heads / P.t[i].head_div) *
                (((long long)P.t[i].rows * P.t[i].head_div + P.rt - 1) / P.rt);
  const long long target = 8LL * kSms;
  long long rpc = chunks > target ? (chunks + target - 1) / target : 1;
  P.rpc = (int)(rpc > (1 << 20) ? (1 << 20) : rpc);
  for (int i = 0; i < 3; ++i) {
    const int n_mats = P.t[i].heads / P.t[i].head_div;
    const long long pairs = (long long)P.t[i].rows * P.t[i].head_div;
    const long long tiles = (long long)n_mats * ((((pairs + P.rt - 1) / P.rt) + P.rpc - 1) / P.rpc);
    if (tiles > 0x3fffffffLL) return KVQ_ERR_UNSUPPORTED;
    P.n_dense[i] = P.t[i].mode == ROT_DENSE ? (int)tiles : 0;
  }
  P.dense_total = P.n_dense[0] + P.n_dense[1] + P.n_dense[2];
  long long blocks = (long long)P.dense_total + (P.warp_total + 7) / 8;
  if (blocks == 0) return KVQ_OK;
  if (blocks > 0x7fffffffLL) return KVQ_ERR_UNSUPPORTED;
  return launch_pdl(P.rpc > 1 ? rotate_kernel<true> : rotate_kernel<false>, dim3((unsigned)blocks), dim3(256), 0,
                    stream, P) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
