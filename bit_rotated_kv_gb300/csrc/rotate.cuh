// Shared declarations of the kv_rotate_qk kernels: the per-call parameters, the destination of
// a transformed row, and the rounding decision from a bounded approximation.
#pragma once
#include "common.cuh"
#include "launch.h"
#include "exact.cuh"
#include "quant.cuh"

namespace kvq {

enum RotMode { ROT_DENSE = 0, ROT_WHT = 1, ROT_COPY = 2 };

struct RotTensor {
  const uint16_t* src;   // [rows][heads][d]
  int rows, heads;
  int mode;              // RotMode
  const float* mat;      // [mat_heads][d][d] for ROT_DENSE
  int head_div;          // matrix index = head / head_div
  int is_query;          // 1: write to q_out; 0: write into the cache
  uint16_t* dst_q;       // q_out
  uint16_t* sink;        // cache destination (keys or values)
  uint16_t* ring;
  int update_len;        // raise seq_len (keys only)
  int which;             // 0 keys, 1 values (quantizer constants of appended rows)
};

struct RotParams {
  RotTensor t[3];
  int rt;                // rows per chunk of a dense tile (rows that share one matrix)
  int rpc;               // chunks per dense tile (the matrix is loaded once per tile)
  int rpw;               // items per warp for exact copies
  int n_dense[3];        // dense tiles per tensor (0 when not dense)
  int n_warp[3];         // warp items per tensor (0 when dense)
  int dense_total, warp_total;
  const int32_t* seq_idx;
  const int32_t* pos;
  int32_t* seq_len;
  const int32_t* s_quant;
  int s_sink, ring_cap, batch, hkv;
  int32_t* status;
  // kv_append_chunk: the rows of sequence b are cu_rows[b] .. cu_rows[b+1] - 1, at positions
  // seq_len[b] - (cu_rows[b+1] - row) (seq_len and s_quant already advanced by the flush
  // step of the call); rows below s_quant[b] are quantized straight into their page.
  const int32_t* cu_rows;   // nullptr: kv_rotate_qk (rows placed by seq_idx / pos)
  uint8_t* pages;
  const int32_t* page_table;
  int max_pages, num_pages, page_bytes, ng, l2;
  QuantSpec qs[2];          // keys, values
};

// Sequence of appended row `row`: the b with cu_rows[b] <= row < cu_rows[b + 1] (-1 if none).
__device__ __forceinline__ int append_seq(const int32_t* cu_rows, int batch, int row) {
  if (row < __ldg(cu_rows) || row >= __ldg(cu_rows + batch)) return -1;
  int lo = 0, hi = batch - 1;            // cu_rows[lo] <= row < cu_rows[hi + 1]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu_rows + mid) <= row) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Destination kinds of an appended row.
constexpr int kDstNone = 0, kDstRow = 1, kDstPage = 2;

// Destination of appended row `row`, head h of tensor T (b = append_seq(row)): the BF16 sink
// or ring row (kDstRow), or the (page, kv head) chunk and token slot tp of its INT2 page
// (kDstPage).  Reads seq_len and s_quant: only after the flush step of the call.
__device__ __forceinline__ int append_dst(const RotParams& P, const RotTensor& T, int row, int h, int b,
                                          bool leader, void*& dst, int& tp) {
  dst = nullptr;
  tp = 0;
  if (b < 0) {
    if (leader) set_status(P.status, KVQ_ERR_BOUNDS);
    return kDstNone;
  }
  const int L = P.seq_len[b], sq = P.s_quant[b];
  const int p = L - (__ldg(P.cu_rows + b + 1) - row);
  if (p < 0 || sq < P.s_sink) {
    if (leader) set_status(P.status, KVQ_ERR_BOUNDS);
    return kDstNone;
  }
  if (p < P.s_sink) {
    dst = T.sink + (((size_t)b * P.hkv + h) * P.s_sink + p) * kHeadDim;
    return kDstRow;
  }
  if (p < sq) {
    const int lp = p - P.s_sink, pidx = lp >> 4;
    const int pid = pidx < P.max_pages ? P.page_table[(size_t)b * P.max_pages + pidx] : -1;
    if (pid < 0 || pid >= P.num_pages) {
      if (leader) set_status(P.status, KVQ_ERR_BOUNDS);
      return kDstNone;
    }
    dst = P.pages + ((size_t)pid * P.hkv + h) * P.page_bytes;
    tp = lp & (kPage - 1);
    return kDstPage;
  }
  if (p >= sq + P.ring_cap) {
    if (leader) set_status(P.status, KVQ_ERR_BOUNDS);
    return kDstNone;
  }
  dst = T.ring + (((size_t)b * P.hkv + h) * P.ring_cap + (p % P.ring_cap)) * kHeadDim;
  return kDstRow;
}

// Destination of row `row`, head `h` of tensor tt (b = seq_idx[row], p = pos[row] for cache
// rows, loaded by the caller; sq_loaded = s_quant[b] when the caller has loaded it, else -1);
// nullptr when the row is skipped.
__device__ __forceinline__ uint16_t* rot_dst(const RotParams& P, const RotTensor& T, int row, int h, int b,
                                             int p, bool leader, int sq_loaded = -1) {
  if (T.is_query) return T.dst_q + ((size_t)row * T.heads + h) * kHeadDim;
  if (b < 0 || b >= P.batch || p < 0) {
    if (leader) set_status(P.status, KVQ_ERR_BOUNDS);
    return nullptr;
  }
  uint16_t* dst;
  if (p < P.s_sink) {
    dst = T.sink + (((size_t)b * P.hkv + h) * P.s_sink + p) * kHeadDim;
  } else {
    const int sq = sq_loaded >= 0 ? sq_loaded : P.s_quant[b];   // s_quant[b], if already loaded
    if (p < sq || p >= sq + P.ring_cap) {
      if (leader) set_status(P.status, KVQ_ERR_BOUNDS);
      return nullptr;
    }
    dst = T.ring + (((size_t)b * P.hkv + h) * P.ring_cap + (p % P.ring_cap)) * kHeadDim;
  }
  if (leader && T.update_len && h == 0) atomicMax(P.seq_len + b, p + 1);
  return dst;
}

__device__ __forceinline__ void find_item(const int* counts, int idx, int& tt, int& item) {
  tt = 0;
  while (tt < 2 && idx >= counts[tt]) { idx -= counts[tt]; ++tt; }
  item = idx;
}

// (row, head) of the p-th pair that uses matrix mh: heads [mh * head_div, (mh + 1) * head_div)
// share it, so pairs run over rows x those heads.
__device__ __forceinline__ void tile_row(const RotTensor& T, int mh, int p, int& row, int& head) {
  row = p / T.head_div;
  head = mh * T.head_div + p % T.head_div;
}

// bf16 bits of the exact value y, decided from an fp32 value v with |v - y| <= e: the result
// when no bf16 rounding midpoint lies within e of v, else -1 (y must be computed exactly).
__device__ __forceinline__ int bf16_if_decided(float v, float e) {
  const uint32_t b = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v));
  const float bv = __uint_as_float(b << 16);
  const float lo = __uint_as_float(((b - 1u) & 0xffffu) << 16);   // adjacent bf16 values
  const float hi = __uint_as_float(((b + 1u) & 0xffffu) << 16);
  const float m1 = 0.5f * (bv + lo), m2 = 0.5f * (bv + hi);        // exact midpoints
  return (fabsf(v - m1) > e && fabsf(v - m2) > e) ? (int)b : -1;   // NaN compares false
}

// Exact recomputation of output o of a bf16 row x (128 values, 8-byte aligned, shared or
// global memory) against T row o (float32, global), over one warp (exact.cuh); lane 0
// stores the correctly rounded bf16 result to dst[o].
__device__ __forceinline__ void exact_output_warp(const float* trow, const uint16_t* xrow, uint16_t* dst, int o,
                                                  int lane) {
  const float4 t4 = reinterpret_cast<const float4*>(trow)[lane];
  const uint2 xr = reinterpret_cast<const uint2*>(xrow)[lane];
  const float4 x4 = make_float4(__uint_as_float(xr.x << 16), __uint_as_float(xr.x & 0xffff0000u),
                                __uint_as_float(xr.y << 16), __uint_as_float(xr.y & 0xffff0000u));
  const uint32_t r = exact_dot_bf16_warp(t4, x4, lane);
  if (lane == 0) dst[o] = (uint16_t)r;
}

// Dense (row, head) pairs from which a call runs its dense tensors on the tensor cores
// (rotate_tc.cu): about one 128-row block per SM.
constexpr long long kTcMinPairs = 128LL * kSms;

// Tiles of the dense tensors of P on the tensor cores: P.rpc, P.n_dense and P.dense_total.
int plan_rotate_tc(RotParams& P);

// Launch of the dense tensors of P on the tensor cores (P.n_dense and the tile sizes are set
// here; the warp items must already have been launched).
int launch_rotate_tc(RotParams P, cudaStream_t stream);



}  // namespace kvq
