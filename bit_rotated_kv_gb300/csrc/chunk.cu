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
//   3. the dense transforms on the tensor cores; the decided rows of each 64-row chunk are
//      staged in shared memory, then copied to their window row or quantized into their page
//      by the same octet quantizer (rotate_tc.cu).
#include "rotate.cuh"

#include <algorithm>

namespace kvq {
namespace {

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

int launch_append_copy(const RotParams& P, cudaStream_t stream) {
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
  P.page_bytes = page_head_bytes(cfg->group_size, cfg->key_l2norm);
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
  return launch_rotate_tc(P, stream);
}
