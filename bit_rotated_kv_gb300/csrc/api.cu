// The C ABI: argument validation (host only, before any CUDA call) and dispatch to the
// kernels.  See include/kvq.h for the contract of every entry point.
#include "common.cuh"
#include "launch.h"

namespace {

using namespace kvq;

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

int check_config(const kvq_config* c) {
  if (!c) return KVQ_ERR_INVALID_ARG;
  if (c->head_dim != kHeadDim || c->page_size != kPage) return KVQ_ERR_UNSUPPORTED;
  if (c->group_size != 32 && c->group_size != 64 && c->group_size != 128) return KVQ_ERR_UNSUPPORTED;
  if (c->n_kv_heads < 1 || c->n_q_heads < 1 || c->n_q_heads % c->n_kv_heads) return KVQ_ERR_INVALID_ARG;
  const int g = c->n_q_heads / c->n_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return KVQ_ERR_UNSUPPORTED;
  if (c->quantizer != KVQ_QUANT_AFFINE_KAPPA && c->quantizer != KVQ_QUANT_QUEST_RMS) return KVQ_ERR_INVALID_ARG;
  if (c->quantizer == KVQ_QUANT_QUEST_RMS && c->key_l2norm) return KVQ_ERR_UNSUPPORTED;
  if (c->key_axis != KVQ_KEY_PER_TOKEN && c->key_axis != KVQ_KEY_PER_CHANNEL) return KVQ_ERR_INVALID_ARG;
  if (c->key_axis == KVQ_KEY_PER_CHANNEL && (c->quantizer != KVQ_QUANT_AFFINE_KAPPA || c->s_flush % kPage))
    return KVQ_ERR_UNSUPPORTED;
  if (c->key_l2norm != 0 && c->key_l2norm != 1) return KVQ_ERR_INVALID_ARG;
  if (!(c->kappa_k >= 0.5 && c->kappa_k <= 1.0) || !(c->kappa_v >= 0.5 && c->kappa_v <= 1.0))
    return KVQ_ERR_INVALID_ARG;
  if (c->quantizer == KVQ_QUANT_QUEST_RMS && !(c->quest_alpha > 0.0)) return KVQ_ERR_INVALID_ARG;
  if (c->s_sink < 0 || c->s_keep < 0 || c->s_flush < 1) return KVQ_ERR_INVALID_ARG;
  if (c->ring_cap < kPage || c->ring_cap % kPage || c->ring_cap < c->s_keep + c->s_flush)
    return KVQ_ERR_INVALID_ARG;
  if (c->batch < 1 || c->max_pages_per_seq < 1 || c->num_pages < 1 || c->attn_splits < 0)
    return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

int check_cache(const kvq_config* c, const kvq_cache* k) {
  if (!k || !k->pages || !k->page_table || !k->seq_len || !k->s_quant || !k->ring_k || !k->ring_v ||
      !k->counters)
    return KVQ_ERR_INVALID_ARG;
  if (c->s_sink > 0 && (!k->sink_k || !k->sink_v)) return KVQ_ERR_INVALID_ARG;
  if (!aligned(k->pages, 128) || !aligned(k->ring_k, 16) || !aligned(k->ring_v, 16)) return KVQ_ERR_INVALID_ARG;
  if (c->s_sink > 0 && (!aligned(k->sink_k, 16) || !aligned(k->sink_v, 16))) return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

}  // namespace

extern "C" {

KVQ_API int kvq_version(void) { return 100; }

KVQ_API int kvq_selftest_scale_division(unsigned long long* d_mismatches, void* stream) {
  if (!d_mismatches) return KVQ_ERR_INVALID_ARG;
  return kvq_launch_div_selftest(d_mismatches, (cudaStream_t)stream);
}

KVQ_API int kvq_selftest_tc_integer_sums(unsigned long long* d_mismatches, void* stream) {
  if (!d_mismatches) return KVQ_ERR_INVALID_ARG;
  return kvq_launch_tc_selftest(d_mismatches, (cudaStream_t)stream);
}

KVQ_API const char* kvq_status_string(int code) {
  switch (code) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported shape or option";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_BOUNDS: return "page id, position or ring slot out of range (device)";
    case KVQ_ERR_NONFINITE: return "non-finite scale, zero point or norm (device)";
    case KVQ_ERR_TIMEOUT: return "bounded wait on an asynchronous copy ran out (device)";
    case KVQ_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

KVQ_API size_t kvq_page_head_bytes(const kvq_config* cfg) {
  if (check_config(cfg) != KVQ_OK) return 0;
  return (size_t)page_head_bytes(cfg->group_size, cfg->key_l2norm, cfg->key_axis);
}

KVQ_API size_t kvq_page_bytes(const kvq_config* cfg) {
  if (check_config(cfg) != KVQ_OK) return 0;
  return (size_t)page_head_bytes(cfg->group_size, cfg->key_l2norm, cfg->key_axis) * cfg->n_kv_heads;
}

KVQ_API size_t kv_attn_workspace_bytes(const kvq_config* cfg, int32_t max_ctx) {
  if (check_config(cfg) != KVQ_OK || max_ctx < 0) return 0;
  return kvq_attn_ws_bytes(cfg, max_ctx);
}

KVQ_API int kv_rotate_qk(const kvq_config* cfg, const kvq_transform* tr, const uint16_t* q, uint16_t* q_out,
                         int32_t n_q_rows, const uint16_t* k, const uint16_t* v, const int32_t* seq_idx,
                         const int32_t* pos, int32_t n_kv_rows, const kvq_cache* cache, int32_t* d_status,
                         void* stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!tr || (tr->kind != KVQ_TRANSFORM_DENSE && tr->kind != KVQ_TRANSFORM_HADAMARD)) return KVQ_ERR_INVALID_ARG;
  if (n_q_rows < 0 || n_kv_rows < 0) return KVQ_ERR_INVALID_ARG;
  if (n_q_rows > 0) {
    if (!q || !q_out || !aligned(q, 16) || !aligned(q_out, 8)) return KVQ_ERR_INVALID_ARG;
    if (tr->kind == KVQ_TRANSFORM_DENSE && (!tr->t_k_inv_t || !aligned(tr->t_k_inv_t, 16)))
      return KVQ_ERR_INVALID_ARG;
  }
  if (n_kv_rows > 0) {
    rc = check_cache(cfg, cache);
    if (rc) return rc;
    if (!k || !v || !seq_idx || !pos || !aligned(k, 16) || !aligned(v, 16)) return KVQ_ERR_INVALID_ARG;
    if (tr->kind == KVQ_TRANSFORM_DENSE && (!tr->t_k || !aligned(tr->t_k, 16))) return KVQ_ERR_INVALID_ARG;
    if (tr->t_v && !aligned(tr->t_v, 16)) return KVQ_ERR_INVALID_ARG;
  }
  if (n_q_rows == 0 && n_kv_rows == 0) return KVQ_OK;
  kvq_cache empty{};
  return kvq_launch_rotate(cfg, tr, q, q_out, n_q_rows, k, v, seq_idx, pos, n_kv_rows,
                           n_kv_rows > 0 ? cache : &empty, d_status, (cudaStream_t)stream);
}

KVQ_API int kv_quant_flush(const kvq_config* cfg, const kvq_cache* cache, int32_t max_tokens_per_seq,
                           int32_t* d_status, void* stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  rc = check_cache(cfg, cache);
  if (rc) return rc;
  if (max_tokens_per_seq < 0) return KVQ_ERR_INVALID_ARG;
  return kvq_launch_flush(cfg, cache, max_tokens_per_seq, d_status, (cudaStream_t)stream);
}

KVQ_API int kv_append_chunk(const kvq_config* cfg, const kvq_transform* tr, const uint16_t* k, const uint16_t* v,
                            const int32_t* cu_rows, int32_t n_rows, const kvq_cache* cache, int32_t* d_status,
                            void* stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  rc = check_cache(cfg, cache);
  if (rc) return rc;
  if (!tr || (tr->kind != KVQ_TRANSFORM_DENSE && tr->kind != KVQ_TRANSFORM_HADAMARD)) return KVQ_ERR_INVALID_ARG;
  if (tr->kind == KVQ_TRANSFORM_HADAMARD || cfg->key_axis != KVQ_KEY_PER_TOKEN) return KVQ_ERR_UNSUPPORTED;
  if (n_rows < 0 || !cu_rows || !aligned(cu_rows, 4)) return KVQ_ERR_INVALID_ARG;
  if (n_rows > 0) {
    if (!k || !v || !aligned(k, 16) || !aligned(v, 16)) return KVQ_ERR_INVALID_ARG;
    if (!tr->t_k || !aligned(tr->t_k, 16)) return KVQ_ERR_INVALID_ARG;
    if (tr->t_v && !aligned(tr->t_v, 16)) return KVQ_ERR_INVALID_ARG;
  }
  return kvq_launch_append(cfg, tr, k, v, cu_rows, n_rows, cache, d_status, (cudaStream_t)stream);
}

KVQ_API int kv_attn_decode(const kvq_config* cfg, const kvq_cache* cache, const uint16_t* q_rot, float* out,
                           float sm_scale, int32_t max_ctx, void* workspace, size_t ws_bytes, int32_t* d_status,
                           void* stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  rc = check_cache(cfg, cache);
  if (rc) return rc;
  if (!q_rot || !out || !aligned(q_rot, 16) || !aligned(out, 16) || max_ctx < 0) return KVQ_ERR_INVALID_ARG;
  if (!(sm_scale == sm_scale)) return KVQ_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return KVQ_ERR_INVALID_ARG;
  if (ws_bytes < kvq_attn_ws_bytes(cfg, max_ctx)) return KVQ_ERR_WORKSPACE;
  return kvq_launch_attn(cfg, cache, q_rot, out, 0, sm_scale, max_ctx, workspace, d_status, (cudaStream_t)stream);
}

KVQ_API int kv_attn_decode_bf16(const kvq_config* cfg, const kvq_cache* cache, const uint16_t* q_rot, uint16_t* out,
                                float sm_scale, int32_t max_ctx, void* workspace, size_t ws_bytes, int32_t* d_status,
                                void* stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  rc = check_cache(cfg, cache);
  if (rc) return rc;
  if (!q_rot || !out || !aligned(q_rot, 16) || !aligned(out, 8) || max_ctx < 0) return KVQ_ERR_INVALID_ARG;
  if (!(sm_scale == sm_scale)) return KVQ_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return KVQ_ERR_INVALID_ARG;
  if (ws_bytes < kvq_attn_ws_bytes(cfg, max_ctx)) return KVQ_ERR_WORKSPACE;
  return kvq_launch_attn(cfg, cache, q_rot, out, 1, sm_scale, max_ctx, workspace, d_status, (cudaStream_t)stream);
}

KVQ_API size_t kv_attn_chunk_workspace_bytes(const kvq_config* cfg, int32_t n_rows, int32_t max_ctx) {
  if (check_config(cfg) != KVQ_OK || max_ctx < 0 || n_rows < 0 || n_rows > 65535) return 0;
  return kvq_attn_chunk_ws_bytes(cfg, n_rows, max_ctx);
}

KVQ_API int kv_attn_chunk(const kvq_config* cfg, const kvq_cache* cache, const uint16_t* q_rot, const int32_t* cu_rows,
                          int32_t n_rows, float* out, float sm_scale, int32_t max_ctx, void* workspace, size_t ws_bytes,
                          int32_t* d_status, void* stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  rc = check_cache(cfg, cache);
  if (rc) return rc;
  if (n_rows < 0 || max_ctx < 0 || !cu_rows || !aligned(cu_rows, 4)) return KVQ_ERR_INVALID_ARG;
  if (n_rows > 65535) return KVQ_ERR_UNSUPPORTED;                  // one grid row per query row
  if (n_rows == 0) return KVQ_OK;
  if (!q_rot || !out || !aligned(q_rot, 16) || !aligned(out, 16)) return KVQ_ERR_INVALID_ARG;
  if (!(sm_scale == sm_scale)) return KVQ_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return KVQ_ERR_INVALID_ARG;
  if (ws_bytes < kvq_attn_chunk_ws_bytes(cfg, n_rows, max_ctx)) return KVQ_ERR_WORKSPACE;
  return kvq_launch_attn_chunk(cfg, cache, q_rot, cu_rows, n_rows, out, sm_scale, max_ctx, workspace, d_status,
                               (cudaStream_t)stream);
}

KVQ_API int kv_attn_decode_noalloc(const kvq_config* cfg, const kvq_cache* cache, const uint16_t* q_rot,
                                   float* out, float sm_scale, int32_t max_ctx, int32_t* d_status, void* stream) {
  int rc = check_config(cfg);
  if (rc) return rc;
  rc = check_cache(cfg, cache);
  if (rc) return rc;
  if (!q_rot || !out || !aligned(q_rot, 16) || !aligned(out, 16) || max_ctx < 0) return KVQ_ERR_INVALID_ARG;
  if (!(sm_scale == sm_scale)) return KVQ_ERR_INVALID_ARG;
  return kvq_launch_attn_noalloc(cfg, cache, q_rot, out, sm_scale, max_ctx, d_status, (cudaStream_t)stream);
}

}  // extern "C"
