// Internal launchers shared between the translation units of the library (not exported).
#pragma once

#include <cuda_runtime.h>
#include "../../include/kvq.h"

extern "C" {
int kvq_launch_rotate(const kvq_config* cfg, const kvq_transform* tr, const uint16_t* q, uint16_t* q_out,
                      int32_t n_q_rows, const uint16_t* k, const uint16_t* v, const int32_t* seq_idx,
                      const int32_t* pos, int32_t n_kv_rows, const kvq_cache* cache, int32_t* d_status,
                      cudaStream_t stream);
int kvq_launch_flush(const kvq_config* cfg, const kvq_cache* cache, int32_t max_tokens, int32_t* d_status,
                     cudaStream_t stream);
int kvq_launch_flush_append(const kvq_config* cfg, const kvq_cache* cache, const int32_t* cu_rows,
                            int32_t* d_status, cudaStream_t stream);
int kvq_launch_append(const kvq_config* cfg, const kvq_transform* tr, const uint16_t* k, const uint16_t* v,
                      const int32_t* cu_rows, int32_t n_rows, const kvq_cache* cache, int32_t* d_status,
                      cudaStream_t stream);
int kvq_launch_attn(const kvq_config* cfg, const kvq_cache* cache, const uint16_t* q_rot, void* out, int out_bf16,
                    float sm_scale, int32_t max_ctx, void* ws, int32_t* d_status, cudaStream_t stream);
int kvq_launch_attn_chunk(const kvq_config* cfg, const kvq_cache* cache, const uint16_t* q_rot, const int32_t* cu_rows,
                          int32_t n_rows, float* out, float sm_scale, int32_t max_ctx, void* ws, int32_t* d_status,
                          cudaStream_t stream);
size_t kvq_attn_chunk_ws_bytes(const kvq_config* cfg, int32_t n_rows, int32_t max_ctx);
int kvq_launch_attn_noalloc(const kvq_config* cfg, const kvq_cache* cache, const uint16_t* q_rot, float* out,
                            float sm_scale, int32_t max_ctx, int32_t* d_status, cudaStream_t stream);
int kvq_launch_div_selftest(unsigned long long* d_mismatches, cudaStream_t stream);
int kvq_launch_tc_selftest(unsigned long long* d_mismatches, cudaStream_t stream);
size_t kvq_attn_counter_bytes(const kvq_config* cfg, int32_t max_ctx);
size_t kvq_attn_ws_bytes(const kvq_config* cfg, int32_t max_ctx);
void kvq_attn_splits(const kvq_config* cfg, int32_t max_ctx, int* n_int2, int* n_win);
}
