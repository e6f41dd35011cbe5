/*
 * kvq.h -- C ABI of the rotated INT2 paged KV cache for GB300 (sm_103a).
 *
 * Three calls make up the serving hot path shared by the methods on these pages:
 *   [OSCAR] "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache
 *           Quantization" (paperlayer summary)
 *   [OScaR] "OScaR: The Occam's Razor for Extreme KV Cache Quantization in LLMs and
 *           Beyond" (reading note, in Chinese)
 *   [WUSH]  "WUSH-KV: KV Cache Quantization with Data-Adaptive Transforms" (digest)
 *
 *   kv_rotate_qk    fixed per-head transform of new keys/values on write and the
 *                   matching compensation of queries ([WUSH] core method and
 *                   inference algorithm; [OScaR] step 1 "Canalized Rotation";
 *                   [OSCAR] section 3 "Online Deployment").
 *   kv_quant_flush  quantize-on-write of the BF16 tokens that left the recent
 *                   window into INT2 pages ([WUSH] inference algorithm, S_flush
 *                   spans; [OSCAR] section 4 "KV Cache Update"; [OScaR] step 2
 *                   "Omni-Token Scaling" and the integer-quantization basics).
 *   kv_attn_decode  GQA decode attention reading the mixed BF16 / INT2 cache
 *                   directly ([OSCAR] section 4 "Decoding Attention Kernel";
 *                   [OScaR] "系统设计与 CUDA 实现"; [WUSH] GQA background).
 *   kv_attn_chunk   causal attention of a chunk's queries over the same cache
 *                   (the prefill path; [WUSH] inference algorithm).
 *   kv_append_chunk the first two fused for a prefill chunk: transform on write
 *                   and quantize-on-write in one pass, rows bound for INT2 never
 *                   written as BF16 ([OScaR] "系统设计与 CUDA 实现", key-quant
 *                   kernel; [OSCAR] section 4 "KV Cache Update").
 *
 * Conventions shared by every call
 *   - Every pointer inside a struct or argument is a DEVICE pointer unless said
 *     otherwise; the structs themselves live in host memory and are read during
 *     the call only.  The caller allocates, owns and frees every buffer; the
 *     library never allocates, frees, synchronizes, or keeps a pointer after it
 *     returns.
 *   - bf16 values are passed as uint16_t bit patterns; float16 scale data as
 *     uint16_t bit patterns.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).
 *   - Return value: KVQ_OK, or a negative KVQ_ERR_* code for a fault found on
 *     the host before anything is launched (bad argument, unsupported shape,
 *     CUDA launch error).
 *   - Faults found on the device (a page id or position out of range, a
 *     non-finite scale, a bounded wait that ran out) never trap: the offending
 *     unit of work is skipped and the first such code is stored into
 *     *d_status (a device int32 the caller zeroes and reads when it likes).
 *   - Overlap between consecutive calls: every kernel lets the next kernel of the
 *     stream begin early (programmatic dependent launch) and waits for the kernel
 *     before it -- the caller's or this library's -- to complete before it reads a
 *     per-call input (q, k, v, seq_idx, pos, cu_rows) or touches the cache state.
 *     Configuration is read before that wait: the transform matrices (kv_rotate_qk,
 *     kv_append_chunk) and the page table (kv_attn_decode, kv_attn_chunk).  These
 *     must not be written by the kernel launched immediately before the call on
 *     the same stream; a copy, or any earlier kernel, may write them.
 *
 * Supported shapes: head_dim 128; page_size 16; group_size 32, 64 or 128;
 * GQA ratio Hq/Hkv in {1, 2, 4, 8}; 2-bit codes.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__) || defined(__clang__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------------- */
#define KVQ_OK                 0
#define KVQ_ERR_INVALID_ARG   (-1)  /* null pointer, inconsistent sizes, bad enum          */
#define KVQ_ERR_UNSUPPORTED   (-2)  /* valid but not implemented (head_dim, G, GQA ratio)  */
#define KVQ_ERR_CUDA          (-3)  /* a CUDA runtime call or launch failed                */
#define KVQ_ERR_BOUNDS        (-4)  /* device: page id / position / ring slot out of range */
#define KVQ_ERR_NONFINITE     (-5)  /* device: a scale, zero point or norm is not finite   */
#define KVQ_ERR_TIMEOUT       (-6)  /* device: a bounded wait on an async copy ran out     */
#define KVQ_ERR_WORKSPACE     (-7)  /* workspace smaller than kv_attn_workspace_bytes()    */

/* ---- enums ----------------------------------------------------------------- */
#define KVQ_QUANT_AFFINE_KAPPA 0  /* kappa-quantile clipped asymmetric affine (OSCAR / WUSH) */
#define KVQ_QUANT_QUEST_RMS    1  /* QuEST RMS grid: Delta = 2 alpha rms / 3, z = 1.5 (WUSH) */

#define KVQ_KEY_PER_TOKEN      0  /* keys: Delta, z per token and group of G channels (OSCAR / WUSH) */
#define KVQ_KEY_PER_CHANNEL    1  /* keys: Delta, z per channel and 16-token page (KIVI, OScaR)     */

#define KVQ_TRANSFORM_DENSE    0  /* dense per-head float32 matrices T_K, T_K^{-T}, T_V       */
#define KVQ_TRANSFORM_HADAMARD 1  /* normalised Walsh-Hadamard on keys and queries (OScaR)    */

/* ---- configuration ----------------------------------------------------------
 * One POD struct, passed to every call (the pages' hyper-parameters plus shapes).
 * kappa: the quantile level of the clipping range, in [0.5, 1]; the group range
 * is [(1-kappa)-quantile, kappa-quantile] of the group's own values with linear
 * interpolation; kappa = 1 is min/max.  Windows: tokens [0, s_sink) stay BF16,
 * tokens [s_quant, L) are the BF16 recent window, [s_sink, s_quant) is INT2; the
 * flush rule quantizes [s_quant, s_quant + s_flush) while L - s_quant >= s_keep +
 * s_flush.  ring_cap: capacity of the BF16 recent ring in tokens (a multiple of
 * page_size; at least s_keep + s_flush + the most tokens appended between two
 * flushes).  attn_splits: INT2 splits per (sequence, kv head) in kv_attn_decode
 * (0 = automatic).  key_axis: KVQ_KEY_PER_TOKEN quantizes each key like each value,
 * per token and group of G channels; KVQ_KEY_PER_CHANNEL quantizes keys per channel
 * over the 16 tokens of a page -- KIVI's blocks along the token axis, the range of
 * channel j being the kappa-quantile range of its 16 values ([OScaR] "背景：KIVI 与逐通道
 * 量化范式" and algorithm, key processing) -- after the l2 scaling when key_l2norm;
 * it needs the AFFINE_KAPPA quantizer and s_flush a multiple of 16 (every flush then
 * quantizes whole pages; KVQ_ERR_UNSUPPORTED otherwise).  Values are per token either
 * way. */
typedef struct kvq_config {
  int32_t head_dim;          /* d  (128)                               */
  int32_t n_q_heads;         /* Hq                                     */
  int32_t n_kv_heads;        /* Hkv; query head hq reads kv head hq / (Hq/Hkv) */
  int32_t page_size;         /* P  (16 tokens per page)                */
  int32_t group_size;        /* G  (32, 64, 128 channels per group)    */
  int32_t quantizer;         /* KVQ_QUANT_*                            */
  int32_t key_l2norm;        /* 1: keys are l2-scaled after the transform, norm kept as float16 */
  int32_t s_sink;            /* BF16 sink tokens                       */
  int32_t s_keep;            /* BF16 recent tokens kept after a flush  */
  int32_t s_flush;           /* tokens quantized per flush span        */
  int32_t ring_cap;          /* BF16 recent ring capacity (tokens)     */
  int32_t batch;             /* B: sequences                           */
  int32_t max_pages_per_seq; /* columns of the page table              */
  int32_t num_pages;         /* physical pages in the pool             */
  int32_t attn_splits;       /* 0 = automatic                          */
  int32_t key_axis;          /* KVQ_KEY_PER_*                          */
  double  kappa_k;           /* key clipping quantile                  */
  double  kappa_v;           /* value clipping quantile                */
  double  quest_alpha;       /* QuEST clip in RMS units                */
} kvq_config;

/* ---- the cache ----------------------------------------------------------------
 * All device memory, owned by the caller.
 *
 * pages      [num_pages][Hkv][kvq_page_head_bytes(cfg)] bytes.  Logical INT2 page
 *            p of sequence b holds tokens [s_sink + 16p, s_sink + 16p + 16) and
 *            lives in physical page page_table[b * max_pages_per_seq + p].  One
 *            (page, kv head) chunk, tokens t = 0..15 of the page:
 *              [0, 512)      key codes in MMA-fragment order: u32 word 4*l + r
 *                            (l = 0..31, r = 0..3) holds token (l/4) + 8*(r%2);
 *                            its bits 2s and 16+2s (s = 0..7) hold the codes of
 *                            channels 16s + 2*(l%4) + 8*(r/2) + e, e = 0 / 1.
 *              [512, 1024)   value codes in MMA-fragment order: u32 word 4*l + r,
 *                            bits 2m + 16e (m = 0..7) hold the code of channel
 *                            16m + (l/4) + 8*(r%2) of token 2*(l%4) + 8*(r/2) + e.
 *              [1024, ...)   key scales: KVQ_KEY_PER_TOKEN: (Delta16, z16) float16
 *                            pairs [16 tokens][d/G] (64 d/G bytes); KVQ_KEY_PER_CHANNEL:
 *                            Delta16 [256 bytes] then z16 [256 bytes], each 64 u32
 *                            pairs, pair 16 q + 2 s + h holding channels
 *                            16 s + 8 h + 2 q and + 1 (the B-fragment order of the
 *                            decode's MMAs: q = 0..3, s = 0..7, h = 0..1); then
 *                            value Delta16 [8 token pairs][d/G][2] and value z16
 *                            [8 token pairs][d/G][2] (token t at pair t/2, slot t%2);
 *                            then (only when key_l2norm) key norms s16 float16 [16];
 *                            then (KVQ_KEY_PER_CHANNEL only) int32 E: the binary
 *                            exponent of the page's largest key Delta16 (at least -14);
 *                            the chunk is padded to a multiple of 32 bytes.
 *            Token t dequantizes as x_hat_c = s16 * Delta16 * (code_c - z16), with
 *            s16 = 1 without key_l2norm ([OScaR] step 2 dequantisation), Delta16 and
 *            z16 those of its group or, for per-channel keys, of channel c.
 * page_table [B][max_pages_per_seq] int32 physical page ids (-1 = none).
 * seq_len    [B] int32 tokens in each sequence; kv_rotate_qk raises it to
 *            pos + 1 for every row it writes.
 * s_quant    [B] int32 right edge of the INT2 region; must start at s_sink;
 *            kv_quant_flush advances it.
 * sink_k/v   [B][Hkv][s_sink][d] bf16 rows of tokens 0 .. s_sink-1.
 * ring_k/v   [B][Hkv][ring_cap][d] bf16; token t >= s_sink lives in slot t % ring_cap
 *            while it is in the recent window.
 * counters   [B] int32, zero before the first call; every call leaves it zero.
 */
typedef struct kvq_cache {
  void*          pages;
  const int32_t* page_table;
  int32_t*       seq_len;
  int32_t*       s_quant;
  uint16_t*      sink_k;
  uint16_t*      sink_v;
  uint16_t*      ring_k;
  uint16_t*      ring_v;
  int32_t*       counters;
} kvq_cache;

/* ---- the per-head transforms (device pointers, float32, row-major) -----------
 * DENSE:    k' = T_K k, q' = T_K^{-T} q (so q'^T k' = q^T k for any invertible
 *           T_K; for orthogonal T_K pass T_K itself), v' = T_V v (t_v NULL: values
 *           are stored unchanged, T_V folded into the projection weights).
 *           t_k, t_k_inv_t, t_v: [Hkv][d][d], element (i, j) at i*d + j.
 * HADAMARD: k' = H k, q' = H q with the normalised Walsh-Hadamard matrix (entries
 *           +-1/sqrt(d)); t_k and t_k_inv_t are ignored; t_v as for DENSE.
 * Every output row is the exact product rounded once to bf16 (nearest-even). */
typedef struct kvq_transform {
  int32_t      kind;         /* KVQ_TRANSFORM_* */
  int32_t      reserved;
  const float* t_k;
  const float* t_k_inv_t;
  const float* t_v;
} kvq_transform;

/* Bytes of one (page, kv head) chunk, and of one physical page (all kv heads). */
KVQ_API size_t kvq_page_head_bytes(const kvq_config* cfg);
KVQ_API size_t kvq_page_bytes(const kvq_config* cfg);

/* kv_rotate_qk: transform new rows on write, compensate queries on read.
 *   q        [n_q_rows][Hq][d] bf16 queries (may be NULL when n_q_rows == 0)
 *   q_out    [n_q_rows][Hq][d] bf16: q' (query head hq uses kv head hq/(Hq/Hkv))
 *   k, v     [n_kv_rows][Hkv][d] bf16 new keys / values (NULL when n_kv_rows == 0)
 *   seq_idx  [n_kv_rows] int32 sequence of each row; pos [n_kv_rows] int32 token
 *            position.  Row r goes to the sink (pos < s_sink) or to ring slot
 *            pos % ring_cap; pos must satisfy s_quant[b] <= pos < s_quant[b] +
 *            ring_cap for pos >= s_sink, otherwise the row is skipped with
 *            KVQ_ERR_BOUNDS in *d_status.  seq_len[b] is raised to pos + 1.
 * q, k, v and the matrices must be 16-byte aligned, q_out 8-byte aligned
 * (KVQ_ERR_INVALID_ARG otherwise).
 * Execution: one kernel for decode-sized calls.  From 19,456 dense (row, head) pairs on
 * (about one 128-row block per SM) the dense rows run on the tensor cores and the copies /
 * Hadamard rows in a second kernel launched first; the outputs are bit-identical either way
 * (see kvq_selftest_tc_integer_sums for the one hardware property that path relies on).
 * Source: [WUSH] inference algorithm (transform each new key and query, append at
 * full precision); [OScaR] algorithm, key and query processing (online FHT of K and Q). */
KVQ_API int kv_rotate_qk(const kvq_config* cfg, const kvq_transform* tr,
                 const uint16_t* q, uint16_t* q_out, int32_t n_q_rows,
                 const uint16_t* k, const uint16_t* v,
                 const int32_t* seq_idx, const int32_t* pos, int32_t n_kv_rows,
                 const kvq_cache* cache, int32_t* d_status, void* stream);

/* kv_quant_flush: apply the flush rule to every sequence: while seq_len - s_quant
 * >= s_keep + s_flush, quantize tokens [s_quant, s_quant + s_flush) of every kv
 * head from the BF16 ring into their INT2 page and advance s_quant.  At most
 * min(max_tokens_per_seq, ring_cap - s_keep) tokens (rounded down to whole
 * spans) are quantized per sequence by one call; the rest wait for the next call
 * (the ring never holds more than ring_cap - s_keep tokens past S_keep).  Per token (all float
 * operations IEEE round-to-nearest, none fused):
 *   key_l2norm (keys only): s = sqrt(sum x^2) in float64, s16 = fp16(s),
 *     y = x / s16 in float32 (y = 0 when s16 = 0);
 *   per group of G values, AFFINE_KAPPA: sorted a[], pos = (G-1)*kappa in float64,
 *     i = floor(pos), f = fp32(pos - i), hi = a[i] + f*(a[i+1] - a[i]) (a[G-1] when
 *     i = G-1), lo likewise at (G-1)*(1-kappa); Delta = (hi - lo)/3,
 *     Delta16 = fp16(Delta) (1 if it rounds to 0), z16 = fp16(-(lo / Delta16));
 *   QUEST_RMS: rms = sqrt(sum y^2 / G) in float64, Delta16 = fp16(2*alpha*rms/3)
 *     (1 if 0), z16 = 1.5 (not combined with key_l2norm);
 *   code = clamp(round_half_even(y / Delta16 + z16), 0, 3).
 * Source: [WUSH] inference algorithm (S_quant, S_flush-aligned spans, per-group
 * quantizer in place); [OSCAR] section 4 "KV Cache Update"; [OScaR] algorithm,
 * key processing (norm, residual buffer quantized when full) and the
 * integer-quantization formulas. */
KVQ_API int kv_quant_flush(const kvq_config* cfg, const kvq_cache* cache, int32_t max_tokens_per_seq,
                   int32_t* d_status, void* stream);

/* kv_append_chunk: append a chunk of new tokens to every sequence -- the effect of
 * kv_rotate_qk on those rows followed by kv_quant_flush, in one pass.
 *   k, v     [n_rows][Hkv][d] bf16 new keys / values (16-byte aligned; NULL when
 *            n_rows == 0)
 *   cu_rows  [B + 1] int32 (device): the rows of sequence b are cu_rows[b] ..
 *            cu_rows[b+1] - 1, in token order; cu_rows[0] = 0 and cu_rows[B] =
 *            n_rows (rows outside [cu_rows[0], cu_rows[B]) are skipped with
 *            KVQ_ERR_BOUNDS).  A sequence may append no rows.
 * Row r of sequence b gets position p = seq_len[b] + r - cu_rows[b]; seq_len[b]
 * then advances by cu_rows[b+1] - cu_rows[b], and the flush rule of
 * kv_quant_flush runs on the advanced length with no cap (s_quant advances by
 * whole S_flush spans while seq_len - s_quant >= s_keep + s_flush).  Keys are
 * transformed by T_K (DENSE only: KVQ_ERR_UNSUPPORTED for HADAMARD), values by T_V
 * or copied.  A row with p < s_sink goes to the sink, one below the new s_quant is
 * quantized straight into its INT2 page (as kv_quant_flush would), the others go
 * to their ring slot; tokens already in the ring that the new s_quant passes are
 * quantized from the ring.  Every byte written -- pages, sink and ring rows,
 * seq_len, s_quant -- equals what kv_rotate_qk at those positions followed by
 * kv_quant_flush (max_tokens_per_seq large enough) writes; the ring only has to
 * hold the tokens that stay in the window, not the whole chunk.
 * Execution: three kernels (flush of the ring tokens, copied rows, dense rows on
 * the tensor cores); meant for prefill-sized chunks (decode-sized appends are
 * cheaper through kv_rotate_qk + kv_quant_flush).
 * Source: [OScaR] "系统设计与 CUDA 实现" (key-quant kernel: transform, scaling and
 * INT2 packing on chip, input read once, codes written once); [OSCAR] section 4
 * "KV Cache Update" (fused prefill clip + quantize); [WUSH] inference algorithm. */
KVQ_API int kv_append_chunk(const kvq_config* cfg, const kvq_transform* tr,
                    const uint16_t* k, const uint16_t* v, const int32_t* cu_rows, int32_t n_rows,
                    const kvq_cache* cache, int32_t* d_status, void* stream);

/* kv_attn_chunk: attention of the queries of an appended chunk (the prefill path) over the
 * cache as it stands after the append.
 *   q_rot    [n_rows][Hq][d] bf16 compensated queries (kv_rotate_qk output), row r of
 *            sequence b for cu_rows[b] <= r < cu_rows[b+1] (the layout of kv_append_chunk)
 *   cu_rows  [B + 1] int32 (device): rows of sequence b; row r sits at position
 *            p = seq_len[b] - (cu_rows[b+1] - r), i.e. the rows are the last tokens of the
 *            sequence, in order (rows outside [cu_rows[0], cu_rows[B]) get KVQ_ERR_BOUNDS)
 *   out      [n_rows][Hq][d] float32
 * Row r attends causally to tokens [0, p] as the cache holds them: BF16 sink rows, INT2
 * tokens below min(s_quant, p + 1) dequantized, BF16 ring rows from s_quant to p -- the
 * result of kv_attn_decode for a sequence whose length were p + 1.  max_ctx bounds seq_len as
 * for kv_attn_decode; n_rows is at most 65535 (KVQ_ERR_UNSUPPORTED beyond); workspace of
 * kv_attn_chunk_workspace_bytes(cfg, n_rows, max_ctx) bytes, zero-filled before its first use
 * (every call leaves its ticket counters zero).
 * Execution: the decode kernel with one grid row per query row, so each query streams its own
 * prefix of the cache (L2 keeps a sequence's pages between the rows that share them).
 * Source: [WUSH] inference algorithm (mixed-precision attention over the S_sink / S_keep windows
 * and the INT2 middle); [OSCAR] section 4 "Decoding Attention Kernel" (BF16 and INT2 segments
 * of one attention). */
KVQ_API size_t kv_attn_chunk_workspace_bytes(const kvq_config* cfg, int32_t n_rows, int32_t max_ctx);
KVQ_API int kv_attn_chunk(const kvq_config* cfg, const kvq_cache* cache, const uint16_t* q_rot,
                  const int32_t* cu_rows, int32_t n_rows, float* out, float sm_scale, int32_t max_ctx,
                  void* workspace, size_t ws_bytes, int32_t* d_status, void* stream);

/* kv_attn_decode: one decode step of GQA attention for every sequence.
 *   q_rot   [B][Hq][d] bf16 compensated queries (kv_rotate_qk output)
 *   out     [B][Hq][d] float32 attention output (in the T_V space)
 *   sm_scale logit scale (1/sqrt(d) for standard attention)
 *   max_ctx  an upper bound of seq_len over the batch (sizes the split grid)
 *   workspace, ws_bytes: device scratch of at least kv_attn_workspace_bytes(cfg,
 *            max_ctx) bytes, zero-filled before its first use; every call leaves the
 *            ticket counters at its head zero again (the rest is overwritten).
 * Softmax over sink | INT2 | recent tokens with online (max, sum) merging across
 * splits in one launch; all g = Hq/Hkv query heads of a kv head share one read.
 * batch <= 65535 (KVQ_ERR_UNSUPPORTED otherwise: it is a grid dimension).
 * Source: [OSCAR] section 4 "Decoding Attention Kernel"; [OScaR] attention fused
 * kernel (in-register dequantisation, split attention); [WUSH] GQA. */
KVQ_API int kv_attn_decode(const kvq_config* cfg, const kvq_cache* cache, const uint16_t* q_rot,
                   float* out, float sm_scale, int32_t max_ctx,
                   void* workspace, size_t ws_bytes, int32_t* d_status, void* stream);

/* kv_attn_decode_bf16: kv_attn_decode with a bf16 output.
 *   out     [B][Hq][d] bf16 (8-byte aligned): the float32 result of kv_attn_decode rounded
 *           once to bf16 (nearest-even) -- the same kernel, only the final store differs.
 * Arguments, workspace and errors as kv_attn_decode.  For callers whose next GEMM (the
 * output projection, in the T_V space) takes bf16 activations; the rounding adds up to
 * 2^-9 relative per element on top of the float32 result.
 * Source: [OSCAR] section 4 "Decoding Attention Kernel" (decode attention over the mixed
 * cache); the output precision is not fixed by the pages. */
KVQ_API int kv_attn_decode_bf16(const kvq_config* cfg, const kvq_cache* cache, const uint16_t* q_rot,
                                uint16_t* out, float sm_scale, int32_t max_ctx,
                                void* workspace, size_t ws_bytes, int32_t* d_status, void* stream);

/* kv_attn_decode_noalloc: kv_attn_decode without a caller-supplied workspace, for callers
 * that cannot allocate device memory on this path -- for example a plugin running inside a
 * serving framework whose memory pool owns the whole device and forbids direct cudaMalloc,
 * or code that must not call cudaMalloc because it can synchronize the device.  This call
 * allocates nothing: its scratch is a fixed array of KVQ_NOALLOC_WORKSPACE_BYTES (8 MiB) of
 * device memory inside the library, held by every GPU that loads the library until the
 * process exits.  Arguments, results and errors are those of kv_attn_decode, except:
 *   - KVQ_ERR_WORKSPACE when kv_attn_workspace_bytes(cfg, max_ctx) exceeds the fixed size;
 *   - the first call on a device does a set-up, once per device, while that device is
 *     current: it looks up the array's device address and zero-fills the array (an async
 *     memset on `stream`), so make that first call before any stream capture; later calls
 *     add nothing to the stream but the decode kernel (each completed call leaves the ticket
 *     counters at the array's head zero again, as kv_attn_decode does for its workspace);
 *   - the address is kept for the life of the process: do not use this entry point after a
 *     cudaDeviceReset (or any other teardown of the device's primary context) in the same
 *     process, because the kept address no longer names device memory then;
 *   - every call shares the one array, which keeps the last call's contents; calls whose
 *     work overlaps on the GPU (other streams, other threads) race on it and give wrong
 *     results -- serialize them.
 * This entry point has no counterpart on the pages; it only changes where the scratch of
 * kv_attn_decode lives. */
#define KVQ_NOALLOC_WORKSPACE_BYTES (8u << 20)
KVQ_API int kv_attn_decode_noalloc(const kvq_config* cfg, const kvq_cache* cache, const uint16_t* q_rot,
                                   float* out, float sm_scale, int32_t max_ctx, int32_t* d_status, void* stream);

/* Workspace bytes kv_attn_decode needs for contexts up to max_ctx (host only). */
KVQ_API size_t kv_attn_workspace_bytes(const kvq_config* cfg, int32_t max_ctx);

/* Static description of a status code. */
KVQ_API const char* kvq_status_string(int code);

/* kvq_selftest_scale_division: the quantizer divides by a float16 scale with a
 * correctly rounded reciprocal and one exact-remainder correction instead of an IEEE
 * division.  This launches a check of that path against IEEE division on the device:
 * every finite bf16 dividend with every positive finite float16 scale, plus 2^29 hashed
 * float32 dividends (the l2-scaled keys); the number of bitwise differences is ADDED to
 * *d_mismatches (a device uint64 the caller zeroes).  Not part of the method on the pages:
 * a self-test of this implementation.  Returns KVQ_ERR_INVALID_ARG for a NULL pointer. */
KVQ_API int kvq_selftest_scale_division(unsigned long long* d_mismatches, void* stream);

/* kvq_selftest_tc_integer_sums: for prefill-sized calls kv_rotate_qk runs its dense rows on
 * the tensor cores with both operands written as integer digits in [-128, 128] (exact
 * bf16 values), so every accumulated sum is an integer below 2^23; the outputs are exact
 * as long as the tensor cores add such integers exactly, which the hardware documentation
 * does not state.  This launches a check of that on the device: hashed and extreme digit
 * matrices through the rotation's own sequence of MMAs, every accumulator compared with
 * the integer sum formed on the CUDA cores; the number of differences is ADDED to
 * *d_mismatches (a device uint64 the caller zeroes).  Not part of the method on the pages:
 * a self-test of this implementation.  Returns KVQ_ERR_INVALID_ARG for a NULL pointer. */
KVQ_API int kvq_selftest_tc_integer_sums(unsigned long long* d_mismatches, void* stream);

/* Library ABI version (major * 100 + minor). */
KVQ_API int kvq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
