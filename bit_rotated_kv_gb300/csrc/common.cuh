// Shared device helpers of the rotated INT2 KV-cache library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kHeadDim = 128;
constexpr int kPage = 16;
constexpr int kCodeBytes = 512;      // 16 tokens x 128 channels x 2 bits, per K or V
constexpr int kMaxGqa = 8;
constexpr int kSms = 152;          // SMs of one GB300 (two dies of 76): launch shapes aim at waves of it

// Bytes of one (page, kv head) chunk: K codes, V codes, K scales, V scales, [K norms],
// [per-channel keys: the exponent E of the largest key Delta], padded to 32 bytes.  Key
// scales: per token (16 tokens x d/G (Delta16, z16) pairs) or per channel (d Delta16, then
// d z16, each in the decode's B-fragment order).
__host__ __device__ inline int key_scale_bytes(int ng, int key_axis) {
  return key_axis ? 2 * kHeadDim * 2 : kPage * ng * 4;
}
__host__ __device__ inline int page_head_bytes(int group_size, int key_l2norm, int key_axis = 0) {
  int ng = kHeadDim / group_size;
  int b = 2 * kCodeBytes + key_scale_bytes(ng, key_axis) + kPage * ng * 4 + (key_l2norm ? kPage * 2 : 0) +
          (key_axis ? 4 : 0);
  return (b + 31) / 32 * 32;
}
__host__ __device__ inline int k_scale_off() { return 2 * kCodeBytes; }
// per-channel keys: Delta16 and z16 pairs, pair 16 q + 2 s + h = channels 16 s + 8 h + 2 q, + 1
__host__ __device__ inline int kc_delta_off() { return 2 * kCodeBytes; }
__host__ __device__ inline int kc_zero_off() { return 2 * kCodeBytes + kHeadDim * 2; }
__host__ __device__ inline int kc_pair_index(int channel) {     // channel even
  return 16 * ((channel & 7) >> 1) + 2 * (channel >> 4) + ((channel >> 3) & 1);
}
__host__ __device__ inline int v_scale_off(int ng, int key_axis = 0) {
  return 2 * kCodeBytes + key_scale_bytes(ng, key_axis);
}
__host__ __device__ inline int norm_off(int ng, int key_axis = 0) { return v_scale_off(ng, key_axis) + kPage * ng * 4; }
__host__ __device__ inline int kc_exp_off(int ng, int key_l2norm) { return norm_off(ng, 1) + (key_l2norm ? kPage * 2 : 0); }
// Value scales: Delta16 then z16, each laid out [token pair][group][2 tokens] (fp16), so one
// load gives the two tokens (2i, 2i+1) of every group.
__host__ __device__ inline int v_delta_off(int ng, int tp, int g, int key_axis = 0) {
  return v_scale_off(ng, key_axis) + (((tp >> 1) * ng + g) * 2 + (tp & 1)) * 2;
}
__host__ __device__ inline int v_zero_off(int ng, int tp, int g, int key_axis = 0) {
  return v_delta_off(ng, tp, g, key_axis) + kPage * ng * 2;
}

// First device fault wins; never traps.
__device__ __forceinline__ void set_status(int32_t* st, int code) {
  if (st) atomicCAS(st, 0, code);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) { return __uint_as_float(b16 << 16); }

// ---- error-free float arithmetic (no contraction: explicit _rn intrinsics) ----------
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  e = __fsub_rn(b, __fsub_rn(s, a));
}
// (hi, lo) += a * b, keeping the product's rounding error.
__device__ __forceinline__ void ff_mac(float& hi, float& lo, float a, float b) {
  float p = __fmul_rn(a, b);
  float pe = __fmaf_rn(a, b, -p);
  float s, e;
  two_sum(hi, p, s, e);
  hi = s;
  lo = __fadd_rn(lo, __fadd_rn(e, pe));
}
__device__ __forceinline__ void ff_add(float ah, float al, float bh, float bl, float& sh, float& sl) {
  float s, e;
  two_sum(ah, bh, s, e);
  e = __fadd_rn(e, __fadd_rn(al, bl));
  fast_two_sum(s, e, sh, sl);
}

// Round the double-float value hi + lo (|lo| <= ulp(hi)/2 after fast_two_sum) to bf16,
// nearest-even, deciding exact float32 ties by the sign of lo.
__device__ __forceinline__ uint16_t ff_to_bf16(float hi, float lo) {
  float h, l;
  fast_two_sum(hi, lo, h, l);
  uint32_t b = __float_as_uint(h);
  if ((b & 0x7f800000u) == 0x7f800000u) {                      // inf / nan
    return (uint16_t)((b >> 16) | ((b & 0x007fffffu) ? 0x40u : 0u));
  }
  uint32_t rem = b & 0xffffu;
  uint32_t up = b >> 16;
  if (rem > 0x8000u) {
    up += 1;
  } else if (rem == 0x8000u) {
    if (l != 0.0f) {
      if ((l > 0.0f) == (h > 0.0f)) up += 1;                     // beyond the midpoint
    } else {
      up += (up & 1u);                                           // exact tie: to even
    }
  }
  return (uint16_t)up;
}

// float64 -> float16, nearest-even, in one rounding: round to odd into float32 first
// (24 >= 11 + 2 bits keeps the final rounding correct), then float32 -> float16.
__device__ __forceinline__ __half double_to_half_rn(double d) {
  float f = __double2float_rz(d);
  if ((double)f != d && isfinite(d) && fabs(d) < 3.0e38) {
    uint32_t u = __float_as_uint(f) | 1u;
    f = __uint_as_float(u);
  }
  return __float2half_rn(f);
}

// Programmatic dependent launch: a kernel lets the next kernel of the stream start launching
// as soon as it begins (trigger), and waits for its predecessors' results (wait) before it
// reads anything they wrote.  Kernels that do not trigger simply complete first.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Ticket counter: atomic add with release (this CTA's prior writes, ordered before by a CTA
// barrier) and acquire (the writes released by earlier tickets) semantics at GPU scope.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int32_t* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Atomic add with release semantics only (orders this thread's earlier accesses before it;
// later ones are not held back, so the result can be consumed much later).
__device__ __forceinline__ int atomic_add_release_gpu(int32_t* p, int v) {
  int old;
  asm volatile("atom.add.release.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Warm L2 with [src, src + bytes) (16-byte aligned, multiple of 16) or with the line holding
// src: no data reaches the SM and nothing is ordered, so a kernel may issue these before its
// producer kernel has finished (before pdl_wait); the reads that count come after the wait.
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_l2_line(const void* src) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(src) : "memory");
}

template <typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace kvq
