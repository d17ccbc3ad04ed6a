// kda_device.cuh -- device helpers shared by the KDA kernels (sm_103a).
//
// The A0 "fold" of the gated delta rule lives here: L2 normalisation of q and
// k, the bounded gate g = lower_bound * sigmoid(exp(A_log[h]) * (a + dt_bias)),
// and beta = sigmoid(raw beta).  Flags and argument names follow chunk_kda in
// "PR #35197 report: fix(kernel) Fix Helion small-token prefill bug" (key
// source snippet of kda_prefill.py): use_qk_l2norm_in_kernel, A_log, dt_bias,
// lower_bound, and beta_is_raw from "[KDA] Support Helion MTP verification and
// harden prefill, decode" (sglang PR #42857, Modifications).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr int kHeadDim = 128;    // K == V == 128 in this build
constexpr float kNormEps = 1e-6f;

struct GateArgs {
  const float* A_log;    // [HV] or nullptr
  const float* dt_bias;  // [HV*K] or nullptr
  float lower_bound;
  int beta_is_raw;
  int use_qk_l2norm;
  float scale;
};

__device__ __forceinline__ float bf16_bits_to_float(uint16_t x) {
  return __uint_as_float(static_cast<uint32_t>(x) << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Token tensors (q, k, v, gate input, beta, packed rows) and the output o
// hold 16-bit elements: BF16 (F16 = false) or FP16 (F16 = true), per
// kda_dims.dtype.  Widening is exact; narrowing rounds to nearest even.
template <bool F16>
__device__ __forceinline__ float in16_to_float(uint16_t x) {
  if constexpr (F16)
    return __half2float(__ushort_as_half(x));
  else
    return bf16_bits_to_float(x);
}

template <bool F16>
__device__ __forceinline__ uint16_t float_to_out16(float x) {
  if constexpr (F16)
    return __half_as_ushort(__float2half_rn(x));
  else
    return float_to_bf16_bits(x);
}

// Four consecutive 16-bit elements (one 8-byte word) widened to float.
template <bool F16>
__device__ __forceinline__ float4 in16x4_to_f4(uint2 u) {
  if constexpr (F16) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
  } else {
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
  }
}

// Two floats narrowed to one 32-bit word of 16-bit output elements (lo first).
template <bool F16>
__device__ __forceinline__ uint32_t pack_out16x2(float lo, float hi) {
  return (uint32_t)float_to_out16<F16>(lo) | ((uint32_t)float_to_out16<F16>(hi) << 16);
}

__device__ __forceinline__ float sigmoidf_(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// exp(x) for decay factors.  Results below the smallest normal FP32 value
// (x < -87) are flushed to zero instead of being produced as denormals: such
// factors multiply O(1) terms into nothing, and the denormal results are slow.
__device__ __forceinline__ float decay_exp(float x) { return x < -87.0f ? 0.0f : __expf(x); }

// Log-decay of one channel from the gate input (bounded gate), or the input
// itself when A_log is absent.
__device__ __forceinline__ float gate_log_decay(const GateArgs& ga, float a_in, float exp_alog,
                                                float bias) {
  return ga.A_log ? ga.lower_bound * sigmoidf_(exp_alog * (a_in + bias)) : a_in;
}

__device__ __forceinline__ float fold_beta(const GateArgs& ga, float b_in) {
  return ga.beta_is_raw ? sigmoidf_(b_in) : b_in;
}

// Packed FP32 pair arithmetic (sm_100+ f32x2 instructions).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
        "l"(*reinterpret_cast<uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}

__device__ __forceinline__ void set_error(int32_t* err_flag, int bits) {
  if (err_flag) atomicOr(err_flag, bits);
}

// Asynchronous global -> shared copies (not through registers); the issuing
// thread waits for its own copies with cp_async_wait_all.  16-byte copies want
// both addresses 16-byte aligned, 4-byte copies 4-byte aligned.
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst_smem))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst_smem, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst_smem))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

}  // namespace kda
