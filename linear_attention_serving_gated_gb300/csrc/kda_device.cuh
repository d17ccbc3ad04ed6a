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

// Four consecutive BF16 values (8-byte aligned) widened to float.
__device__ __forceinline__ float4 load_bf16x4(const kda_bf16* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  float4 r;
  r.x = __uint_as_float(u.x << 16);
  r.y = __uint_as_float(u.x & 0xffff0000u);
  r.z = __uint_as_float(u.y << 16);
  r.w = __uint_as_float(u.y & 0xffff0000u);
  return r;
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

}  // namespace kda
