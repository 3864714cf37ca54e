// Device helpers shared by the library's kernels (internal).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "kvq_internal.h"

namespace kvq {

// 16-bit activation bits -> float (exact).
__device__ __forceinline__ float act_to_float(uint16_t bits, int bf16) {
  if (bf16) return __uint_as_float(static_cast<uint32_t>(bits) << 16);
  return __half2float(__ushort_as_half(bits));
}

// float -> 16-bit activation bits, round to nearest even.
__device__ __forceinline__ uint16_t float_to_act(float x, int bf16) {
  if (bf16) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  return __half_as_ushort(__float2half_rn(x));
}

// One RoPE pair rotation with every product and sum rounded on its own.
__device__ __forceinline__ void rope_pair(float a, float b, float c, float s, float* ra, float* rb) {
  *ra = __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, s));
  *rb = __fadd_rn(__fmul_rn(a, s), __fmul_rn(b, c));
}

__device__ __forceinline__ void set_error(int* flag, int code) {
  if (flag) atomicExch(flag, code);
}

// Value the device error flag takes when a bounded wait gives up (the
// public KV_ERR_TIMEOUT).
constexpr int kErrTimeout = 5;

// Bounded wait budget for spin loops: about one second of SM clock.
constexpr long long kWaitCycles = 1ll << 31;

}  // namespace kvq
