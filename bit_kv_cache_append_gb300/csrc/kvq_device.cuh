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

// Rotate 8 RoPE pairs (channels c0..c0+7 with c0+D/2..) held as act-dtype
// bits, at table row `tab_row` ([D/2][2] cos, sin); results rounded back to
// the activation dtype (posttrainllm "StreamingLLM + KIVI", "RoPE caveat":
// keys keep the rotation of their absolute position).
__device__ __forceinline__ void rotate8(uint4& lo, uint4& hi, const float* tab_row, int c0, int bf16) {
  uint16_t* pl = reinterpret_cast<uint16_t*>(&lo);
  uint16_t* ph = reinterpret_cast<uint16_t*>(&hi);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float x = act_to_float(pl[i], bf16), y = act_to_float(ph[i], bf16);
    const float c = tab_row[2 * (c0 + i)], s = tab_row[2 * (c0 + i) + 1];
    float rx, ry;
    rope_pair(x, y, c, s, &rx, &ry);
    pl[i] = float_to_act(rx, bf16);
    ph[i] = float_to_act(ry, bf16);
  }
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
