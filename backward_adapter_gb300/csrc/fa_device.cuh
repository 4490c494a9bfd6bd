// Small device helpers shared by the kernels: element loads/stores and the
// per-pair visibility rule of the op.
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>
#include <stdint.h>

#include "fa_internal.h"

namespace fa {

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ void from_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void from_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Threshold at and below which an additive mask value hides a pair (the
// "mask floor" of the tiled backward in llama.cpp PR #57, commit 86c140d).
constexpr float kMaskFloor = -1e9f;

// Whether query row i may attend to key j, and the additive bias of the pair.
// Rows/keys outside [0, Sq) x [0, Sk) are invisible.
__device__ __forceinline__ bool pair_visible(const Shape& s, const void* mask, int b, int i, int j,
                                             float& bias) {
  bias = 0.f;
  if (i >= s.Sq || j >= s.Sk) return false;
  if (s.causal && (long long)j > s.q_offset + i) return false;
  if (s.window > 0 && llabs(s.q_offset + i - (long long)j) > s.window) return false;
  if (s.mask_kind != MK_NONE) {
    const size_t mb = (s.mask_batch > 1) ? (size_t)b : 0;
    const size_t idx = (mb * (size_t)s.Sq + (size_t)i) * (size_t)s.Sk + (size_t)j;
    if (s.mask_kind == MK_ADD) {
      const float m = static_cast<const float*>(mask)[idx];
      if (!(m > kMaskFloor)) return false;
      bias = m;
    } else {
      if (static_cast<const uint8_t*>(mask)[idx] == 0) return false;
    }
  }
  return true;
}

}  // namespace fa
