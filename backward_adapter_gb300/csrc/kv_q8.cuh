// Reading a q8_0-style K/V cache in place (llama.cpp PR #57, commit 2394a4c: a q8_0 cache trains
// in place; the backward admits a quantized source where it only casts a tile to F32). The cache
// holds, per (batch, key/value head, key), D signed 8-bit values and one fp16 scale per block of
// 32 consecutive features: x[d] = scale[d / 32] * q[d]. The tcgen05 kernels dequantize a 128-key
// tile straight into the bf16 128-byte-swizzled shared-memory layout their MMAs read (the layout
// TMA would have written for a bf16 tile): 64-feature boxes of 128 rows x 128 bytes, 16-byte
// chunk c of row r stored at chunk c ^ (r & 7). Keys at or past Sk are written as zeros.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "tc_ptx.cuh"

namespace fa {

// Byte k of w as a signed 8-bit value, in float, without an int-to-float conversion: the byte
// (offset by 128) becomes the low mantissa byte of 2^23, and the bias 2^23 + 128 is subtracted.
__device__ __forceinline__ float s8_to_f32(uint32_t w_offset, int k) {
  const uint32_t bits = __byte_perm(w_offset, 0x4B000000u, 0x7540u | (uint32_t)k);
  return __uint_as_float(bits) - 8388736.0f;
}

template <int D>
__device__ __forceinline__ void dequant_q8_tile(const int8_t* __restrict__ xq, const __half* __restrict__ xd,
                                                size_t row0, int key0, int Sk, uint8_t* tile, int r_begin, int r_end,
                                                int tid, int nthreads) {
  constexpr int SEG = D / 16;   // 16-feature segments per key row (one 16-byte load each)
  constexpr int BATCH = 8;      // loads in flight per thread before any is used
  const int items = (r_end - r_begin) * SEG;
  for (int base = tid; base < items; base += BATCH * nthreads) {
    int4 raw[BATCH];
    float scale[BATCH];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int it = base + u * nthreads;
      const int key = key0 + r_begin + it / SEG, sg = it % SEG;
      raw[u] = make_int4(0, 0, 0, 0);
      scale[u] = 0.f;
      if (it < items && key < Sk) {
        const size_t row = row0 + (size_t)key;
        raw[u] = __ldg(reinterpret_cast<const int4*>(xq + row * D + sg * 16));
        scale[u] = __half2float(xd[row * (D / 32) + sg / 2]);
      }
    }
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int it = base + u * nthreads;
      if (it >= items) break;
      const int r = r_begin + it / SEG, sg = it % SEG;
      const uint32_t uw[4] = {(uint32_t)raw[u].x ^ 0x80808080u, (uint32_t)raw[u].y ^ 0x80808080u,
                              (uint32_t)raw[u].z ^ 0x80808080u, (uint32_t)raw[u].w ^ 0x80808080u};
      uint32_t w[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t word = uw[k / 2];
        const int b0 = (k % 2) * 2;
        w[k] = tc::pack_bf16x2(s8_to_f32(word, b0) * scale[u], s8_to_f32(word, b0 + 1) * scale[u]);
      }
      const int c = sg * 16;                    // first feature of the segment
      const int ch = (c % 64) / 8;              // its first 16-byte chunk within the 64-feature box
      const uint32_t rowp = tc::smem_u32(tile + (c / 64) * (128 * 128) + r * 128);
      tc::st_shared_v4(rowp + ((ch ^ (r & 7)) * 16), w[0], w[1], w[2], w[3]);
      tc::st_shared_v4(rowp + (((ch + 1) ^ (r & 7)) * 16), w[4], w[5], w[6], w[7]);
    }
  }
}

}  // namespace fa
