// HBM-bound helper passes of the fused attention training op:
//   * D precompute: D_i = <dO_i, O_i> in fp32, fused with zeroing the fp32 dQ
//     accumulator (llama.cpp PR #57, commit 86c140d: the tiled backward forms
//     LSE and D before the per-tile gradients);
//   * dQ convert: dQ = scale * dQ_acc, rounded to the output type;
//   * mask tile classification: one byte per 128x128 tile saying whether the
//     tile is fully hidden (skipped), fully open with zero bias (no mask reads
//     in the hot loop) or mixed.
// Each thread moves 16-byte vectors; rows are split across 8..16 lanes. The file also holds
// the self-test of the kernels' bounded waits.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "fa_device.cuh"
#include "fa_internal.h"
#include "kv_q8.cuh"
#include "tc_ptx.cuh"

namespace fa {
namespace {

// 8 consecutive elements as fp32, from a 16-byte (bf16) or 32-byte (fp32) vector.
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* x) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 f = __bfloat1622float2(h[t]);
    x[2 * t] = f.x;
    x[2 * t + 1] = f.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float* x) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float* x) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int t = 0; t < 4; ++t) h[t] = __floats2bfloat162_rn(x[2 * t], x[2 * t + 1]);
  *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void store8(float* p, const float* x) {
  reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}

template <typename T, int D>
__global__ void __launch_bounds__(256) dsum_kernel(const T* __restrict__ o, const T* __restrict__ dO,
                                                   float* __restrict__ dsum, float* __restrict__ dq_acc,
                                                   long long rows, int groups, uint32_t* __restrict__ zero_words,
                                                   int n_zero, const Shape s) {
  constexpr int LPR = D / 8;  // lanes per row
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (tid < n_zero) zero_words[tid] = 0u;
  const long long row = tid / LPR;   // over [B, Hq, Sq], like D and the dQ accumulators
  const int part = (int)(tid % LPR);
  float acc = 0.f;
  if (row < rows) {
    size_t at = (size_t)row * D;   // [B, Hq, Sq, D]: the row's offset directly
    if (s.layout) {
      const long long bh = row / s.Sq, i = row % s.Sq;
      at = head_base(s, (int)(bh / s.Hq), (int)(bh % s.Hq), s.Hq, s.Sq) + (size_t)i * row_stride(s, s.Hq);
    }
    float a[8], g[8];
    load8(o + at + part * 8, a);
    load8(dO + at + part * 8, g);
#pragma unroll
    for (int t = 0; t < 8; ++t) acc = fmaf(a[t], g[t], acc);
    if (dq_acc != nullptr) {
      const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int gi = 0; gi < groups; ++gi) store8(dq_acc + ((long long)gi * rows + row) * D + part * 8, z);
    }
  }
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && part == 0) dsum[row] = acc;
}

// Each thread converts kConvVecs 8-element vectors, a grid stride apart, with all of their loads
// issued before the first store (more bytes in flight per thread).
constexpr int kConvVecs = 4;

template <typename T>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc, T* __restrict__ dq,
                                                         float scale, long long vecs, int groups, const Shape s) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  float x[kConvVecs][8];
#pragma unroll
  for (int u = 0; u < kConvVecs; ++u) {
    const long long i = i0 + u * stride;
    if (i < vecs) load8(acc + i * 8, x[u]);
  }
#pragma unroll
  for (int u = 0; u < kConvVecs; ++u) {
    const long long i = i0 + u * stride;
    if (i >= vecs) break;
    for (int g = 1; g < groups; ++g) {   // the key-tile groups' accumulators, always in group order
      float y[8];
      load8(acc + ((long long)g * vecs + i) * 8, y);
#pragma unroll
      for (int t = 0; t < 8; ++t) x[u][t] += y[t];
    }
    const long long e = i * 8;   // element of the accumulator, [B, Hq, Sq, D]
    size_t at = (size_t)e;        // the same element of dQ when dQ is [B, Hq, Sq, D] too
    if (s.layout) {
      const long long row = e / s.D, bh = row / s.Sq, qi = row % s.Sq;
      at = head_base(s, (int)(bh / s.Hq), (int)(bh % s.Hq), s.Hq, s.Sq) + (size_t)qi * row_stride(s, s.Hq) +
           (size_t)(e % s.D);
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) x[u][t] *= scale;
    store8(dq + at, x[u]);
  }
}

// One block per (mask batch, q-tile, k-tile) of 128 x 128, flattened in that order.
// One block per 128 x 128 tile. With vec (every row of the mask starts on a 16-byte boundary:
// Sk % 4 == 0 for fp32, Sk % 16 == 0 for bytes) each thread reads 16-byte vectors, all of its loads
// independent (a tile is 64 KB of fp32: latency, not bandwidth, sets the time); otherwise one
// element at a time.
template <bool ADD, bool VEC>
__global__ void __launch_bounds__(512) mask_classify_kernel(Shape s, const void* __restrict__ mask,
                                                            uint8_t* __restrict__ tilemap, int nqt, int nkt) {
  const long long tile = blockIdx.x;
  const int kt = (int)(tile % nkt);
  const int qt = (int)((tile / nkt) % nqt);
  const int mb = (int)(tile / ((long long)nkt * nqt));
  bool any_vis = false, all_open = true;
  const int i0 = qt * 128, j0 = kt * 128;
  constexpr int EPV = ADD ? 4 : 16;             // elements per 16-byte vector
  constexpr int VPR = 128 / EPV;                // vectors per tile row
  constexpr int PER_THREAD = 128 * VPR / 512;   // 8 (fp32) or 2 (bytes)
  if (VEC) {
#pragma unroll
    for (int t = 0; t < PER_THREAD; ++t) {
      const int v = t * 512 + (int)threadIdx.x;
      const int i = i0 + v / VPR, j = j0 + (v % VPR) * EPV;
      if (i >= s.Sq || j >= s.Sk) continue;   // rows and tails past the mask (Sk is a multiple of EPV)
      const size_t idx = ((size_t)mb * s.Sq + i) * s.Sk + j;
      if (ADD) {
        const float4 m = *reinterpret_cast<const float4*>(static_cast<const float*>(mask) + idx);
        any_vis |= (m.x > kMaskFloor) | (m.y > kMaskFloor) | (m.z > kMaskFloor) | (m.w > kMaskFloor);
        all_open &= (m.x == 0.f) & (m.y == 0.f) & (m.z == 0.f) & (m.w == 0.f);
      } else {
        const uint4 m = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(mask) + idx);
        const uint32_t w[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          // a byte is visible when nonzero: some byte of w is visible iff w != 0, and
          // (w - 0x01010101) & ~w & 0x80808080 is nonzero iff some byte of w is zero
          any_vis |= w[u] != 0u;
          all_open &= ((w[u] - 0x01010101u) & ~w[u] & 0x80808080u) == 0u;
        }
      }
    }
  } else {
    for (int e = threadIdx.x; e < 128 * 128; e += 512) {
      const int i = i0 + e / 128, j = j0 + e % 128;
      if (i >= s.Sq || j >= s.Sk) continue;
      const size_t idx = ((size_t)mb * s.Sq + i) * s.Sk + j;
      if (ADD) {
        const float m = static_cast<const float*>(mask)[idx];
        any_vis |= m > kMaskFloor;
        all_open &= (m == 0.f);
      } else {
        const bool vis = static_cast<const uint8_t*>(mask)[idx] != 0;
        any_vis |= vis;
        all_open &= vis;
      }
    }
  }
  any_vis = __syncthreads_or(any_vis);
  all_open = __syncthreads_and(all_open);
  if (threadIdx.x == 0)
    tilemap[tile] = !any_vis ? TILE_SKIP : (all_open ? TILE_OPEN : TILE_MIXED);
}

}  // namespace

cudaError_t launch_dsum(const BwdArgs& a, float* dsum, float* dq_acc_to_zero, int groups, uint32_t* zero_words,
                        int n_zero) {
  const Shape& s = a.s;
  const long long rows = (long long)s.B * s.Hq * s.Sq;
  if (rows == 0 && n_zero == 0) return cudaSuccess;
  const long long threads = std::max<long long>(rows * (s.D / 8), n_zero);
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  cudaError_t e = prof_begin(KID_BWD_DSUM, a.stream);
  if (e != cudaSuccess) return e;
  if (s.dtype == DT_BF16) {
    if (s.D == 64)
      dsum_kernel<__nv_bfloat16, 64><<<blocks, 256, 0, a.stream>>>(
          (const __nv_bfloat16*)a.o, (const __nv_bfloat16*)a.dO, dsum, dq_acc_to_zero, rows, groups, zero_words,
          n_zero, s);
    else
      dsum_kernel<__nv_bfloat16, 128><<<blocks, 256, 0, a.stream>>>(
          (const __nv_bfloat16*)a.o, (const __nv_bfloat16*)a.dO, dsum, dq_acc_to_zero, rows, groups, zero_words,
          n_zero, s);
  } else {
    if (s.D == 64)
      dsum_kernel<float, 64><<<blocks, 256, 0, a.stream>>>((const float*)a.o, (const float*)a.dO, dsum,
                                                           dq_acc_to_zero, rows, groups, zero_words, n_zero, s);
    else
      dsum_kernel<float, 128><<<blocks, 256, 0, a.stream>>>((const float*)a.o, (const float*)a.dO, dsum,
                                                            dq_acc_to_zero, rows, groups, zero_words, n_zero, s);
  }
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return prof_end(KID_BWD_DSUM, a.stream);
}

cudaError_t launch_dq_convert(const BwdArgs& a, const float* dq_acc, int groups) {
  const Shape& s = a.s;
  const long long vecs = (long long)s.B * s.Hq * s.Sq * s.D / 8;
  if (vecs == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((vecs + 256LL * kConvVecs - 1) / (256LL * kConvVecs));
  cudaError_t e = prof_begin(KID_BWD_DQCONV, a.stream);
  if (e != cudaSuccess) return e;
  if (s.dtype == DT_BF16)
    dq_convert_kernel<__nv_bfloat16><<<blocks, 256, 0, a.stream>>>(dq_acc, (__nv_bfloat16*)a.dq, s.scale, vecs,
                                                                   groups, s);
  else
    dq_convert_kernel<float><<<blocks, 256, 0, a.stream>>>(dq_acc, (float*)a.dq, s.scale, vecs, groups, s);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return prof_end(KID_BWD_DQCONV, a.stream);
}

cudaError_t launch_mask_classify(const Shape& s, const void* mask, uint8_t* tilemap, cudaStream_t st) {
  if (s.mask_kind == MK_NONE || s.Sq == 0) return cudaSuccess;
  const int nqt = (s.Sq + 127) / 128, nkt = (s.Sk + 127) / 128;
  const long long tiles = (long long)s.mask_batch * nqt * nkt;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaError_t e = prof_begin(KID_MASK, st);
  if (e != cudaSuccess) return e;
  const bool add = s.mask_kind == MK_ADD;
  // rows start on 16-byte boundaries when Sk is a multiple of the vector width (the mask pointer
  // itself is 16-byte aligned, checked by the entry points)
  const bool vec = add ? (s.Sk % 4 == 0) : (s.Sk % 16 == 0);
  if (add && vec) mask_classify_kernel<true, true><<<(unsigned)tiles, 512, 0, st>>>(s, mask, tilemap, nqt, nkt);
  else if (add) mask_classify_kernel<true, false><<<(unsigned)tiles, 512, 0, st>>>(s, mask, tilemap, nqt, nkt);
  else if (vec) mask_classify_kernel<false, true><<<(unsigned)tiles, 512, 0, st>>>(s, mask, tilemap, nqt, nkt);
  else mask_classify_kernel<false, false><<<(unsigned)tiles, 512, 0, st>>>(s, mask, tilemap, nqt, nkt);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return prof_end(KID_MASK, st);
}

}  // namespace fa

// ---------------------------------------------------------------------------------------------
// Self-test of the bounded waits: one thread waits on an mbarrier that nothing ever arrives on,
// with a short limit; the wait gives up, records its site in the status word and the kernel
// returns normally, leaving the context usable.
// ---------------------------------------------------------------------------------------------

namespace fa {
namespace {

__global__ void wait_selftest_kernel(unsigned* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  tc::mbar_init(&bar, 1);
  tc::fence_barrier_init();
  __syncwarp();
  // phase 0 never completes: nobody arrives
  tc::mbar_wait(&bar, 0, nullptr, status, kSelfTestSite, limit_ns);
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t st) {
  unsigned* status = device_status_ptr();
  if (status == nullptr) return cudaErrorUnknown;
  wait_selftest_kernel<<<1, 1, 0, st>>>(status, limit_ns);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace fa

namespace fa {
namespace {

// One thread per 16 features of a key row: one 16-byte load of values, one scale, 32 bytes out.
__global__ void __launch_bounds__(256) q8_dequant_kernel(const int8_t* __restrict__ xq, const __half* __restrict__ xd,
                                                         __nv_bfloat16* __restrict__ out, long long segs) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= segs) return;
  const long long e0 = i * 16;           // first feature of the segment; its scale is e0 / 32
  const int4 raw = __ldg(reinterpret_cast<const int4*>(xq + e0));
  const float scale = __half2float(xd[e0 / 32]);
  const uint32_t uw[4] = {(uint32_t)raw.x ^ 0x80808080u, (uint32_t)raw.y ^ 0x80808080u,
                          (uint32_t)raw.z ^ 0x80808080u, (uint32_t)raw.w ^ 0x80808080u};
  uint32_t w[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    w[k] = tc::pack_bf16x2(s8_to_f32(uw[k / 2], (k % 2) * 2) * scale, s8_to_f32(uw[k / 2], (k % 2) * 2 + 1) * scale);
  uint4* dst = reinterpret_cast<uint4*>(out + e0);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

}  // namespace

cudaError_t launch_q8_dequant(const Shape& s, const int8_t* xq, const void* xd, void* out, cudaStream_t st) {
  const long long segs = (long long)s.B * s.Hkv * s.Sk * s.D / 16;
  if (segs == 0) return cudaSuccess;
  const long long blocks = (segs + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  q8_dequant_kernel<<<(unsigned)blocks, 256, 0, st>>>(xq, static_cast<const __half*>(xd),
                                                       static_cast<__nv_bfloat16*>(out), segs);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace fa

namespace fa {
namespace {

// One thread per 8 elements: one 16-byte load of fp16, one 16-byte store of bf16 (each value
// widened exactly to fp32, then rounded to nearest even).
__global__ void __launch_bounds__(256) f16_to_bf16_kernel(const uint4* __restrict__ x, uint4* __restrict__ out,
                                                          long long segs) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= segs) return;
  const uint4 raw = __ldg(x + i);
  const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&in[k]));
    w[k] = tc::pack_bf16x2(f.x, f.y);
  }
  out[i] = make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace

cudaError_t launch_f16_to_bf16(const void* x, void* out, long long n, cudaStream_t st) {
  if (n % 8 != 0) return cudaErrorInvalidValue;
  const long long segs = n / 8;
  if (segs == 0) return cudaSuccess;
  const long long blocks = (segs + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  f16_to_bf16_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<const uint4*>(x), static_cast<uint4*>(out), segs);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace fa
