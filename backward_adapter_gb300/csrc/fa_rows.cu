// SET_ROWS backward: the gradient of the rows a chunk wrote into its cached K/V window is the
// window gradient at those rows (llama.cpp PR #57, commit 2394a4c: "the written source's
// gradient is the result's gradient at the written rows; the destination, a cache, carries
// none"). A gather out of the fp32 window accumulator, HBM-bound: each thread moves 16 bytes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

// A block covers up to 256 / (D / 4) (head, output row) pairs, one float4 column per thread.
// idx == nullptr reads the contiguous rows row0 .. row0 + n_rows - 1.
template <typename T>
__global__ void __launch_bounds__(256) set_rows_backward_kernel(const float* __restrict__ acc, int heads, int S,
                                                                int D, const int64_t* __restrict__ idx,
                                                                long long row0, int n_rows, T* __restrict__ out,
                                                                unsigned* status, int H, int layout) {
  const int vec = D / 4;                              // float4 per row
  const int rows_per_block = blockDim.x / vec;
  const long long g = (long long)blockIdx.x * rows_per_block + threadIdx.x / vec;   // (bh, r) flattened
  const int c = threadIdx.x % vec;
  if (threadIdx.x >= rows_per_block * vec || g >= (long long)heads * n_rows) return;
  const int bh = (int)(g / n_rows), r = (int)(g % n_rows);
  const int b = bh / H, h = bh % H;
  // [B, H, rows, D], or [B, rows, H, D] when layout == 1
  auto at = [&](long long rows, long long i) -> size_t {
    return layout ? (((size_t)b * rows + i) * H + h) * D : (((size_t)b * H + h) * rows + i) * D;
  };
  const long long src = idx != nullptr ? __ldg(idx + r) : row0 + r;
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (src >= 0 && src < S) {
    v = __ldg(reinterpret_cast<const float4*>(acc + at(S, src)) + c);
  } else if (c == 0 && status != nullptr) {
    atomicCAS(status, 0u, 0x40000000u | kSiteRowIndex);
  }
  T* dst = out + at(n_rows, r) + 4 * c;
  if constexpr (sizeof(T) == 4) {
    *reinterpret_cast<float4*>(dst) = v;
  } else {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst) = u;
  }
}

}  // namespace

static cudaError_t gather_rows(const float* acc, int heads, int S, int D, const int64_t* idx, long long row0,
                               int n_rows, void* out, int out_dtype, unsigned* status, cudaStream_t st, int H = 1,
                               int layout = 0) {
  const int vec = D / 4;
  const int rows_per_block = 256 / vec;
  const long long total = (long long)heads * n_rows;
  const long long blocks = (total + rows_per_block - 1) / rows_per_block;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (blocks == 0) return cudaSuccess;
  if (out_dtype == DT_BF16)
    set_rows_backward_kernel<__nv_bfloat16><<<(unsigned)blocks, rows_per_block * vec, 0, st>>>(
        acc, heads, S, D, idx, row0, n_rows, static_cast<__nv_bfloat16*>(out), status, H, layout);
  else
    set_rows_backward_kernel<float><<<(unsigned)blocks, rows_per_block * vec, 0, st>>>(
        acc, heads, S, D, idx, row0, n_rows, static_cast<float*>(out), status, H, layout);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_set_rows_backward(const float* acc, int heads, int S, int D, const int64_t* idx, int n_rows,
                                     void* out, int out_dtype, unsigned* status, cudaStream_t st) {
  return gather_rows(acc, heads, S, D, idx, 0, n_rows, out, out_dtype, status, st);
}

cudaError_t launch_rows_copy(const Shape& s, const float* dk_acc, const float* dv_acc, long long row0, int n_rows,
                             void* dk_rows, void* dv_rows, cudaStream_t st) {
  cudaError_t e = gather_rows(dk_acc, s.B * s.Hkv, s.Sk, s.D, nullptr, row0, n_rows, dk_rows, s.dtype, nullptr, st,
                              s.Hkv, s.layout);
  if (e == cudaSuccess)
    e = gather_rows(dv_acc, s.B * s.Hkv, s.Sk, s.D, nullptr, row0, n_rows, dv_rows, s.dtype, nullptr, st, s.Hkv, s.layout);
  return e;
}

}  // namespace fa
