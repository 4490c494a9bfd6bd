// SIMT fp32 kernels for the fused attention training op.
//
// These carry the fp32-input path (where bf16 tensor cores would not meet an
// fp32 tolerance) and any shape the tensor-core path does not take. They
// compute in fp32 with accurate expf/logf and follow the op's definition
// directly: an online softmax in the forward, P recomputed from LSE in the
// backward (llama.cpp PR #57, commit 86c140d: LSE, D, then per-tile
// gradients, GQA group-sum), and two atomic-free backward kernels: one owns
// key columns (dK, dV summed over the query heads of its group), the other
// owns query rows (dQ).
#include <cuda_runtime.h>

#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kThreads = 256;  // 8 warps

// ---------------------------------------------------------------------------
// Forward: a block takes 16 query rows of one (batch, query head); each warp
// owns 2 rows. Keys are walked in tiles of 32 staged in shared memory; lane j
// scores key j of the tile against the warp's row, then the row's running max,
// sum and the lane's slice of O are updated (online softmax).
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(Shape s, const T* __restrict__ q,
                                                            const T* __restrict__ k,
                                                            const T* __restrict__ v, const void* mask,
                                                            T* __restrict__ o, float* __restrict__ lse) {
  constexpr int KT = 32, ROWS = 16, DP = D + 1, NT = D / 32;
  __shared__ float Ks[KT][DP];
  __shared__ float Vs[KT][DP];
  __shared__ float Qs[ROWS][D];

  const int b = blockIdx.z, h = blockIdx.y;
  const int kvh = h / (s.Hq / s.Hkv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * ROWS;
  const size_t qs = row_stride(s, s.Hq), ks = row_stride(s, s.Hkv);   // row strides of one head
  const T* qh = q + head_base(s, b, h, s.Hq, s.Sq);
  const T* kh = k + head_base(s, b, kvh, s.Hkv, s.Sk);
  const T* vh = v + head_base(s, b, kvh, s.Hkv, s.Sk);

  for (int idx = threadIdx.x; idx < ROWS * D; idx += kThreads) {
    const int r = idx / D, d = idx % D, i = row0 + r;
    Qs[r][d] = (i < s.Sq) ? to_f(qh[(size_t)i * qs + d]) : 0.f;
  }

  float m[2] = {-CUDART_INF_F, -CUDART_INF_F};
  float l[2] = {0.f, 0.f};
  float acc[2][NT];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr)
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[rr][t] = 0.f;

  long long kend = s.Sk;
  if (s.causal) {
    const long long last_row = (long long)min(row0 + ROWS, s.Sq) - 1;
    kend = min(kend, s.q_offset + last_row + 1);
  }

  for (int j0 = 0; j0 < kend; j0 += KT) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < KT * D; idx += kThreads) {
      const int r = idx / D, d = idx % D, j = j0 + r;
      const bool in = j < s.Sk;
      Ks[r][d] = in ? to_f(kh[(size_t)j * ks + d]) : 0.f;
      Vs[r][d] = in ? to_f(vh[(size_t)j * ks + d]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int r = warp * 2 + rr, i = row0 + r, j = j0 + lane;
      float dot = 0.f;
#pragma unroll 16
      for (int d = 0; d < D; ++d) dot = fmaf(Qs[r][d], Ks[lane][d], dot);
      float bias;
      const bool vis = pair_visible(s, mask, b, i, j, bias);
      const float sc = vis ? fmaf(dot, s.scale, bias) : -CUDART_INF_F;
      const float mnew = fmaxf(m[rr], warp_max(sc));
      if (mnew == -CUDART_INF_F) continue;  // nothing visible yet (warp-uniform)
      const float alpha = expf(m[rr] - mnew);
      const float p = vis ? expf(sc - mnew) : 0.f;
      l[rr] = l[rr] * alpha + warp_sum(p);
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[rr][t] *= alpha;
#pragma unroll 8
      for (int jj = 0; jj < KT; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[rr][t] = fmaf(pj, Vs[jj][lane + 32 * t], acc[rr][t]);
      }
      m[rr] = mnew;
    }
  }

#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int i = row0 + warp * 2 + rr;
    if (i >= s.Sq) continue;
    const bool alive = l[rr] > 0.f;
    const float inv = alive ? 1.f / l[rr] : 0.f;
    T* orow = o + head_base(s, b, h, s.Hq, s.Sq) + (size_t)i * qs;
#pragma unroll
    for (int t = 0; t < NT; ++t) from_f(orow + lane + 32 * t, acc[rr][t] * inv);
    if (lane == 0) lse[(size_t)(b * s.Hq + h) * s.Sq + i] = alive ? m[rr] + logf(l[rr]) : 0.f;
  }
}

// ---------------------------------------------------------------------------
// Backward, key-column owner: a block owns 32 keys of one (batch, kv head);
// each warp owns 4 of them and keeps their dK, dV slices in registers while it
// walks every query row of every query head of the GQA group. Lane i scores
// query row i of the staged tile; the per-pair P and dS are then broadcast.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) bwd_dkdv_simt_kernel(
    Shape s, const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, const void* mask,
    const float* __restrict__ lse, const T* __restrict__ dO, const float* __restrict__ dsum, void* dk_out,
    void* dv_out, bool accum, long long rows_begin, int n_rows, T* dk_rows, T* dv_rows) {
  constexpr int KT = 32, QT = 32, DP = D + 1, NT = D / 32, KPW = KT / 8;
  extern __shared__ float smem_dkdv[];
  float (*Qs)[DP] = reinterpret_cast<float (*)[DP]>(smem_dkdv);
  float (*dOs)[DP] = reinterpret_cast<float (*)[DP]>(smem_dkdv + QT * DP);
  float (*Ks)[D] = reinterpret_cast<float (*)[D]>(smem_dkdv + 2 * QT * DP);
  float (*Vs)[D] = reinterpret_cast<float (*)[D]>(smem_dkdv + 2 * QT * DP + KT * D);
  float* lse_s = smem_dkdv + 2 * QT * DP + 2 * KT * D;
  float* dsum_s = lse_s + QT;

  const int b = blockIdx.z, kvh = blockIdx.y;
  const int G = s.Hq / s.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j0 = blockIdx.x * KT;
  const size_t qs = row_stride(s, s.Hq), ks = row_stride(s, s.Hkv);   // row strides of one head
  const T* kh = k + head_base(s, b, kvh, s.Hkv, s.Sk);
  const T* vh = v + head_base(s, b, kvh, s.Hkv, s.Sk);

  for (int idx = threadIdx.x; idx < KT * D; idx += kThreads) {
    const int r = idx / D, d = idx % D, j = j0 + r;
    const bool in = j < s.Sk;
    Ks[r][d] = in ? to_f(kh[(size_t)j * ks + d]) : 0.f;
    Vs[r][d] = in ? to_f(vh[(size_t)j * ks + d]) : 0.f;
  }

  float dk[KPW][NT], dv[KPW][NT];
#pragma unroll
  for (int kk = 0; kk < KPW; ++kk)
#pragma unroll
    for (int t = 0; t < NT; ++t) dk[kk][t] = dv[kk][t] = 0.f;

  // Under the causal rule, rows below j0 - q_offset see none of these keys.
  int ibeg = 0;
  if (s.causal) {
    const long long first = (long long)j0 - s.q_offset;
    ibeg = first <= 0 ? 0 : (int)((first / QT) * QT);
  }

  for (int hh = 0; hh < G; ++hh) {
    const int h = kvh * G + hh;
    const size_t rowbase = (size_t)(b * s.Hq + h) * s.Sq;   // LSE and D rows
    const size_t qbase = head_base(s, b, h, s.Hq, s.Sq);
    for (int i0 = ibeg; i0 < s.Sq; i0 += QT) {
      __syncthreads();
      for (int idx = threadIdx.x; idx < QT * D; idx += kThreads) {
        const int r = idx / D, d = idx % D, i = i0 + r;
        const bool in = i < s.Sq;
        Qs[r][d] = in ? to_f(q[qbase + (size_t)i * qs + d]) : 0.f;
        dOs[r][d] = in ? to_f(dO[qbase + (size_t)i * qs + d]) : 0.f;
      }
      if (threadIdx.x < QT) {
        const int i = i0 + threadIdx.x;
        lse_s[threadIdx.x] = i < s.Sq ? lse[rowbase + i] : 0.f;
        dsum_s[threadIdx.x] = i < s.Sq ? dsum[rowbase + i] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < KPW; ++kk) {
        const int jl = warp * KPW + kk, j = j0 + jl, i = i0 + lane;
        float sdot = 0.f, pdot = 0.f;
#pragma unroll 16
        for (int d = 0; d < D; ++d) {
          sdot = fmaf(Qs[lane][d], Ks[jl][d], sdot);
          pdot = fmaf(dOs[lane][d], Vs[jl][d], pdot);
        }
        float bias;
        const bool vis = pair_visible(s, mask, b, i, j, bias);
        const float p = vis ? expf(fmaf(sdot, s.scale, bias) - lse_s[lane]) : 0.f;
        const float ds = p * (pdot - dsum_s[lane]);
#pragma unroll 8
        for (int il = 0; il < QT; ++il) {
          const float pi = __shfl_sync(0xffffffffu, p, il);
          const float dsi = __shfl_sync(0xffffffffu, ds, il);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            dv[kk][t] = fmaf(pi, dOs[il][lane + 32 * t], dv[kk][t]);
            dk[kk][t] = fmaf(dsi, Qs[il][lane + 32 * t], dk[kk][t]);
          }
        }
      }
    }
  }

#pragma unroll
  for (int kk = 0; kk < KPW; ++kk) {
    const int j = j0 + warp * KPW + kk;
    if (j >= s.Sk) continue;
    const size_t base = head_base(s, b, kvh, s.Hkv, s.Sk) + (size_t)j * ks;
    // the fused SET_ROWS backward: this key's finished sum is also one of the read-back rows
    const long long rr = (long long)j - rows_begin;
    const bool read_back = accum && rr >= 0 && rr < n_rows;
    const size_t rbase = head_base(s, b, kvh, s.Hkv, n_rows) + (size_t)(read_back ? rr : 0) * ks;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const size_t idx = base + lane + 32 * t;
      const float gk = dk[kk][t] * s.scale, gv = dv[kk][t];
      if (accum) {
        const float nk = static_cast<float*>(dk_out)[idx] + gk, nv = static_cast<float*>(dv_out)[idx] + gv;
        static_cast<float*>(dk_out)[idx] = nk;
        static_cast<float*>(dv_out)[idx] = nv;
        if (read_back) {
          from_f(dk_rows + rbase + lane + 32 * t, nk);
          from_f(dv_rows + rbase + lane + 32 * t, nv);
        }
      } else {
        from_f(static_cast<T*>(dk_out) + idx, gk);
        from_f(static_cast<T*>(dv_out) + idx, gv);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Backward, query-row owner: a block owns 32 query rows of one (batch, query
// head); each warp owns 4 rows and keeps their dQ slices in registers while it
// walks the keys. Lane j scores key j of the staged tile.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) bwd_dq_simt_kernel(Shape s, const T* __restrict__ q,
                                                               const T* __restrict__ k,
                                                               const T* __restrict__ v, const void* mask,
                                                               const float* __restrict__ lse,
                                                               const T* __restrict__ dO,
                                                               const float* __restrict__ dsum,
                                                               T* __restrict__ dq) {
  constexpr int KT = 32, ROWS = 32, DP = D + 1, NT = D / 32, RPW = ROWS / 8;
  extern __shared__ float smem_dq[];
  float (*Ks)[DP] = reinterpret_cast<float (*)[DP]>(smem_dq);
  float (*Vs)[DP] = reinterpret_cast<float (*)[DP]>(smem_dq + KT * DP);
  float (*Qs)[D] = reinterpret_cast<float (*)[D]>(smem_dq + 2 * KT * DP);
  float (*dOs)[D] = reinterpret_cast<float (*)[D]>(smem_dq + 2 * KT * DP + ROWS * D);

  const int b = blockIdx.z, h = blockIdx.y;
  const int kvh = h / (s.Hq / s.Hkv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * ROWS;
  const size_t rowbase = (size_t)(b * s.Hq + h) * s.Sq;   // LSE and D rows
  const size_t qs = row_stride(s, s.Hq), ks = row_stride(s, s.Hkv);   // row strides of one head
  const size_t qbase = head_base(s, b, h, s.Hq, s.Sq);
  const T* kh = k + head_base(s, b, kvh, s.Hkv, s.Sk);
  const T* vh = v + head_base(s, b, kvh, s.Hkv, s.Sk);

  for (int idx = threadIdx.x; idx < ROWS * D; idx += kThreads) {
    const int r = idx / D, d = idx % D, i = row0 + r;
    const bool in = i < s.Sq;
    Qs[r][d] = in ? to_f(q[qbase + (size_t)i * qs + d]) : 0.f;
    dOs[r][d] = in ? to_f(dO[qbase + (size_t)i * qs + d]) : 0.f;
  }
  float row_lse[RPW], row_d[RPW];
#pragma unroll
  for (int rr = 0; rr < RPW; ++rr) {
    const int i = row0 + warp * RPW + rr;
    row_lse[rr] = i < s.Sq ? lse[rowbase + i] : 0.f;
    row_d[rr] = i < s.Sq ? dsum[rowbase + i] : 0.f;
  }
  float acc[RPW][NT];
#pragma unroll
  for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[rr][t] = 0.f;

  long long kend = s.Sk;
  if (s.causal) {
    const long long last_row = (long long)min(row0 + ROWS, s.Sq) - 1;
    kend = min(kend, s.q_offset + last_row + 1);
  }

  for (int j0 = 0; j0 < kend; j0 += KT) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < KT * D; idx += kThreads) {
      const int r = idx / D, d = idx % D, j = j0 + r;
      const bool in = j < s.Sk;
      Ks[r][d] = in ? to_f(kh[(size_t)j * ks + d]) : 0.f;
      Vs[r][d] = in ? to_f(vh[(size_t)j * ks + d]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
      const int r = warp * RPW + rr, i = row0 + r, j = j0 + lane;
      float sdot = 0.f, pdot = 0.f;
#pragma unroll 16
      for (int d = 0; d < D; ++d) {
        sdot = fmaf(Qs[r][d], Ks[lane][d], sdot);
        pdot = fmaf(dOs[r][d], Vs[lane][d], pdot);
      }
      float bias;
      const bool vis = pair_visible(s, mask, b, i, j, bias);
      const float p = vis ? expf(fmaf(sdot, s.scale, bias) - row_lse[rr]) : 0.f;
      const float ds = p * (pdot - row_d[rr]);
#pragma unroll 8
      for (int jj = 0; jj < KT; ++jj) {
        const float dsj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[rr][t] = fmaf(dsj, Ks[jj][lane + 32 * t], acc[rr][t]);
      }
    }
  }

#pragma unroll
  for (int rr = 0; rr < RPW; ++rr) {
    const int i = row0 + warp * RPW + rr;
    if (i >= s.Sq) continue;
#pragma unroll
    for (int t = 0; t < NT; ++t) from_f(dq + qbase + (size_t)i * qs + lane + 32 * t, acc[rr][t] * s.scale);
  }
}

template <typename T, int D>
cudaError_t simt_fwd_t(const FwdArgs& a) {
  const Shape& s = a.s;
  dim3 grid((s.Sq + 15) / 16, s.Hq, s.B);
  cudaError_t e = prof_begin(KID_FWD, a.stream);
  if (e != cudaSuccess) return e;
  fwd_simt_kernel<T, D><<<grid, kThreads, 0, a.stream>>>(s, (const T*)a.q, (const T*)a.k, (const T*)a.v,
                                                         a.mask, (T*)a.o, a.lse);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return prof_end(KID_FWD, a.stream);
}

template <typename T, int D>
cudaError_t simt_bwd_t(const BwdArgs& a, const float* dsum) {
  const Shape& s = a.s;
  const size_t sm1 = sizeof(float) * (2 * 32 * (D + 1) + 2 * 32 * D + 2 * 32);
  const size_t sm2 = sizeof(float) * (2 * 32 * (D + 1) + 2 * 32 * D);
  cudaError_t e = cudaFuncSetAttribute(bwd_dkdv_simt_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sm1);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_dq_simt_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2);
  if (e != cudaSuccess) return e;
  dim3 g1((s.Sk + 31) / 32, s.Hkv, s.B);
  if ((e = prof_begin(KID_BWD_MAIN, a.stream)) != cudaSuccess) return e;
  bwd_dkdv_simt_kernel<T, D><<<g1, kThreads, sm1, a.stream>>>(s, (const T*)a.q, (const T*)a.k, (const T*)a.v,
                                                            a.mask, a.lse, (const T*)a.dO, dsum, a.dk, a.dv,
                                                            a.accum, a.rows_begin, a.accum ? a.n_rows : 0,
                                                            (T*)a.dk_rows, (T*)a.dv_rows);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 g2((s.Sq + 31) / 32, s.Hq, s.B);
  bwd_dq_simt_kernel<T, D><<<g2, kThreads, sm2, a.stream>>>(s, (const T*)a.q, (const T*)a.k, (const T*)a.v,
                                                          a.mask, a.lse, (const T*)a.dO, dsum, (T*)a.dq);
  count_launches(2);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return prof_end(KID_BWD_MAIN, a.stream);
}

}  // namespace

cudaError_t simt_fwd(const FwdArgs& a) {
  if (a.s.dtype == DT_F32) return a.s.D == 64 ? simt_fwd_t<float, 64>(a) : simt_fwd_t<float, 128>(a);
  return a.s.D == 64 ? simt_fwd_t<__nv_bfloat16, 64>(a) : simt_fwd_t<__nv_bfloat16, 128>(a);
}

cudaError_t simt_bwd(const BwdArgs& a, float* dsum) {
  cudaError_t e = launch_dsum(a, dsum, nullptr);
  if (e != cudaSuccess) return e;
  if (a.s.dtype == DT_F32)
    return a.s.D == 64 ? simt_bwd_t<float, 64>(a, dsum) : simt_bwd_t<float, 128>(a, dsum);
  return a.s.D == 64 ? simt_bwd_t<__nv_bfloat16, 64>(a, dsum) : simt_bwd_t<__nv_bfloat16, 128>(a, dsum);
}

}  // namespace fa
