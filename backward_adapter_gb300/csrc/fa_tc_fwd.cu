// Forward of the fused attention training op on the 5th-generation tensor
// cores (tcgen05, sm_103a): O = softmax(scale * Q K^T + mask) V and the per-row
// LSE (flash-attn-training skill, trap list item 9: a fully-masked row gives
// O = 0 and LSE = 0; llama.cpp PR #57, commit 86c140d: the backward needs LSE).
//
// One CTA takes 256 query rows (two 128-row tiles Q0, Q1) of one (batch, query
// head) and walks the visible 128-key tiles of its key/value head:
//   warp 0      TMA producer: Q0/Q1 once, then a ring of stages, each holding V of
//               one key tile and K of the next (one wait per tile for the issuer; the
//               stage is released by the completion of the tile's last MMA group);
//   warp 1      MMA issuer (one thread) and TMEM owner:
//                 S_t = Q_t K_j^T  (SMEM x SMEM -> TMEM fp32)
//                 O_t += P_t V_j   (P from TMEM, V from SMEM -> TMEM fp32);
//   warps 4-7   softmax for Q0, warps 8-11 softmax for Q1: a thread owns one
//               query row, reads its 128 scores from TMEM, applies scale, mask
//               and the causal rule, keeps the running max / sum in the log2
//               domain and writes P (bf16) back into TMEM over its scores.
// The two softmax groups ping-pong: while one works on its scores, the tensor
// core runs the other tile's S and PV MMAs. O is rescaled in TMEM only when a
// row's running max grows by more than 2^8 (otherwise P keeps the older max,
// which bounds P by 256 and leaves O, l and LSE consistent).
//
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256, 256+D), O1 [256+D, 256+2D).
// Long key windows with few query rows split the keys over CTAs; each split
// writes unnormalised (O, m, l) partials and a combine kernel merges them.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_device.cuh"
#include "fa_internal.h"
#include "tc_ptx.cuh"

namespace fa {
namespace {

using namespace tc;

constexpr int kBM = 128;        // query rows per tile
constexpr int kBN = 128;        // keys per tile
constexpr int kRowsPerCta = 2 * kBM;
constexpr int kThreads = 384;   // 12 warps
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8
constexpr int kRegsControl = 80;
constexpr int kRegsSoftmax = 208;
static_assert((kRegsControl + 2 * kRegsSoftmax) * 128 <= kThreads * 168, "register split exceeds the launch pool");

struct FwdTcParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_o;
  Shape s;
  const void* mask;
  const uint8_t* tilemap;   // [mask_batch, nqt, nkt] or null
  __nv_bfloat16* o;
  float* lse;
  float* part_o;            // [splits, rows, D] when split
  float* part_ml;           // [splits, rows, 2] when split
  int kv_splits;
  int n_qpairs;
  int nqt, nkt;
  unsigned* status;
};

template <int D>
struct FwdSmem {
  static constexpr int kBoxBytes = 128 * 128;            // 128 rows x 64 bf16 (one 128B-swizzled box)
  static constexpr int kTileBytes = kBM * D * 2;         // one Q or K or V tile
  static constexpr int kSlots = D == 128 ? 4 : 8;        // ring slots for K and V tiles
  static constexpr int kStages = kSlots / 2;             // a stage: V of one key tile and K of the next
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = 2 * kTileBytes;
  static constexpr int kBarOff = kKVOff + kSlots * kTileBytes;
  static constexpr int kBytes = kBarOff + 256 + 1024;    // barriers + alignment slack
};

// Key-tile range of a CTA after causal / sliding-window clipping and the split.
struct KvRange {
  int begin, end;  // tile indices [begin, end)
};

__host__ __device__ __forceinline__ KvRange kv_range(const FwdTcParams& p, int q_row0, int split) {
  const Shape& s = p.s;
  const long long last_row = (long long)min(q_row0 + kRowsPerCta, s.Sq) - 1;
  long long kv_beg = 0, kv_end = s.Sk;
  if (s.causal) kv_end = min(kv_end, s.q_offset + last_row + 1);
  if (s.window > 0) {
    kv_beg = max(0LL, s.q_offset + q_row0 - s.window);
    kv_end = min(kv_end, s.q_offset + last_row + s.window + 1);
  }
  const int t0 = (int)(kv_beg / kBN);
  const int n = max(0, (int)((kv_end + kBN - 1) / kBN) - t0);
  const int per = (n + p.kv_splits - 1) / p.kv_splits;
  KvRange r;
  r.begin = t0 + min(n, split * per);
  r.end = t0 + min(n, split * per + per);
  return r;
}

// A work unit: 256 query rows (two 128-row tiles) of one (batch, head), and its key range.
struct FwdUnit {
  int bh, b, h, kvh, q_row0, qt0, mb, split;
  KvRange kr;
};

// Unit ui of this CTA (false past its last one). PERSIST: a persistent grid of G CTAs, CTA c runs
// the units c, 2G-1-c, 2G+c, ... (units heaviest first); otherwise one unit (and key split) per CTA.
template <bool PERSIST>
__device__ __forceinline__ bool fwd_unit(const FwdTcParams& p, int ui, FwdUnit& u) {
  const Shape& s = p.s;
  const int BH = s.B * s.Hq;
  long long rest;
  int split = 0;
  if constexpr (PERSIST) {
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    rest = (long long)ui * G + ((ui & 1) ? G - 1 - c : c);
    if (rest >= (long long)p.n_qpairs * BH) return false;
  } else {
    if (ui > 0) return false;
    split = (int)(blockIdx.x % p.kv_splits);
    rest = blockIdx.x / p.kv_splits;
  }
  u.bh = (int)(rest % BH);
  const int qpair = p.n_qpairs - 1 - (int)(rest / BH);   // heaviest first (causal work grows with rows)
  u.b = u.bh / s.Hq;
  u.h = u.bh % s.Hq;
  u.kvh = u.h / (s.Hq / s.Hkv);
  u.q_row0 = qpair * kRowsPerCta;
  u.qt0 = u.q_row0 / kBM;
  u.mb = s.mask_batch > 1 ? u.b : 0;
  u.split = split;
  u.kr = kv_range(p, u.q_row0, split);
  return true;
}

// Tile-map code of (query tile qt, key tile j), TILE_OPEN without a mask.
__device__ __forceinline__ int tile_code(const FwdTcParams& p, int mb, int qt, int j) {
  if (p.tilemap == nullptr) return TILE_OPEN;
  if (qt >= p.nqt) return TILE_SKIP;
  return p.tilemap[((size_t)mb * p.nqt + qt) * p.nkt + j];
}

__device__ __forceinline__ bool skip_tile(const FwdTcParams& p, int mb, int qt0, int j) {
  return tile_code(p, mb, qt0, j) == TILE_SKIP && tile_code(p, mb, qt0 + 1, j) == TILE_SKIP;
}

// MASKED: the call has a mask tensor (without one, the instance has no mixed-tile code).
template <int D, bool MASKED, bool POS_SCALE, bool PERSIST>
__global__ void __launch_bounds__(kThreads, 1) fwd_tc_kernel(const __grid_constant__ FwdTcParams p) {
  using L = FwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + L::kQOff;
  uint8_t* sKV = smem + L::kKVOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* bar_q = bars + 0;                     // [2]: query tile t of the unit loaded
  uint64_t* bar_qfree = bars + 2;                 // [2]: its buffer drained by the unit's epilogue
  uint64_t* bar_full = bars + 4;                  // [kStages]: stage filled
  uint64_t* bar_empty = bar_full + L::kStages;    // [kStages]: MMAs of the stage's step done
  uint64_t* bar_s = bar_empty + L::kStages;       // [2]
  uint64_t* bar_p = bar_s + 2;                    // [2]
  uint64_t* bar_o = bar_p + 2;                    // [2]
  uint64_t* bar_done = bar_o + 2;                 // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const Shape& s = p.s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar_q[t], 1);
      mbar_init(&bar_qfree[t], 1);
    }
    for (int i = 0; i < L::kStages; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar_s[t], 1);
      mbar_init(&bar_p[t], 4);
      mbar_init(&bar_o[t], 1);
    }
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Register split by warpgroup (setmaxnreg, inside each role's branch): the launch holds
  // 384 x 168 registers; the control warpgroup keeps 80 and the two softmax warpgroups take 208
  // each: (80 + 208 + 208) x 128 = 63488 <= 64512.
  if (warp < 4) {
   regs_dec<kRegsControl>();   // all four warps of the control warpgroup
   if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&p.tm_q);
      prefetch_tmap(&p.tm_k);
      prefetch_tmap(&p.tm_v);
      // Stage st of the ring holds V of the (st-1)-th key tile and K of the st-th: the MMAs of one
      // step read exactly one stage, so a step costs the issuer one wait. The issuer commits a
      // stage's MMAs to its bar_empty; fill k of a stage waits for the k-th completion of that
      // barrier, which cannot complete again before fill k, so its phase parity cannot alias.
      uint32_t used_mask = 0, phase_mask = 0;  // per stage: filled at least once / parity of its last fill
      if constexpr (!PERSIST) {
        FwdUnit u;
        fwd_unit<false>(p, 0, u);
        mbar_arrive_expect_tx(&bar_q[0], 2 * L::kTileBytes);
        for (int t = 0; t < 2; ++t)
          for (int box = 0; box < D / 64; ++box)
            tma_load_4d(sQ + t * L::kTileBytes + box * L::kBoxBytes, &p.tm_q, &bar_q[0], box * 64,
                        u.q_row0 + t * kBM, u.h, u.b);
        int st = 0, prev = -1;
        for (int j = u.kr.begin;; ++j) {
          while (j < u.kr.end && skip_tile(p, u.mb, u.qt0, j)) ++j;
          const bool has_k = j < u.kr.end;
          if (!has_k && prev < 0) break;
          const int sb = st % L::kStages;
          const uint32_t ph = (st / L::kStages) & 1;
          if (st >= L::kStages &&
              !mbar_wait<true>(&bar_empty[sb], ((st / L::kStages) - 1) & 1, abort_flag, p.status, 1))
            break;
          mbar_arrive_expect_tx(&bar_full[sb], (prev >= 0 ? L::kTileBytes : 0) + (has_k ? L::kTileBytes : 0));
          for (int box = 0; box < D / 64; ++box) {
            if (prev >= 0)
              tma_load_4d(sKV + (2 * sb + 1) * L::kTileBytes + box * L::kBoxBytes, &p.tm_v, &bar_full[sb],
                          box * 64, prev * kBN, u.kvh, u.b);
            if (has_k)
              tma_load_4d(sKV + 2 * sb * L::kTileBytes + box * L::kBoxBytes, &p.tm_k, &bar_full[sb], box * 64,
                          j * kBN, u.kvh, u.b);
          }
          used_mask |= 1u << sb;
          phase_mask = (phase_mask & ~(1u << sb)) | (ph << sb);
          ++st;
          if (!has_k) break;
          prev = j;
        }
        // Drain: every copy this thread issued has landed before the block can exit.
        mbar_wait<true>(&bar_q[0], 0, nullptr, p.status, 2);
      } else {
        // The key tiles of this CTA's units form one stream, so at a unit boundary one stage carries
        // the previous unit's last V and the next unit's first K. A unit's Q tile t is loaded once
        // the previous unit's epilogue has drained its buffer (bar_qfree), after the boundary stage
        // whose V that epilogue waits for.
        int st = 0;
        int nq[2] = {0, 0};   // Q loads issued per tile: the drain waits for the last of each
        int prev = -1, prev_kvh = 0, prev_b = 0;   // the stream's key tile whose V is still to load
        bool ok = true;
        auto stage = [&](bool has_k, int j, int kvh_k, int b_k) -> bool {
          const int sb = st % L::kStages;
          const uint32_t ph = (st / L::kStages) & 1;
          if (st >= L::kStages && !mbar_wait<true>(&bar_empty[sb], ((st / L::kStages) - 1) & 1, abort_flag, p.status, 1))
            return false;
          mbar_arrive_expect_tx(&bar_full[sb], (prev >= 0 ? L::kTileBytes : 0) + (has_k ? L::kTileBytes : 0));
          for (int box = 0; box < D / 64; ++box) {
            if (prev >= 0)
              tma_load_4d(sKV + (2 * sb + 1) * L::kTileBytes + box * L::kBoxBytes, &p.tm_v, &bar_full[sb], box * 64,
                          prev * kBN, prev_kvh, prev_b);
            if (has_k)
              tma_load_4d(sKV + 2 * sb * L::kTileBytes + box * L::kBoxBytes, &p.tm_k, &bar_full[sb], box * 64, j * kBN,
                          kvh_k, b_k);
          }
          used_mask |= 1u << sb;
          phase_mask = (phase_mask & ~(1u << sb)) | (ph << sb);
          ++st;
          prev = has_k ? j : -1;
          prev_kvh = kvh_k;
          prev_b = b_k;
          return true;
        };
        for (int ui = 0; ok; ++ui) {
          FwdUnit u;
          if (!fwd_unit<PERSIST>(p, ui, u)) break;
          int j = u.kr.begin;
          while (j < u.kr.end && skip_tile(p, u.mb, u.qt0, j)) ++j;
          if (j < u.kr.end) {
            ok = stage(true, j, u.kvh, u.b);
            ++j;
          }
          for (int t = 0; t < 2 && ok; ++t) {
            if (ui > 0 && !(ok = mbar_wait<true>(&bar_qfree[t], (ui - 1) & 1, abort_flag, p.status, 4))) break;
            mbar_arrive_expect_tx(&bar_q[t], L::kTileBytes);
            for (int box = 0; box < D / 64; ++box)
              tma_load_4d(sQ + t * L::kTileBytes + box * L::kBoxBytes, &p.tm_q, &bar_q[t], box * 64,
                          u.q_row0 + t * kBM, u.h, u.b);
            nq[t] = ui + 1;
          }
          for (; ok; ++j) {
            while (j < u.kr.end && skip_tile(p, u.mb, u.qt0, j)) ++j;
            if (j >= u.kr.end) break;
            ok = stage(true, j, u.kvh, u.b);
          }
        }
        if (ok && prev >= 0) stage(false, 0, 0, 0);   // the stream's last stage: V only
        // Drain: every copy this thread issued has landed before the block can exit.
        for (int t = 0; t < 2; ++t)
          if (nq[t] > 0) mbar_wait<true>(&bar_q[t], (nq[t] - 1) & 1, nullptr, p.status, 2);
      }
      for (int i = 0; i < L::kStages; ++i)
        if (used_mask >> i & 1u) mbar_wait<true>(&bar_full[i], (phase_mask >> i) & 1u, nullptr, p.status, 3);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, 0, 0);
      const uint32_t idesc_pv = idesc_bf16_f32(kBM, D, 0, 1);
      const uint32_t sQa = smem_u32(sQ), sKVa = smem_u32(sKV);
      // one base descriptor per operand tile; every k-step adds a compile-time byte offset
      auto issue_pv = [&](int t, int v_slot, uint32_t first_acc) {
        const uint64_t dv0 = smem_desc_sw128(sKVa + v_slot * L::kTileBytes, L::kBoxBytes, 1024);
        const uint32_t d_tmem = tmem + 256 + t * D, a_tmem = tmem + t * 128;
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)   // 16 keys (2048 B of V, 8 TMEM columns of P) per step
          mma_ts(d_tmem, a_tmem + k * 8, desc_add(dv0, k * 2048), idesc_pv, (first_acc || k > 0) ? 1u : 0u);
      };
      auto issue_s = [&](int t, int k_slot) {
        const uint64_t dq0 = smem_desc_sw128(sQa + t * L::kTileBytes, 16, 1024);
        const uint64_t dk0 = smem_desc_sw128(sKVa + k_slot * L::kTileBytes, 16, 1024);
        const uint32_t d_tmem = tmem + t * 128;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * L::kBoxBytes + (k & 3) * 32;
          mma_ss(d_tmem, desc_add(dq0, off), desc_add(dk0, off), idesc_qk, k > 0 ? 1u : 0u);
        }
      };
      if constexpr (!PERSIST) {
        // One unit (both Q tiles on bar_q[0]): a step issues tile t's P V of the previous key tile
        // then its S of this one, tile 0 then tile 1 (the softmax groups ping-pong).
        FwdUnit u;
        fwd_unit<false>(p, 0, u);
        bool ok = mbar_wait<true>(&bar_q[0], 0, abort_flag, p.status, 10);
        tc_fence_after();
        int idx = 0;  // visible key tiles processed = ring stages consumed
        for (int j = u.kr.begin; ok && j < u.kr.end; ++j) {
          if (skip_tile(p, u.mb, u.qt0, j)) continue;
          const int sb = idx % L::kStages;
          if (!(ok = mbar_wait<true>(&bar_full[sb], (idx / L::kStages) & 1, abort_flag, p.status, 11))) break;
          tc_fence_after();
#pragma unroll 1
          for (int t = 0; t < 2 && ok; ++t) {
            if (idx > 0) {
              if (!(ok = mbar_wait<true>(&bar_p[t], (idx - 1) & 1, abort_flag, p.status, 12))) break;
              tc_fence_after();
              issue_pv(t, 2 * sb + 1, idx - 1 > 0);
            }
            issue_s(t, 2 * sb);
            mma_commit(&bar_s[t]);
          }
          if (!ok) break;
          mma_commit(&bar_empty[sb]);
          ++idx;
        }
        if (ok && idx > 0) {
          // the last stage holds only V of the last visible tile
          const int sb = idx % L::kStages;
          ok = mbar_wait<true>(&bar_full[sb], (idx / L::kStages) & 1, abort_flag, p.status, 15);
#pragma unroll 1
          for (int t = 0; t < 2 && ok; ++t) {
            if (!(ok = mbar_wait<true>(&bar_p[t], (idx - 1) & 1, abort_flag, p.status, 14))) break;
            tc_fence_after();
            issue_pv(t, 2 * sb + 1, idx - 1 > 0);
            mma_commit(&bar_o[t]);
          }
        }
      } else {
        // The stream of key tiles over this CTA's units (see the producer), stepped as above within
        // a unit. At a unit boundary the previous unit's last P V of both tiles goes first, each
        // followed by its commit to bar_o (that unit's epilogue), and then this unit's first S of
        // each tile once its Q is in.
        bool ok = true;
        int gidx = 0;              // key tiles of the stream issued: stage index, bar_s / bar_p phases
        bool pend = false;         // a key tile whose P V is still to be issued
        bool pend_first = false;   // ... and it was its unit's first (that P V starts O afresh)
        for (int ui = 0; ok; ++ui) {
          FwdUnit u;
          if (!fwd_unit<PERSIST>(p, ui, u)) break;
          bool unit_first = true;
          for (int j = u.kr.begin; ok && j < u.kr.end; ++j) {
            if (skip_tile(p, u.mb, u.qt0, j)) continue;
            const int sb = gidx % L::kStages;
            if (!(ok = mbar_wait<true>(&bar_full[sb], (gidx / L::kStages) & 1, abort_flag, p.status, 11))) break;
            tc_fence_after();
            if (unit_first) {
#pragma unroll 1
              for (int t = 0; t < 2 && ok && pend; ++t) {
                if (!(ok = mbar_wait<true>(&bar_p[t], (gidx - 1) & 1, abort_flag, p.status, 12))) break;
                tc_fence_after();
                issue_pv(t, 2 * sb + 1, pend_first ? 0u : 1u);
                mma_commit(&bar_o[t]);
              }
#pragma unroll 1
              for (int t = 0; t < 2 && ok; ++t) {
                if (!(ok = mbar_wait<true>(&bar_q[t], ui & 1, abort_flag, p.status, 10))) break;
                tc_fence_after();
                issue_s(t, 2 * sb);
                mma_commit(&bar_s[t]);
              }
              if (ok) mma_commit(&bar_empty[sb]);
              unit_first = false;
              pend_first = true;
            } else {
#pragma unroll 1
              for (int t = 0; t < 2 && ok; ++t) {
                if (!(ok = mbar_wait<true>(&bar_p[t], (gidx - 1) & 1, abort_flag, p.status, 12))) break;
                tc_fence_after();
                issue_pv(t, 2 * sb + 1, pend_first ? 0u : 1u);
                issue_s(t, 2 * sb);
                mma_commit(&bar_s[t]);
              }
              if (ok) mma_commit(&bar_empty[sb]);
              pend_first = false;
            }
            if (!ok) break;
            pend = true;
            ++gidx;
          }
        }
        if (ok && pend) {
          // the stream's last stage holds only V of its last key tile
          const int sb = gidx % L::kStages;
          ok = mbar_wait<true>(&bar_full[sb], (gidx / L::kStages) & 1, abort_flag, p.status, 15);
#pragma unroll 1
          for (int t = 0; t < 2 && ok; ++t) {
            if (!(ok = mbar_wait<true>(&bar_p[t], (gidx - 1) & 1, abort_flag, p.status, 14))) break;
            tc_fence_after();
            issue_pv(t, 2 * sb + 1, pend_first ? 0u : 1u);
            mma_commit(&bar_o[t]);
          }
        }
      }
      // Every MMA this thread issued is complete before TMEM is released.
      mma_commit(bar_done);
      mbar_wait<true>(bar_done, 0, nullptr, p.status, 16);
    }
   }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax, one row per thread
    const int t = (warp - 4) / 4;
    const int wq = warp & 3;                       // TMEM lane slice of this warp
    const int r = wq * 32 + lane;                  // row within the query tile
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + t * 128 + lane_off;
    const uint32_t tO = tmem + 256 + t * D + lane_off;
    const float sl2 = s.scale * kLog2e;
    // POS_SCALE (scale > 0): the scores stay unscaled in registers and the scale is folded into
    // the exponent's FMA, one instruction per score fewer on a loop that is issue-bound; the tile
    // max of the unscaled scores times sl2 is the max of the scaled ones. A scale of 0 or below
    // takes the scaled copy (its max does not commute with the scaling).
    const float inv_scale = POS_SCALE ? 1.f / s.scale : 0.f;
    // mask rows start on 16-byte boundaries (the mask pointer itself is 16-byte aligned)
    const bool mask_vec = s.mask_kind == MK_ADD ? (s.Sk % 4 == 0) : (s.Sk % 16 == 0);
    bool ok = true;
    int gidx = 0;   // key tiles of the stream: bar_s / bar_p phases
    int n_o = 0;    // units with key tiles finished: bar_o phase
    for (int ui = 0; ok; ++ui) {
      FwdUnit u;
      if (!fwd_unit<PERSIST>(p, ui, u)) break;
      const int i = u.q_row0 + t * kBM + r;   // query row
      const int mb = u.mb, qt0 = u.qt0;
      // visible keys of this row: [key_lo, key_hi] from the causal rule and the window
      long long key_lo = 0, key_hi = (long long)s.Sk - 1;
      if (s.causal) key_hi = min(key_hi, s.q_offset + i);
      if (s.window > 0) {
        key_lo = s.q_offset + i - s.window;
        key_hi = min(key_hi, s.q_offset + i + s.window);
      }
      const size_t mrow = ((size_t)mb * s.Sq + (size_t)min(i, s.Sq - 1)) * (size_t)s.Sk;
      float m = -CUDART_INF_F, l = 0.f;
      int idx = 0;   // this unit's key tiles
      for (int j = u.kr.begin; j < u.kr.end; ++j) {
        if (skip_tile(p, mb, qt0, j)) continue;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait<true>(&bar_s[t], gidx & 1, abort_flag, p.status, 20)))) break;
        tc_fence_after();
        // scale into the log2 domain, then hide what the mask, the causal rule or the key tail hides
        const int code = tile_code(p, mb, qt0 + t, j);
        const int key0 = j * kBN;
        const bool dead = (code == TILE_SKIP) || i >= s.Sq;
        const bool full = !dead && code == TILE_OPEN && key0 >= key_lo && key0 + kBN - 1 <= key_hi;
        // x_e = log2(e) * (scale * s_e + bias_e), or -inf where the pair is hidden
        // first / last visible key of this row inside the tile (relative; lim < lo = none) from the
        // causal rule, the window and the key tail: integer compares per element on partial tiles
        int lo = 0, lim = 0;
        if (!full && !dead) {
          lo = (int)max(0LL, min(key_lo - key0, (long long)kBN));
          lim = (int)max(-1LL, min(key_hi - key0, (long long)kBN - 1));
        }
        // the whole score row of this tile in registers (one TMEM wait), masked and scaled in place
        float x[kBN];
        auto masked = [&](const uint32_t (&raw)[32], int c0) {
          if (!MASKED || full || dead || code != TILE_MIXED) {
            // full, dead and partial tiles share one copy of the unrolled scaling (code size matters
            // here); a dead or partial tile then hides the keys outside [lo, lim] of this 32-key chunk
#pragma unroll
            for (int e = 0; e < 32; ++e) x[c0 + e] = POS_SCALE ? __uint_as_float(raw[e]) : __uint_as_float(raw[e]) * sl2;
            if (!full) {
              const int a = max(lo - c0, 0), z = min(lim - c0 + 1, 32);
              const uint32_t vis = (dead || z <= a) ? 0u : (uint32_t)(((1ull << z) - 1ull) & ~((1ull << a) - 1ull));
#pragma unroll
              for (int e = 0; e < 32; ++e) x[c0 + e] = (vis >> e) & 1u ? x[c0 + e] : -CUDART_INF_F;
            }
          } else if (s.mask_kind == MK_ADD) {
            // the row's 32 mask values first (independent loads), then the arithmetic; 16-byte loads
            // when the chunk lies inside the row's visible keys and mask rows are 16-byte aligned
            const float* mp = static_cast<const float*>(p.mask) + mrow + key0 + c0;
            float mv[32];
            if (mask_vec && c0 >= lo && c0 + 31 <= lim) {
#pragma unroll
              for (int v4 = 0; v4 < 8; ++v4) {
                const float4 m4 = __ldg(reinterpret_cast<const float4*>(mp) + v4);
                mv[4 * v4] = m4.x; mv[4 * v4 + 1] = m4.y; mv[4 * v4 + 2] = m4.z; mv[4 * v4 + 3] = m4.w;
              }
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) mv[e] = (c0 + e >= lo && c0 + e <= lim) ? __ldg(mp + e) : -CUDART_INF_F;
            }
#pragma unroll
            for (int e = 0; e < 32; ++e)
              x[c0 + e] = (mv[e] > kMaskFloor) ? (POS_SCALE ? fmaf(mv[e], inv_scale, __uint_as_float(raw[e]))
                                                            : fmaf(__uint_as_float(raw[e]), sl2, mv[e] * kLog2e))
                                               : -CUDART_INF_F;
          } else {
            const uint8_t* mp = static_cast<const uint8_t*>(p.mask) + mrow + key0 + c0;
            uint32_t mb8[32];
            if (mask_vec && c0 >= lo && c0 + 31 <= lim) {
#pragma unroll
              for (int v = 0; v < 2; ++v) {
                const uint4 m16 = __ldg(reinterpret_cast<const uint4*>(mp) + v);
                const uint32_t w[4] = {m16.x, m16.y, m16.z, m16.w};
#pragma unroll
                for (int e = 0; e < 16; ++e) mb8[16 * v + e] = (w[e / 4] >> (8 * (e % 4))) & 0xffu;
              }
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) mb8[e] = (c0 + e >= lo && c0 + e <= lim) ? __ldg(mp + e) : 0u;
            }
#pragma unroll
            for (int e = 0; e < 32; ++e)
              x[c0 + e] = mb8[e] ? (POS_SCALE ? __uint_as_float(raw[e]) : __uint_as_float(raw[e]) * sl2) : -CUDART_INF_F;
          }
        };
        // (TMEM loads and stores are warp-collective: every lane issues them, hidden rows just get -inf)
        {
          uint32_t raw[2][32];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            tmem_ld32(tS + half * 64, raw[0]);
            tmem_ld32(tS + half * 64 + 32, raw[1]);
            tmem_wait_ld();
            reg_fence(raw[0]);
            reg_fence(raw[1]);
            masked(raw[0], half * 64);
            masked(raw[1], half * 64 + 32);
          }
        }
        float tm4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};  // 4 independent chains
#pragma unroll
        for (int e = 0; e < kBN; e += 2) tm4[(e >> 1) & 3] = max3f(tm4[(e >> 1) & 3], x[e], x[e + 1]);
        const float tmax_x = fmaxf(fmaxf(tm4[0], tm4[1]), fmaxf(tm4[2], tm4[3]));
        const float tmax = (POS_SCALE && tmax_x != -CUDART_INF_F) ? tmax_x * sl2 : tmax_x;
        const float m_new = fmaxf(m, tmax);
        const bool rescale = m_new > m + kRescaleThreshold;   // false while nothing is visible
        const float m_use = rescale ? m_new : m;
        const float alpha = rescale ? ex2_approx(m - m_new) : 1.f;
        const float m_sub = (m_use == -CUDART_INF_F) ? 0.f : m_use;
        // P = 2^(x - m) as bf16 over the first 64 columns of the score block (all scores are in registers);
        // the exponent's FMA (or subtraction) and the row sum on packed fp32 pairs: this loop is
        // issue-bound, and a pair instruction does the work of two
        const uint64_t sl2_2 = f32x2(sl2, sl2), negm_2 = f32x2(-m_sub, -m_sub);
        uint64_t sum2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
        for (int cch = 0; cch < kBN / 32; ++cch) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint64_t x2 = f32x2(x[cch * 32 + 2 * e], x[cch * 32 + 2 * e + 1]);
            float t0, t1;
            f32x2_split(POS_SCALE ? fma_f32x2(x2, sl2_2, negm_2) : add_f32x2(x2, negm_2), t0, t1);
            const float p0 = ex2_approx(t0);
            const float p1 = ex2_approx(t1);
            sum2[e & 1] = add_f32x2(sum2[e & 1], f32x2(p0, p1));
            pk[e] = pack_bf16x2(p0, p1);
          }
          tmem_st16(tS + cch * 16, pk);
        }
        float s0, s1, s2, s3;
        f32x2_split(sum2[0], s0, s1);
        f32x2_split(sum2[1], s2, s3);
        const float sum = (s0 + s1) + (s2 + s3);
        l = l * alpha + sum;
        m = m_use;
        if (__any_sync(0xffffffffu, rescale) && idx > 0) {  // alpha = 1 on rows that keep their max
          // O already holds P V of the earlier tiles (their MMAs finished before these scores did).
#pragma unroll
          for (int cch = 0; cch < D / 32; ++cch) {
            uint32_t ov[32];
            tmem_ld32(tO + cch * 32, ov);
            tmem_wait_ld();
            reg_fence(ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(tO + cch * 32, ov);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_p[t]);
        ++idx;
        ++gidx;
      }
      // ---- epilogue: O = acc / l, LSE = (m + log2 l) ln 2; a row with nothing visible gets 0 and 0
      ok = __all_sync(0xffffffffu, ok);
      if (ok && idx > 0) ok = __all_sync(0xffffffffu, mbar_wait<true>(&bar_o[t], n_o & 1, abort_flag, p.status, 21));
      if (idx > 0) ++n_o;
      tc_fence_after();
      const bool row_ok = i < s.Sq;
      const size_t row = (size_t)u.bh * s.Sq + (row_ok ? i : 0);
      const bool alive = l > 0.f;
      if (PERSIST || p.kv_splits == 1) {   // a persistent grid never splits the keys
        // The tile's O rows in bf16 go to its Q buffer, in the 128-byte-swizzled layout of the O
        // tensor map, and leave in one TMA store per 64-column box (rows past Sq are clipped by the
        // map). The buffer is free: the tile's last S MMAs completed before its last PV MMA (bar_o);
        // with no visible key tile, once the Q load itself has landed.
        if (ok) {
          const float inv = alive ? 1.f / l : 0.f;
          if (idx == 0) mbar_wait<true>(&bar_q[PERSIST ? t : 0], PERSIST ? ui & 1 : 0, nullptr, p.status, 22);
          const uint32_t sO = smem_u32(sQ + t * L::kTileBytes) + r * 128;
#pragma unroll
          for (int cch = 0; cch < D / 32; ++cch) {
            uint32_t ov[32];
            if (idx > 0) {
              tmem_ld32(tO + cch * 32, ov);
              tmem_wait_ld();
              reg_fence(ov);
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] = 0u;
            }
            uint32_t pkd[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pkd[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              const int c16 = (cch & 1) * 4 + v4;   // 16-byte chunk of the row inside its box
              st_shared_v4(sO + (cch >> 1) * L::kBoxBytes + ((c16 ^ (r & 7)) << 4), pkd[4 * v4], pkd[4 * v4 + 1],
                           pkd[4 * v4 + 2], pkd[4 * v4 + 3]);
            }
          }
        }
        fence_proxy_async_smem();
        // all four warps of the warpgroup, whatever `ok` says; in a persistent grid they leave with one
        // shared answer, so they run the same units and meet here equally often
        if constexpr (PERSIST)
          ok = named_bar_and(1 + t, 128, ok);
        else
          named_bar_sync(1 + t, 128);
        if (wq == 0 && lane == 0) {
          if (ok && u.q_row0 + t * kBM < s.Sq) {
            for (int box = 0; box < D / 64; ++box)
              tma_store_4d(&p.tm_o, sQ + t * L::kTileBytes + box * L::kBoxBytes, box * 64, u.q_row0 + t * kBM, u.h,
                           u.b);
            bulk_commit_group();
            bulk_wait_group_read0();   // the shared-memory source must outlive the reads
          }
          if (PERSIST) mbar_arrive(&bar_qfree[t]);   // the buffer may take the next unit's Q
        }
        if (ok && row_ok) p.lse[row] = alive ? (m + __log2f(l)) * kLn2 : 0.f;
      } else if (ok) {
        const size_t rows = (size_t)s.B * s.Hq * s.Sq;
        float4* dst = reinterpret_cast<float4*>(p.part_o + ((size_t)u.split * rows + row) * D);
#pragma unroll
        for (int cch = 0; cch < D / 32; ++cch) {
          uint32_t ov[32];
          if (idx > 0) {
            tmem_ld32(tO + cch * 32, ov);
            tmem_wait_ld();
            reg_fence(ov);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = 0u;
          }
          if (row_ok) {
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              dst[cch * 8 + v4] = make_float4(__uint_as_float(ov[4 * v4]), __uint_as_float(ov[4 * v4 + 1]),
                                              __uint_as_float(ov[4 * v4 + 2]), __uint_as_float(ov[4 * v4 + 3]));
          }
        }
        if (row_ok) {
          float2* ml = reinterpret_cast<float2*>(p.part_ml + ((size_t)u.split * rows + row) * 2);
          *ml = make_float2(alive ? m : -CUDART_INF_F, l);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge split-KV partials: m = max m_s, l = sum l_s 2^(m_s - m), O = sum O_s 2^(m_s - m) / l.
template <int D>
__global__ void __launch_bounds__(256) fwd_combine_kernel(const float* __restrict__ part_o,
                                                          const float* __restrict__ part_ml, int splits,
                                                          long long rows, __nv_bfloat16* __restrict__ o,
                                                          float* __restrict__ lse, const Shape s) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  constexpr int E = D / 32;
  float mmax = -CUDART_INF_F;
  for (int sp = 0; sp < splits; ++sp) mmax = fmaxf(mmax, part_ml[((size_t)sp * rows + row) * 2]);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float l = 0.f;
  if (mmax != -CUDART_INF_F) {
    for (int sp = 0; sp < splits; ++sp) {
      const float ms = part_ml[((size_t)sp * rows + row) * 2];
      if (ms == -CUDART_INF_F) continue;
      const float w = ex2_approx(ms - mmax);
      l += part_ml[((size_t)sp * rows + row) * 2 + 1] * w;
      const float* src = part_o + ((size_t)sp * rows + row) * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] += src[e] * w;
    }
  }
  const bool alive = l > 0.f;
  const float inv = alive ? 1.f / l : 0.f;
  const long long bh = row / s.Sq, i = row % s.Sq;   // rows run over [B, Hq, Sq] like LSE
  __nv_bfloat16* dst = o + head_base(s, (int)(bh / s.Hq), (int)(bh % s.Hq), s.Hq, s.Sq) + (size_t)i * row_stride(s, s.Hq) +
                       lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) dst[e] = __float2bfloat16_rn(acc[e] * inv);
  if (lane == 0) lse[row] = alive ? (mmax + __log2f(l)) * kLn2 : 0.f;
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int n_qpairs(const Shape& s) { return (s.Sq + kRowsPerCta - 1) / kRowsPerCta; }

int kv_tiles_total(const Shape& s) {
  long long kv_end = s.Sk;
  if (s.causal) kv_end = min(kv_end, s.q_offset + s.Sq);
  int n = (int)((kv_end + kBN - 1) / kBN);
  // a window confines a CTA's rows to a band of 2w + kRowsPerCta keys
  if (s.window > 0) n = (int)min((long long)n, (2LL * s.window + kRowsPerCta + kBN - 1) / kBN + 1);
  return n;
}

}  // namespace

static EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn encode = nullptr;
  if (encode == nullptr) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) return nullptr;
    encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return encode;
}

// bf16 [heads, S, D] tensor viewed as (D, S, heads), boxes of 64 x box_rows x 1 with 128-byte swizzle.
cudaError_t make_tmap_4d(CUtensorMap* map, const void* base, int layout, int B, int H, int S, int D, int box_rows) {
  EncodeTiledFn encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t row = (cuuint64_t)D * 2, e = 2;
  // byte strides of the S, H and B dimensions
  const cuuint64_t strides[3] = {layout ? (cuuint64_t)H * D * e : row, layout ? row : (cuuint64_t)S * D * e,
                                 (cuuint64_t)S * H * D * e};
  const cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// fp32 [heads, S, D] tensor viewed as (D, S, heads), unswizzled boxes of D x box_rows x 1.
cudaError_t make_tmap_f32_bhsd(CUtensorMap* map, const void* base, int S, int heads, int D, int box_rows) {
  EncodeTiledFn encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)heads};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)S * D * 4};
  const cuuint32_t box[3] = {(cuuint32_t)D, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// fp32 [heads, S, D] tensor viewed as (D, S, heads), boxes of 32 x box_rows x 1 (128-byte rows) with
// 128-byte swizzle: a 32-feature slice of a query tile, staged conflict-free in shared memory.
cudaError_t make_tmap_f32_bhsd_sw128(CUtensorMap* map, const void* base, int S, int heads, int D, int box_rows) {
  EncodeTiledFn encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)heads};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)S * D * 4};
  const cuuint32_t box[3] = {32, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

bool tc_fwd_supported(const Shape& s) { return (s.D == 64 || s.D == 128) && s.Sq > 0; }

int tc_fwd_kv_splits(const Shape& s) {
  const long long units = (long long)s.B * s.Hq * n_qpairs(s);
  const int sms = sm_count();
  if (units >= sms) return 1;
  const int by_waves = (int)((4LL * sms) / units);
  const int by_len = kv_tiles_total(s) / 8;
  return max(1, min(by_waves, by_len));
}

FwdLaunch tc_fwd_launch(const Shape& s, int kv_splits) {
  const long long units = (long long)s.B * s.Hq * n_qpairs(s);
  // Persistent CTAs (more units than SMs) chain their units' key tiles, which needs a key tile in
  // every unit: no split and no mask (whose tile map may skip all of a unit's tiles); a row sees at
  // least its own diagonal key (q_offset + Sq <= Sk), so the range check below only guards that.
  FwdLaunch l;
  l.persistent = kv_splits == 1 && s.mask_kind == MK_NONE && units > sm_count();
  FwdTcParams kp;
  kp.s = s;
  kp.kv_splits = 1;
  for (int qp = 0; qp < n_qpairs(s) && l.persistent; ++qp) {
    const KvRange kr = kv_range(kp, qp * kRowsPerCta, 0);
    if (kr.end <= kr.begin) l.persistent = false;
  }
  l.ctas = l.persistent ? (long long)sm_count() : units * kv_splits;
  return l;
}

template <int D>
static cudaError_t tc_fwd_t(const FwdArgs& a, const FwdPlan& plan, char* ws, unsigned* status) {
  const Shape& s = a.s;
  FwdTcParams p;
  cudaError_t e;
  const int kvl = a.kv_layout >= 0 ? a.kv_layout : s.layout;
  if ((e = make_tmap_4d(&p.tm_q, a.q, s.layout, s.B, s.Hq, s.Sq, D, kBM)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&p.tm_k, a.k, kvl, s.B, s.Hkv, s.Sk, D, kBN)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&p.tm_v, a.v, kvl, s.B, s.Hkv, s.Sk, D, kBN)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&p.tm_o, a.o, s.layout, s.B, s.Hq, s.Sq, D, kBM)) != cudaSuccess) return e;
  p.s = s;
  p.mask = a.mask;
  p.nqt = (s.Sq + kBM - 1) / kBM;
  p.nkt = (s.Sk + kBN - 1) / kBN;
  p.tilemap = nullptr;
  if (s.mask_kind != MK_NONE) {
    uint8_t* tm = reinterpret_cast<uint8_t*>(ws + plan.tilemap_off);
    if ((e = launch_mask_classify(s, a.mask, tm, a.stream)) != cudaSuccess) return e;
    p.tilemap = tm;
  }
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.kv_splits = plan.kv_splits;
  p.part_o = plan.kv_splits > 1 ? reinterpret_cast<float*>(ws + plan.part_o_off) : nullptr;
  p.part_ml = plan.kv_splits > 1 ? reinterpret_cast<float*>(ws + plan.part_ml_off) : nullptr;
  p.n_qpairs = n_qpairs(s);
  p.status = status;
  const FwdLaunch launch = tc_fwd_launch(s, plan.kv_splits);
  const bool persistent = launch.persistent;
  const int smem = FwdSmem<D>::kBytes;
  const bool pos = s.scale > 0.f;
  auto kernel = s.mask_kind != MK_NONE
                    ? (pos ? fwd_tc_kernel<D, true, true, false> : fwd_tc_kernel<D, true, false, false>)
                    : persistent ? (pos ? fwd_tc_kernel<D, false, true, true> : fwd_tc_kernel<D, false, false, true>)
                                 : (pos ? fwd_tc_kernel<D, false, true, false> : fwd_tc_kernel<D, false, false, false>);
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
    return e;
  const long long ctas = launch.ctas;
  if ((e = prof_begin(KID_FWD, a.stream)) != cudaSuccess) return e;
  kernel<<<(unsigned)ctas, kThreads, smem, a.stream>>>(p);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (plan.kv_splits > 1) {
    const long long rows = (long long)s.B * s.Hq * s.Sq;
    fwd_combine_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, a.stream>>>(p.part_o, p.part_ml, plan.kv_splits,
                                                                            rows, p.o, p.lse, s);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return prof_end(KID_FWD, a.stream);
}

cudaError_t tc_fwd(const FwdArgs& a, const FwdPlan& plan, char* ws) {
  unsigned* status = device_status_ptr();
  if (status == nullptr) return cudaErrorUnknown;
  return a.s.D == 64 ? tc_fwd_t<64>(a, plan, ws, status) : tc_fwd_t<128>(a, plan, ws, status);
}

}  // namespace fa
