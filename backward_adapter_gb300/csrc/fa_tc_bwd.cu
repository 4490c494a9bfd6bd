// Backward of the fused attention training op on the 5th-generation tensor
// cores (tcgen05, sm_103a). With P recomputed from LSE, D_i = <dO_i, O_i>
// precomputed, and dS = P (dP - D) (llama.cpp PR #57, commit 86c140d:
// "LSE, D, then grads per tile; GQA group-sum"):
//     dV_j = sum_{h in group} sum_i P_ij dO_i
//     dK_j = scale sum_{h in group} sum_i dS_ij q_i
//     dQ_i = scale sum_j dS_ij k_j
//
// One CTA owns a 128-key tile of one (batch, key/value head). Its dK and dV
// live in TMEM for the whole walk (no atomics on them: the ownership split is by
// key tile), while it walks every query tile of every query head of the GQA
// group that can see its keys. Per step (BQ query rows):
//     S^T  = K Q^T           (SMEM x SMEM -> TMEM)       keys are TMEM lanes
//     dP^T = V dO^T          (SMEM x SMEM -> TMEM)
//     softmax-grad warps: P^T = 2^(S^T scale log2e + bias - LSE log2e), 0 where hidden;
//                         dS^T = P^T (dP^T - D); P^T, dS^T -> TMEM (bf16), dS^T -> SMEM
//     dV  += P^T dO          (TMEM x SMEM)
//     dK  += dS^T Q          (TMEM x SMEM)
//     dQ  = dS K             (SMEM x SMEM -> TMEM)       query rows are TMEM lanes
//     the dQ partial is added into the fp32 dQ accumulator in L2.
// Roles: warp 0 TMA (K, V once; Q, dO per step), warp 1 MMA issue + TMEM owner,
// warp 2 LSE/D staging, warps 4-11 softmax-grad: two warps per TMEM lane quadrant,
// a thread owns one key and a share of the step's query columns; warps 12-15 move
// each step's dQ partial out of TMEM and add it into the accumulator. Each 32-column
// score chunk receives its own P^T (16 columns) and dS^T (16 columns) once read, so no
// warp writes TMEM another warp still reads.
//
// Each step's softmax-grad is split in two rounds of 64 queries; the first round's
// dV / dK MMAs run while the second round is computed. S^T and dP^T complete on separate
// barriers, so the first round's exponentials run under the dP^T MMAs.
// The dQ partial is staged in the step's consumed Q/dO slot (128-byte swizzled 32-feature
// sub-tiles) and added with TMA bulk tensor reduce-adds issued by one thread, which then hands
// the slot back to the producer: per-element red.add from the stager warps took issue slots
// from the softmax-grad warps sharing their sub-partitions.
#include <cuda.h>
#include <cstring>
#include <cmath>
#include <algorithm>
#include <climits>
#include <functional>
#include <queue>
#include <set>
#include <vector>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "fa_device.cuh"
#include "fa_internal.h"
#include "kv_q8.cuh"
#include "tc_ptx.cuh"

namespace fa {
namespace {

using namespace tc;

constexpr int kBN = 128;       // keys per CTA
constexpr int kThreads = 512;  // 16 warps = 4 warpgroups (128 registers per thread at launch)
// Register split by warpgroup (setmaxnreg, inside each role's branch): control warps 0-3 drop to
// 64, the softmax-grad warpgroups take 144 (a 32-query chunk of scores and of dP^T at once), the
// dQ stager (warps 12-15) 160 so it can hold a whole dQ partial row:
// (64 + 144 + 144 + 160) x 128 = 65536 = 512 x 128.
constexpr int kRegsControl = 64;
constexpr int kRegsSoftmax = 144;
constexpr int kRegsStager = 160;
static_assert(kRegsControl + 2 * kRegsSoftmax + kRegsStager <= 4 * 128, "register split exceeds the launch pool");
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int BQ = 128;                        // query rows per step (N = 128 MMAs)
  static constexpr int NBUF = 1;                        // S/dP TMEM blocks
  static constexpr int BUF_COLS = 2 * BQ;               // block b: S^T [b*2BQ, +BQ), dP^T [b*2BQ+BQ, +BQ)
  static constexpr int NCHUNK = BQ / 32;                // 32-column score chunks per step
  static constexpr int CHUNKS_PER_WARP = NCHUNK / 2;    // two warps per lane quadrant
  static constexpr bool TWO_ROUND = CHUNKS_PER_WARP == 2;   // the first 64 queries' dV / dK go early
  // chunk c of the scores (columns [32c, 32c+32)) is overwritten by P^T at [32c, 32c+16)
  // and dS^T at [32c+16, 32c+32) (bf16 pairs) once it has been read
  static constexpr int DQ_COL = BQ;                     // dQ (lanes = query rows) over the dP^T block
  static constexpr int DV_COL = 256;
  static constexpr int DK_COL = 256 + D;
  static constexpr int DQ_CHUNKS = D / 32;             // 32-column TMEM chunks of the dQ partial
  static constexpr int NSTAGE = 2;                      // Q/dO ring depth
  static constexpr int NDS = 1;                         // dS^T shared-memory buffers (the dQ MMA of a
                                                        // step completes before the next dS^T is written)
  // shared memory (bytes)
  static constexpr int KV_BOX = 128 * 128;              // 128 rows x 128 B
  static constexpr int KV_TILE = kBN * D * 2;
  static constexpr int QBOX = BQ * 128;                 // BQ rows x 128 B
  static constexpr int Q_TILE = BQ * D * 2;
  static constexpr int DS_BLOCK = 128 * 128;            // 128 keys x 64 queries (bf16)
  static constexpr int DS_TILE = (BQ / 64) * DS_BLOCK;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = KV_TILE;
  // [NSTAGE] x (Q, dO); once dV/dK of a step have read its slot, the slot holds that step's
  // fp32 dQ partial ([BQ][D] = 2 * Q_TILE bytes) until the reduce-add has read it
  static constexpr int OFF_STAGE = 2 * KV_TILE;
  static constexpr int OFF_DS = OFF_STAGE + NSTAGE * 2 * Q_TILE;   // [NDS] x dS^T (operand of the dQ MMA)
  static constexpr int OFF_LSED = OFF_DS + NDS * DS_TILE;          // [NSTAGE] x (-lse2[BQ], dsum[BQ])
  static constexpr int OFF_BAR = OFF_LSED + NSTAGE * 2 * BQ * 4;
  static constexpr int BYTES = OFF_BAR + 512;
  static_assert(BQ * D * 4 <= 2 * Q_TILE, "dQ partial fits its stage slot");
  static_assert(NBUF * BUF_COLS + 2 * D <= 512, "TMEM columns");
  static_assert(BYTES <= 232448, "shared memory per block");
};

struct BwdTcParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do, tm_dq;
  Shape s;
  const void* mask;
  const uint8_t* tilemap;
  const float* lse;
  const float* dsum;
  float* dq_acc;
  void* dk;  // bf16 [B,Hkv,Sk,D], or fp32 accumulator
  void* dv;
  int accum;
  int* turn;              // deterministic: int32 [B, Hq, nqt] turn counters (zeroed before launch)
  int q8;                 // q8_0 K/V cache: the softmax-grad warps dequantize the CTA's K, V tiles
  const int8_t* kq;
  const __half* kd;
  const int8_t* vq;
  const __half* vd;
  long long rows_begin;   // accumulate: keys [rows_begin, rows_begin + n_rows) are also written, after
  int n_rows;             // the add, to dk_rows / dv_rows (bf16 [B, Hkv, n_rows, D])
  __nv_bfloat16* dk_rows;
  __nv_bfloat16* dv_rows;
  int nqt, nkt;
  unsigned* status;
  // work units (see BwdSplit): n_units == 0 runs one CTA per key tile in key-tile order
  int n_units, n_slots, n_ctas;
  float* part;                  // fp32 dV/dK partials of split key tiles [B * Hkv, n_slots, 2, D / 4, 128] float4
  int* part_sync;               // per (batch, kv head, first slot of a split key tile): tickets, partials written
  uint32_t units[kMaxUnits];    // kt | part << 12 | nparts << 16 | slot << 20
  uint32_t range[kMaxUnits];    // a part's query tiles from the key tile's first: first | end << 16
  uint32_t ctas[kMaxCtas];      // n_ctas > 0: CTA i runs unit ctas[i] & 0xffff of (batch, kv head) ctas[i] >> 16
};

// Query rows [ibeg, iend) that can see a key of tile kt, from the causal rule and the window, with
// ibeg rounded down to a multiple of BQ (shared by the kernel and the host's work planner).
__host__ __device__ inline void key_tile_rows(const Shape& s, int kt, int BQ, int& ibeg, int& iend) {
  const int j0 = kt * kBN;
  long long first = 0, last = (long long)s.Sq - 1;
  if (s.causal) first = (long long)j0 - s.q_offset;
  if (s.window > 0) {
    if (!s.causal) first = (long long)j0 - s.q_offset - s.window;
    last = min(last, (long long)j0 + kBN - 1 - s.q_offset + s.window);
  }
  ibeg = first <= 0 ? 0 : (int)min((first / BQ) * BQ, (long long)s.Sq);
  iend = (int)max((long long)ibeg, last + 1);
}

// The steps of a CTA: (query head of the group, query tile) pairs in a fixed order; the tiles
// run over the rows [ibeg, iend) that can see the CTA's keys. Head-major with ascending tiles by
// default; with tile_major (deterministic dQ) descending tiles with every head of the group at
// each tile, so that all key tiles reach a given query tile at about the same step.
struct StepIter {
  int G, iend, BQ, ibeg, last;
  bool tile_major;
  int hh, i0;
  __device__ void init(int G_, int iend_, int BQ_, int ibeg_, bool tile_major_) {
    G = G_; iend = iend_; BQ = BQ_; ibeg = ibeg_; tile_major = tile_major_;
    last = ibeg < iend ? ibeg + ((iend - 1 - ibeg) / BQ) * BQ : ibeg;
    hh = 0; i0 = tile_major ? last : ibeg;
  }
  __device__ bool valid() const { return ibeg < iend && (tile_major ? i0 >= ibeg : hh < G); }
  __device__ void next() {
    if (tile_major) {
      if (++hh == G) { hh = 0; i0 -= BQ; }
    } else {
      i0 += BQ;
      if (i0 >= iend) { i0 = ibeg; ++hh; }
    }
  }
};

__device__ __forceinline__ int bwd_tile_code(const BwdTcParams& p, int mb, int i0, int kt) {
  if (p.tilemap == nullptr) return TILE_OPEN;
  return p.tilemap[((size_t)mb * p.nqt + i0 / 128) * p.nkt + kt];
}

// MASKED: the call has a mask tensor. Without one no tile is mixed, and that instance has no
// mixed-tile code at all: the softmax-grad loop's unrolled variants compete for the instruction
// cache with every other role's loop, and the unused one cost 3% of the causal backward.
template <int D, bool MASKED, bool DET>
__global__ void __launch_bounds__(kThreads, 1) bwd_tc_kernel(const __grid_constant__ BwdTcParams p) {
  using C = BwdCfg<D>;
  constexpr int BQ = C::BQ;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  // the 128-byte swizzle of TMA and of the MMA descriptors assumes 1024-byte aligned tiles
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, 0x80000000u | 199u);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* bar_kv = bars;                              // 1
  uint64_t* bar_qdo_full = bar_kv + 1;                  // NSTAGE
  uint64_t* bar_qdo_empty = bar_qdo_full + C::NSTAGE;   // NSTAGE
  uint64_t* bar_lsed_full = bar_qdo_empty + C::NSTAGE;  // NSTAGE
  uint64_t* bar_lsed_empty = bar_lsed_full + C::NSTAGE; // NSTAGE
  uint64_t* bar_sdp_full = bar_lsed_empty + C::NSTAGE;  // NBUF
  uint64_t* bar_p_full = bar_sdp_full + C::NBUF;        // NBUF
  uint64_t* bar_p_half = bar_p_full + C::NBUF;          // 1: P^T / dS^T of the step's first 64 queries
  uint64_t* bar_dq_full = bar_p_half + 1;               // NBUF
  uint64_t* bar_dq_free = bar_dq_full + C::NBUF;        // NBUF
  uint64_t* bar_mma_done = bar_dq_free + C::NBUF;       // 1
  uint64_t* bar_stage_full = bar_mma_done + 1;          // 1: the 4 stager warps filled the dQ staging
  uint64_t* bar_s_full = bar_stage_full + 1;            // NBUF: S^T of the block is in TMEM
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_s_full + C::NBUF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_part = abort_flag + 1;   // split key tile: this CTA's part finished last
  volatile int* parts_ready = abort_flag + 2; // ... and the other parts' partials are written
  float* lsed = reinterpret_cast<float*>(smem + C::OFF_LSED);

  const Shape& s = p.s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = s.Hq / s.Hkv;

  // ---- work unit: key tile kt of (b, kvh), or a part of it (consecutive query tiles). Without a
  //      plan, blocks run key-tile-major: under the causal rule the low key tiles carry the most
  //      work, so every head's heavy tiles are in the first wave and the light ones fill the SMs
  //      that free up. With a plan (see plan_bwd_split) the host lists the units per block in the
  //      order that packs them onto the SMs.
  const int nbkv = s.B * s.Hkv;
  int unit = blockIdx.x / nbkv, bkv = blockIdx.x % nbkv;
  if (p.n_ctas > 0) {   // the planned launch order
    const uint32_t c = p.ctas[blockIdx.x];
    unit = (int)(c & 0xffffu);
    bkv = (int)(c >> 16);
  }
  int kt = unit, part = 0, nparts = 1, slot = 0;
  uint32_t range = 0;
  if (p.n_units > 0) {
    const uint32_t u = p.units[unit];
    kt = (int)(u & 0xfffu);
    part = (int)((u >> 12) & 0xfu);
    nparts = (int)((u >> 16) & 0xfu);
    slot = (int)(u >> 20);
    range = p.range[unit];
  }
  const int b = bkv / s.Hkv, kvh = bkv % s.Hkv;
  const int j0 = kt * kBN;
  const int mb = s.mask_batch > 1 ? b : 0;
  int ibeg, iend;
  key_tile_rows(s, kt, BQ, ibeg, iend);
  if (nparts > 1) {   // the part's own query tiles
    const int base = ibeg;
    ibeg = base + (int)(range & 0xffffu) * BQ;
    iend = min(iend, base + (int)(range >> 16) * BQ);
  }

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, p.q8 ? 8 : 1);   // q8: one arrival per softmax-grad warp after dequantizing
    for (int i = 0; i < C::NSTAGE; ++i) {
      mbar_init(&bar_qdo_full[i], 1);
      mbar_init(&bar_qdo_empty[i], 1);
      mbar_init(&bar_lsed_full[i], 1);
      mbar_init(&bar_lsed_empty[i], 8);
    }
    for (int i = 0; i < C::NBUF; ++i) {
      mbar_init(&bar_sdp_full[i], 1);
      mbar_init(&bar_s_full[i], 1);
      mbar_init(&bar_p_full[i], 8);
      mbar_init(&bar_dq_full[i], 1);
      mbar_init(&bar_dq_free[i], 4);
    }
    mbar_init(bar_p_half, 8);
    mbar_init(bar_mma_done, 1);
    mbar_init(bar_stage_full, 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto step_skipped = [&](const StepIter& it) { return bwd_tile_code(p, mb, it.i0, kt) == TILE_SKIP; };
  auto count_steps = [&]() {
    int n = 0;
    StepIter it;
    it.init(G, iend, BQ, ibeg, DET);
    for (; it.valid(); it.next())
      if (!step_skipped(it)) ++n;
    return n;
  };

  if (warp < 4) {
   regs_dec<kRegsControl>();   // all four warps of the control warpgroup
   if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tmap(&p.tm_q);
      prefetch_tmap(&p.tm_do);
      prefetch_tmap(&p.tm_dq);
      if (!p.q8) {
        prefetch_tmap(&p.tm_k);
        prefetch_tmap(&p.tm_v);
        mbar_arrive_expect_tx(bar_kv, 2 * C::KV_TILE);
        for (int box = 0; box < D / 64; ++box) {
          tma_load_4d(smem + C::OFF_K + box * C::KV_BOX, &p.tm_k, bar_kv, box * 64, j0, kvh, b);
          tma_load_4d(smem + C::OFF_V + box * C::KV_BOX, &p.tm_v, bar_kv, box * 64, j0, kvh, b);
        }
      }
      // the stager hands a slot back once the dQ partial staged in it has been reduced
      uint32_t used_mask = 0, phase_mask = 0;
      StepIter it;
      it.init(G, iend, BQ, ibeg, DET);
      for (int st = 0; it.valid(); it.next()) {
        if (step_skipped(it)) continue;
        const int slot = st % C::NSTAGE;
        const uint32_t ph = (st / C::NSTAGE) & 1;
        if (!mbar_wait(&bar_qdo_empty[slot], ph ^ 1, abort_flag, p.status, 101)) break;
        mbar_arrive_expect_tx(&bar_qdo_full[slot], 2 * C::Q_TILE);
        uint8_t* sq = smem + C::OFF_STAGE + slot * 2 * C::Q_TILE;
        const int qh = kvh * G + it.hh;   // query head
        for (int box = 0; box < D / 64; ++box) {
          tma_load_4d(sq + box * C::QBOX, &p.tm_q, &bar_qdo_full[slot], box * 64, it.i0, qh, b);
          tma_load_4d(sq + C::Q_TILE + box * C::QBOX, &p.tm_do, &bar_qdo_full[slot], box * 64, it.i0, qh, b);
        }
        used_mask |= 1u << slot;
        phase_mask = (phase_mask & ~(1u << slot)) | (ph << slot);
        ++st;
      }
      // drain every copy this thread issued
      mbar_wait(bar_kv, 0, nullptr, p.status, 102);
      for (int i = 0; i < C::NSTAGE; ++i)
        if (used_mask >> i & 1u) mbar_wait(&bar_qdo_full[i], (phase_mask >> i) & 1u, nullptr, p.status, 103);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, BQ, 0, 0);        // S^T, dP^T
      const uint32_t idesc_g = idesc_bf16_f32(128, D, 0, 1);         // dV, dK (B = dO / Q, MN-major)
      const uint32_t idesc_q = idesc_bf16_f32(128, D, 1, 1);         // dQ = dS K
      const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
      bool ok = mbar_wait(bar_kv, 0, abort_flag, p.status, 110);
      tc_fence_after();

      // Base descriptors per operand tile; every k-step adds a compile-time byte offset (desc_add).
      const uint64_t dK0 = smem_desc_sw128(sK, 16, 1024), dV0 = smem_desc_sw128(sV, 16, 1024);
      const uint64_t dKmn = smem_desc_sw128(sK, C::KV_BOX, 1024);   // K as an MN-major operand
      // S^T of step st into score block st % NBUF: the block's previous contents (P^T, dS^T of
      // step st - NBUF) were consumed by the dV / dK MMAs issued before (tcgen05 MMAs of a
      // thread run in order)
      auto issue_st = [&](int st) {
        const int slot = st % C::NSTAGE;
        tc_fence_after();
        const uint32_t tb = tmem + (st % C::NBUF) * C::BUF_COLS;
        const uint64_t dq0 = smem_desc_sw128(smem_u32(smem + C::OFF_STAGE + slot * 2 * C::Q_TILE), 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tb, desc_add(dK0, (k / 4) * C::KV_BOX + (k % 4) * 32), desc_add(dq0, (k / 4) * C::QBOX + (k % 4) * 32),
                 idesc_s, k > 0);
        mma_commit(&bar_s_full[st % C::NBUF]);   // the softmax-grad warps start on P^T under dP^T
      };
      // dP^T of step st: its TMEM block held the dQ partial of step st - NBUF, drained by the stager
      auto issue_dp = [&](int st) {
        const int slot = st % C::NSTAGE;
        tc_fence_after();
        const uint32_t tb = tmem + (st % C::NBUF) * C::BUF_COLS;
        const uint64_t ddo0 =
            smem_desc_sw128(smem_u32(smem + C::OFF_STAGE + slot * 2 * C::Q_TILE) + C::Q_TILE, 16, 1024);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          mma_ss(tb + BQ, desc_add(dV0, (k / 4) * C::KV_BOX + (k % 4) * 32),
                 desc_add(ddo0, (k / 4) * C::QBOX + (k % 4) * 32), idesc_s, k > 0);
        mma_commit(&bar_sdp_full[st % C::NBUF]);
      };
      // dV, dK over the step's queries [64h, 64h + 64) (all BQ queries when BQ = 64): k-step k
      // covers queries [16k, 16k+16), score chunk k/2, columns (k%2)*8 within its P^T / dS^T half
      auto issue_dvdk = [&](int st, int h) {
        const int slot = st % C::NSTAGE;
        tc_fence_after();
        const uint32_t tb = tmem + (st % C::NBUF) * C::BUF_COLS;
        const uint32_t sq = smem_u32(smem + C::OFF_STAGE + slot * 2 * C::Q_TILE);
        const uint64_t dqmn = smem_desc_sw128(sq, C::QBOX, 1024), ddomn = smem_desc_sw128(sq + C::Q_TILE, C::QBOX, 1024);
        constexpr int KS = C::TWO_ROUND ? BQ / 32 : BQ / 16;   // k-steps per call
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int k = h * KS + kk;
          mma_ts(tmem + C::DV_COL, tb + 32 * (k / 2) + (k % 2) * 8, desc_add(ddomn, k * 2048), idesc_g,
                 (st > 0 || k > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int k = h * KS + kk;
          mma_ts(tmem + C::DK_COL, tb + 32 * (k / 2) + 16 + (k % 2) * 8, desc_add(dqmn, k * 2048), idesc_g,
                 (st > 0 || k > 0) ? 1u : 0u);
        }
      };
      // dQ of step st (all of its dS^T is in shared memory), over the step's dP^T columns
      auto issue_dq = [&](int st) {
        const uint32_t tb = tmem + (st % C::NBUF) * C::BUF_COLS;
        const uint64_t ds0 =
            smem_desc_sw128(smem_u32(smem + C::OFF_DS + (st % C::NDS) * C::DS_TILE), C::DS_BLOCK, 1024);
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k) {
          mma_ss(tb + C::DQ_COL, desc_add(ds0, k * 2048), desc_add(dKmn, k * 2048), idesc_q, k > 0);
        }
        mma_commit(&bar_dq_full[st % C::NBUF]);   // also frees the dS^T tile
      };

      // Issue whichever MMA group is ready; none that waits holds back one that is ready. With one
      // S/dP block (D = 64):
      //   dV/dK of step ns, first 64 queries: once their P^T / dS^T are written;
      //   dV/dK of the other 64 queries and dQ of step ns: once all of its P^T / dS^T are written;
      //   dP^T of step np: after S^T(np) and once the stager drained the dQ partial of step np-1;
      //   S^T of step nt: after its Q / dO are loaded and step nt-1 was issued completely.
      // The issue order of the groups that accumulate (dV, dK) is fixed, so they are bitwise
      // reproducible.
      const int total = count_steps();
      int nt = 0, np = 0, ns = 0, na = 0;   // na: steps whose first-half dV/dK are issued
      unsigned long long idle_since = globaltimer();
      while (ok && ns < total) {
        bool progressed = false;
        if (na == ns && ns < np && mbar_test(bar_p_half, ns & 1)) {
          issue_dvdk(ns, 0);
          ++na;
          progressed = true;
        } else if (na > ns && mbar_test(&bar_p_full[0], ns & 1)) {
          issue_dvdk(ns, 1);
          issue_dq(ns++);
          progressed = true;
        } else if (np < nt && (np == 0 || mbar_test(&bar_dq_free[0], (np - 1) & 1))) {
          issue_dp(np++);
          progressed = true;
        } else if (nt < total && nt == ns && mbar_test(&bar_qdo_full[nt % C::NSTAGE], (nt / C::NSTAGE) & 1)) {
          issue_st(nt++);
          progressed = true;
        }
        if (progressed) {
          idle_since = globaltimer();
        } else if (*abort_flag) {
          ok = false;
        } else if ((__nanosleep(80), globaltimer() - idle_since > kWaitLimitNs)) {
          *abort_flag = 1;
          atomicCAS(p.status, 0u, 0x80000000u | 111u);
          ok = false;
        }
      }
      mma_commit(bar_mma_done);
      mbar_wait(bar_mma_done, 0, nullptr, p.status, 114);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- LSE / D staging
    StepIter it;
    it.init(G, iend, BQ, ibeg, DET);
    const float l2e = kLog2e;
    for (int st = 0; it.valid(); it.next()) {
      if (step_skipped(it)) continue;
      const int slot = st % C::NSTAGE;
      if (!__all_sync(0xffffffffu, mbar_wait(&bar_lsed_empty[slot], ((st / C::NSTAGE) & 1) ^ 1, abort_flag, p.status,
                                              120)))
        break;
      const size_t rowbase = (size_t)(b * s.Hq + kvh * G + it.hh) * s.Sq;
      float* dst = lsed + slot * 2 * BQ;
#pragma unroll
      for (int r = lane; r < BQ; r += 32) {
        const int i = it.i0 + r;
        const bool in = i < s.Sq;
        dst[r] = in ? -(p.lse[rowbase + i] * l2e) : 0.f;   // negated: the exponent is one FMA
        dst[BQ + r] = in ? p.dsum[rowbase + i] : 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_lsed_full[slot]);
      ++st;
    }
   }
  } else if (warp < 12) {
    regs_inc<kRegsSoftmax>();
    // ---------------------------------------------------------------- softmax-grad
    const int wq = warp & 3;                      // TMEM lane quadrant
    const int half = (warp - 4) >> 2;             // which half of the step's query columns
    const int r = wq * 32 + lane;                 // key row within the tile
    const int j = j0 + r;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const float sl2 = s.scale * kLog2e;
    const uint64_t sl2_2 = f32x2(sl2, sl2);
    const bool key_ok = j < s.Sk;
    const size_t mrow0 = (size_t)mb * s.Sq;
    // query rows that see this key: [row_lo, row_hi] from the causal rule and the window
    long long row_lo = 0, row_hi = (long long)s.Sq - 1;
    if (s.causal) row_lo = (long long)j - s.q_offset;
    if (s.window > 0) {
      if (!s.causal) row_lo = (long long)j - s.q_offset - s.window;
      row_hi = min(row_hi, (long long)j - s.q_offset + s.window);
    }

    if (p.q8) {
      // the CTA's K and V tiles, dequantized once by these eight warps into the bf16 operand tiles
      const int tid = threadIdx.x - 128;
      const size_t kvrow0 = (size_t)(b * s.Hkv + kvh) * s.Sk;
      dequant_q8_tile<D>(p.kq, p.kd, kvrow0, j0, s.Sk, smem + C::OFF_K, 0, kBN, tid, 256);
      dequant_q8_tile<D>(p.vq, p.vd, kvrow0, j0, s.Sk, smem + C::OFF_V, 0, kBN, tid, 256);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_kv);
    }
    StepIter it;
    it.init(G, iend, BQ, ibeg, DET);
    int st = 0;
    bool ok = true;
    for (; it.valid(); it.next()) {
      if (step_skipped(it)) continue;
      const int buf = st % C::NBUF, slot = st % C::NSTAGE, dsb = st % C::NDS;
      ok = mbar_wait(&bar_s_full[buf], (st / C::NBUF) & 1, abort_flag, p.status, 130);
      ok = ok && mbar_wait(&bar_lsed_full[slot], (st / C::NSTAGE) & 1, abort_flag, p.status, 131);
      // the dQ MMA of the previous step has read the dS^T tile (its completion on bar_dq_full)
      if (st > 0) ok = ok && mbar_wait(&bar_dq_full[0], (st - 1) & 1, abort_flag, p.status, 132);
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
      tc_fence_after();
      const uint32_t tb = tmem + buf * C::BUF_COLS + lane_off;
      const uint32_t lse_s = smem_u32(lsed + slot * 2 * BQ);  // [-lse * log2(e) x BQ | D x BQ]
      const int code = bwd_tile_code(p, mb, it.i0, kt);
      // every pair of this step visible for this key: open tile, real key, all BQ rows inside the
      // key's row band (which also ends at the last real row)
      const bool full = code == TILE_OPEN && key_ok && it.i0 >= row_lo && (long long)it.i0 + BQ - 1 <= row_hi;
      const uint32_t sds = smem_u32(smem + C::OFF_DS + dsb * C::DS_TILE) + r * 128;
#pragma unroll 1   // one copy of the round body: the hot loop's code stays small
      for (int cc = 0; cc < C::CHUNKS_PER_WARP; ++cc) {
        // round cc covers queries [64cc, 64cc + 64): the two warps of a lane quadrant take one
        // 32-query chunk each, and the first round is handed to the dV / dK MMAs right away
        const int c = cc * 2 + half;   // score chunk: queries [32c, 32c+32)
        // P^T of the chunk from its scores: in the first round while the dP^T MMAs still run, in
        // the second with dP^T loaded in the same TMEM round trip; the score columns then
        // receive P^T and dS^T
        uint32_t sr[32], dr[32];
        tmem_ld32(tb + c * 32, sr);
        if (cc > 0) tmem_ld32(tb + BQ + c * 32, dr);
        // the chunk's 32 (negated, log2-scaled) LSE values, loaded while the TMEM loads are in flight
        // (the wait below orders every memory access, so loads issued after it would add their
        // latency to it)
        float l2c[32];
#pragma unroll
        for (int v4 = 0; v4 < 8; ++v4) {
          const float4 a = ld_shared_f4(lse_s + (c * 32 + 4 * v4) * 4);
          l2c[4 * v4] = a.x; l2c[4 * v4 + 1] = a.y; l2c[4 * v4 + 2] = a.z; l2c[4 * v4 + 3] = a.w;
        }
        tmem_wait_ld();
        reg_fence(sr);
        float pv[32];
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          const int q0 = c * 32 + sub * 16;   // first query of these 16
          const float* l2 = l2c + sub * 16;
          float* pw = pv + sub * 16;
          if (!MASKED || full || code != TILE_MIXED) {
            // full and partial tiles share the exponentials (one copy of the unrolled loop: code
            // size matters here); a partial tile then zeroes the query rows outside this key's
            // visible rows [rlo, rhi) (causal rule, window, query tail), a 16-bit set
            // the exponents on packed fp32 pairs (this loop is issue-bound)
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              float t0, t1;
              f32x2_split(fma_f32x2(f32x2(__uint_as_float(sr[sub * 16 + e]), __uint_as_float(sr[sub * 16 + e + 1])),
                                    sl2_2, f32x2(l2[e], l2[e + 1])),
                          t0, t1);
              pw[e] = ex2_approx(t0);
              pw[e + 1] = ex2_approx(t1);
            }
            if (!full) {
              const int base = it.i0 + q0;
              const int rlo = (int)max(0LL, min(row_lo - base, 16LL));
              const int rhi = key_ok && code != TILE_SKIP ? (int)max(0LL, min(row_hi - base + 1, 16LL)) : 0;
              const uint32_t vis = rhi > rlo ? ((1u << rhi) - 1u) & ~((1u << rlo) - 1u) : 0u;
#pragma unroll
              for (int e = 0; e < 16; ++e) pw[e] = (vis >> e) & 1u ? pw[e] : 0.f;
            }
          } else {
            // a mixed tile: visible query rows of this key are [rlo, rhi) relative to base (causal
            // rule, window, query tail), and the mask decides within them
            const int base = it.i0 + q0;
            const int rlo = (int)max(0LL, min(row_lo - base, 16LL));
            const int rhi = key_ok ? (int)max(0LL, min(row_hi - base + 1, 16LL)) : 0;
            {
              // the 16 mask values of this key (one per query row) first, then the arithmetic
              float bias[16];
              if (s.mask_kind == MK_ADD) {
                const float* mp = static_cast<const float*>(p.mask) + (mrow0 + base) * (size_t)s.Sk + j;
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  bias[e] = (e >= rlo && e < rhi) ? __ldg(mp + (size_t)e * s.Sk) : -CUDART_INF_F;
#pragma unroll
                for (int e = 0; e < 16; ++e) bias[e] = bias[e] > kMaskFloor ? bias[e] * kLog2e : -CUDART_INF_F;
              } else {
                const uint8_t* mp = static_cast<const uint8_t*>(p.mask) + (mrow0 + base) * (size_t)s.Sk + j;
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  bias[e] = (e >= rlo && e < rhi && __ldg(mp + (size_t)e * s.Sk) != 0) ? 0.f : -CUDART_INF_F;
              }
#pragma unroll
              for (int e = 0; e < 16; ++e)
                pw[e] = bias[e] != -CUDART_INF_F
                            ? ex2_approx(fmaf(__uint_as_float(sr[sub * 16 + e]), sl2, bias[e] + l2[e]))
                            : 0.f;
            }
          }
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) pk[e] = pack_bf16x2(pw[2 * e], pw[2 * e + 1]);
          tmem_st8(tb + c * 32 + sub * 8, pk);   // P^T of these 16 queries
        }
        float dc[32];   // the chunk's 32 D values
        if (cc == 0) {
          // dP^T of the step (its MMAs ran under the exponentials above)
          ok = __all_sync(0xffffffffu, mbar_wait(&bar_sdp_full[buf], (st / C::NBUF) & 1, abort_flag, p.status, 135));
          if (!ok) break;
          tc_fence_after();
          tmem_ld32(tb + BQ + c * 32, dr);
        }
        // loaded while the dP^T TMEM load is in flight (first round)
#pragma unroll
        for (int v4 = 0; v4 < 8; ++v4) {
          const float4 d = ld_shared_f4(lse_s + (BQ + c * 32 + 4 * v4) * 4);
          dc[4 * v4] = d.x; dc[4 * v4 + 1] = d.y; dc[4 * v4 + 2] = d.z; dc[4 * v4 + 3] = d.w;
        }
        if (cc == 0) tmem_wait_ld();
        reg_fence(dr);
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          const int q0 = c * 32 + sub * 16;
          const float* dv_ = dc + sub * 16;
          const float* pw = pv + sub * 16;
          uint32_t dk8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            // dS = P (dP - D) on packed fp32 pairs
            float d0, d1;
            f32x2_split(mul_f32x2(f32x2(pw[2 * e], pw[2 * e + 1]),
                                  sub_f32x2(f32x2(__uint_as_float(dr[sub * 16 + 2 * e]),
                                                  __uint_as_float(dr[sub * 16 + 2 * e + 1])),
                                            f32x2(dv_[2 * e], dv_[2 * e + 1]))),
                        d0, d1);
            dk8[e] = pack_bf16x2(d0, d1);
          }
          tmem_st8(tb + c * 32 + 16 + sub * 8, dk8);   // dS^T of these 16 queries
          // dS^T row of this key into the swizzled SMEM operand of the dQ MMA (2 x 16 B chunks)
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int chunk = (q0 >> 3) + u;          // 16-byte chunk among the BQ / 8 of this row
            const int blk = chunk / 8, cin = chunk % 8;
            st_shared_v4(sds + blk * C::DS_BLOCK + ((cin ^ (r & 7)) * 16), dk8[4 * u], dk8[4 * u + 1],
                         dk8[4 * u + 2], dk8[4 * u + 3]);
          }
        }
        if (C::TWO_ROUND && cc == 0) {
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_p_half);
        }
      }
      if (!ok) {
        tmem_wait_st();
        break;
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bar_p_full[buf]);
        mbar_arrive(&bar_lsed_empty[slot]);
      }
      ++st;
    }
    // ---- epilogue: dV and scale * dK of this thread's key, from TMEM; each warp of the
    //      quadrant pair takes half of the feature columns
    ok = __all_sync(0xffffffffu, ok);
    if (ok && st > 0) ok = __all_sync(0xffffffffu, mbar_wait(bar_mma_done, 0, abort_flag, p.status, 133));
    tc_fence_after();
    // One 32-feature chunk of dV (which = 0) or dK (which = 1) of this thread's key, already scaled,
    // to its destination: the bf16 rows, or the fp32 accumulator (and the read-back rows).
    const size_t row = head_base(s, b, kvh, s.Hkv, s.Sk) + (size_t)(key_ok ? j : 0) * row_stride(s, s.Hkv);
    // the fused SET_ROWS backward: this key's finished sum is also one of the read-back rows
    const long long rr = (long long)j - p.rows_begin;
    const bool read_back = p.accum && key_ok && rr >= 0 && rr < p.n_rows;
    const size_t rrow = head_base(s, b, kvh, s.Hkv, p.n_rows) + (size_t)(read_back ? rr : 0) * row_stride(s, s.Hkv);
    auto store_chunk = [&](int which, int c, const float* x) {
      if (!key_ok) return;
      void* outp = which == 0 ? p.dv : p.dk;
      if (p.accum) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(outp) + row + c * 32);
        // all eight loads first (the read-back stores below could alias them as far as the
        // compiler knows), then the adds and the stores
        float4 a[8];
#pragma unroll
        for (int v4 = 0; v4 < 8; ++v4) a[v4] = dst[v4];
#pragma unroll
        for (int v4 = 0; v4 < 8; ++v4) {
          a[v4].x += x[4 * v4];
          a[v4].y += x[4 * v4 + 1];
          a[v4].z += x[4 * v4 + 2];
          a[v4].w += x[4 * v4 + 3];
          dst[v4] = a[v4];
        }
        if (read_back) {
          uint2* rdst = reinterpret_cast<uint2*>((which == 0 ? p.dv_rows : p.dk_rows) + rrow + c * 32);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            rdst[v4] = make_uint2(pack_bf16x2(a[v4].x, a[v4].y), pack_bf16x2(a[v4].z, a[v4].w));
        }
      } else {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(outp) + row + c * 32);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          uint32_t w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) w[u] = pack_bf16x2(x[8 * v4 + 2 * u], x[8 * v4 + 2 * u + 1]);
          dst[v4] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    };
    // this thread's sums of one chunk from TMEM, scaled (zero when the CTA had no step)
    auto load_chunk = [&](int which, int c, float* x) {
      const float mul = which == 0 ? 1.f : s.scale;
      const uint32_t tcol = tmem + lane_off + (which == 0 ? C::DV_COL : C::DK_COL);
      uint32_t v[32];
      if (st > 0) {
        tmem_ld32(tcol + c * 32, v);
        tmem_wait_ld();
        reg_fence(v);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0u;
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(v[e]) * mul;
    };
    if (nparts > 1) {
      // A part of a split key tile. A ticket per key tile tells the part that finishes last: every
      // other part writes its fp32 sums to its partial slot and counts itself written; the last
      // one waits for those writes, adds the slots and its own sums (from TMEM) in part order and
      // writes dK / dV. All eight warps reach the barriers below whatever `ok` says.
      const size_t slot0 = (size_t)bkv * p.n_slots + (slot - part);
      int* sync = p.part_sync + 2 * slot0;   // [tickets taken, partials written]
      if (warp == 4 && lane == 0) *last_part = atom_add_acq_rel_gpu(sync, 1) == nparts - 1 ? 1 : 0;
      named_bar_sync(1, 256);
      if (*last_part == 0) {
        if (ok) {
          // a slot is [dV, dK] x [D / 4][128 keys] float4: a warp's 32 keys move 512 contiguous bytes
          float4* mine = reinterpret_cast<float4*>(p.part + ((size_t)bkv * p.n_slots + slot) * 2 * kBN * D) + r;
#pragma unroll
          for (int which = 0; which < 2; ++which)
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
              const int c = half * (D / 64) + cc;      // 32-feature chunk
              float x[32];
              load_chunk(which, c, x);
              float4* d4 = mine + ((size_t)which * (D / 4) + c * 8) * kBN;
#pragma unroll
              for (int v4 = 0; v4 < 8; ++v4)
                d4[v4 * kBN] = make_float4(x[4 * v4], x[4 * v4 + 1], x[4 * v4 + 2], x[4 * v4 + 3]);
            }
        }
        __threadfence();
        named_bar_sync(1, 256);
        if (warp == 4 && lane == 0) red_release_gpu_add(sync + 1, 1);
      } else {
        if (warp == 4 && lane == 0) *parts_ready = wait_turn(sync + 1, nparts - 1, abort_flag, p.status, 137) ? 1 : 0;
        named_bar_sync(1, 256);
        if (ok && *parts_ready) {
          fence_acq_rel_gpu();
          const float4* slots = reinterpret_cast<const float4*>(p.part + slot0 * 2 * kBN * D) + r;
#pragma unroll
          for (int which = 0; which < 2; ++which)
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
              const int c = half * (D / 64) + cc;
              float x[32];
#pragma unroll
              for (int e = 0; e < 32; ++e) x[e] = 0.f;
              for (int q = 0; q < nparts; ++q) {
                float y[32];
                if (q == part) {
                  load_chunk(which, c, y);
                } else {
                  const float4* src = slots + (((size_t)q * 2 + which) * (D / 4) + c * 8) * kBN;
#pragma unroll
                  for (int v4 = 0; v4 < 8; ++v4) {
                    const float4 v = __ldcg(src + v4 * kBN);
                    y[4 * v4] = v.x;
                    y[4 * v4 + 1] = v.y;
                    y[4 * v4 + 2] = v.z;
                    y[4 * v4 + 3] = v.w;
                  }
                }
#pragma unroll
                for (int e = 0; e < 32; ++e) x[e] += y[e];
              }
              store_chunk(which, c, x);
            }
        }
      }
    } else if (ok) {
#pragma unroll
      for (int which = 0; which < 2; ++which)
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
          const int c = half * (D / 64) + cc;      // 32-feature chunk
          float x[32];
          load_chunk(which, c, x);
          store_chunk(which, c, x);
        }
    }
  } else {
    regs_inc<kRegsStager>();
    // ---------------------------------------------------------------- dQ stager (warps 12-15)
    // Each step's dQ partial leaves TMEM for the fp32 dQ accumulator, where the add happens in
    // L2: through the step's consumed Q/dO slot and D/32 TMA reduce-adds issued by the leader
    // thread.
    const int wq = warp & 3;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const bool leader = warp == 12 && lane == 0;
    StepIter it;
    it.init(G, iend, BQ, ibeg, DET);
    // Deterministic dQ: the key tiles form groups of det_group(s); each group has its own fp32 dQ
    // accumulator (summed in group order by the convert pass), and within a group the key tiles that
    // see a query tile add their partials to it in ascending key-tile order. A turn counter per
    // (group, batch, query head, query tile) counts the passes: the leader thread of each earlier
    // key tile adds one once its partial is added, steps the tile map skips included. The key tiles
    // that see query tile i0 are the consecutive tiles from kt_first(i0) on, so a tile's rank in its
    // group follows from the shape alone.
    const int det_g = det_group(s);
    const int group = DET ? kt / det_g : 0;
    const size_t bhq = (size_t)s.B * s.Hq;
    auto turn_of = [&](const StepIter& t) -> int* {
      return p.turn + ((size_t)group * bhq + (size_t)(b * s.Hq + kvh * G + t.hh)) * p.nqt + t.i0 / 128;
    };
    auto rank_of = [&](const StepIter& t) -> int {
      const long long kt_first = s.window > 0 ? max(0LL, s.q_offset + t.i0 - s.window) / kBN : 0;
      return kt - (int)max(kt_first, (long long)group * det_g);
    };
    int st = 0;
    for (; it.valid(); it.next()) {
      if (step_skipped(it)) {
        if (!DET) continue;
        // no partial from this key tile here, but its turn still passes
        int* turn = turn_of(it);
        bool ok2 = true;
        if (leader) {
          ok2 = wait_turn(turn, rank_of(it), abort_flag, p.status, 140);
          if (ok2) red_release_gpu_add(turn, 1);
        }
        if (!__shfl_sync(0xffffffffu, ok2 ? 1 : 0, 0)) break;
        continue;
      }
      const int slot = st % C::NSTAGE, buf = st % C::NBUF;
      float* sdq = reinterpret_cast<float*>(smem + C::OFF_STAGE + slot * 2 * C::Q_TILE);
      const uint32_t sbase = smem_u32(sdq);
      if (!__all_sync(0xffffffffu, mbar_wait(&bar_dq_full[buf], (st / C::NBUF) & 1, abort_flag, p.status, 134)))
        break;
      // the whole dQ partial row of this thread into registers, so the TMEM block is released at once
      tc_fence_after();
      uint32_t v[C::DQ_CHUNKS][32];
#pragma unroll
      for (int c = 0; c < C::DQ_CHUNKS; ++c)
        tmem_ld32(tmem + buf * C::BUF_COLS + C::DQ_COL + c * 32 + lane_off, v[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < C::DQ_CHUNKS; ++c) reg_fence(v[c]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_dq_free[buf]);   // the TMEM block is free for the next dP^T
      {
        // then into the slot, whose Q and dO the dV / dK MMAs (issued before this dQ MMA) have read:
        // thread = query row, registers = features 32c + e. Each 32-feature chunk c has its own
        // [BQ][32] fp32 sub-tile with 128-byte rows, 128-byte swizzled (16-byte chunk u of row q
        // at u ^ (q & 7)): conflict-free stores with static register indices, and the layout the
        // reduce's tensor map reads
        const int q = wq * 32 + lane;
#pragma unroll
        for (int c = 0; c < C::DQ_CHUNKS; ++c) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            st_shared_v4(sbase + c * BQ * 128 + q * 128 + ((u ^ (q & 7)) << 4), v[c][4 * u], v[c][4 * u + 1],
                         v[c][4 * u + 2], v[c][4 * u + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_stage_full);
        // the leader waits for all four warps' stores, issues the reduce, and hands the slot back to
        // the producer once the reduce has read it; its warp leaves the loop together on a timeout
        bool filled = true;
        if (leader) filled = mbar_wait(bar_stage_full, st & 1, abort_flag, p.status, 136);
        if (!__shfl_sync(0xffffffffu, filled ? 1 : 0, 0)) break;
        bool ok2 = true;
        if (leader) {
          const int row_head = (int)(group * bhq) + b * s.Hq + kvh * G + it.hh;
          const uint8_t* src = reinterpret_cast<const uint8_t*>(sdq);
          if constexpr (!DET) {
            for (int c = 0; c < C::DQ_CHUNKS; ++c)
              tma_reduce_add_3d(&p.tm_dq, src + c * BQ * 128, c * 32, it.i0, row_head);
            bulk_commit_group();
            bulk_wait_group_read0();
          } else {
            // in turn: the whole add is complete and visible before the turn passes
            int* turn = turn_of(it);
            ok2 = wait_turn(turn, rank_of(it), abort_flag, p.status, 142);
            if (ok2) {
              fence_acq_rel_gpu();
              fence_proxy_async_global();
              for (int c = 0; c < C::DQ_CHUNKS; ++c)
                tma_reduce_add_3d(&p.tm_dq, src + c * BQ * 128, c * 32, it.i0, row_head);
              bulk_commit_group();
              bulk_wait_group0();
              fence_proxy_async_global();
              fence_acq_rel_gpu();
              red_release_gpu_add(turn, 1);
            }
          }
          if (ok2) mbar_arrive(&bar_qdo_empty[slot]);
        }
        if (!__shfl_sync(0xffffffffu, ok2 ? 1 : 0, 0)) break;
      }
      ++st;
    }
    if (leader) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool tc_bwd_supported(const Shape& s) { return (s.D == 64 || s.D == 128) && s.Sq > 0; }

namespace {

// Cost of a CTA in query-tile steps (one step: the five 128 x 128 x D products of a query tile):
// its steps, a fixed cost per CTA (TMEM and barriers, the K / V tiles, filling and draining the
// pipeline, dK / dV out of TMEM) and, for a part of a split key tile, the round trip of its fp32
// partial. Measured per CTA on the causal backward over 4096 keys: about 3.1 us a step, 10 us a
// CTA and 2 us a part.
constexpr double kCtaCost = 3.2, kPartCost = 0.7;
inline double cta_cost(int steps, bool part) { return steps + kCtaCost + (part ? kPartCost : 0.0); }

// The end of a launch under the block scheduler's rule: each block, in launch order, starts on
// the SM that frees up first.
double dispatch_end(const std::vector<double>& cost, int sms) {
  std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
  for (int i = 0; i < sms; ++i) free_at.push(0.0);
  double end = 0.0;
  for (double c : cost) {
    const double t = free_at.top() + c;
    free_at.pop();
    free_at.push(t);
    end = std::max(end, t);
  }
  return end;
}

// Best-fit decreasing: items (costs in descending order) into `sms` SMs of capacity `cap`, each
// into the fullest SM it still fits; false if one does not fit.
bool best_fit(const std::vector<double>& cost, int sms, double cap, std::vector<int>& sm_of) {
  std::multiset<std::pair<double, int>> load;
  for (int i = 0; i < sms; ++i) load.insert({0.0, i});
  for (size_t k = 0; k < cost.size(); ++k) {
    auto it = load.upper_bound({cap - cost[k], INT_MAX});
    if (it == load.begin()) return false;
    --it;
    const std::pair<double, int> e = *it;
    load.erase(it);
    sm_of[k] = e.second;
    load.insert({e.first + cost[k], e.second});
  }
  return true;
}

// Full grid: each candidate cap c splits every key tile of more than c query tiles into parts of c
// (the last one shorter); its CTAs are packed onto the SMs by best-fit decreasing at the smallest
// capacity that holds them, and launched in the packing's planned start order. The plan with the
// earliest end under the dispatch rule is taken if it beats the key-tile order by 2%.
bool plan_full_grid(const int* tiles, int nkt, int G, int nbkv, int sms, BwdSplit& out) {
  std::vector<double> base;
  int most = 0;
  for (int kt = 0; kt < nkt; ++kt) {
    most = std::max(most, tiles[kt]);
    for (int i = 0; i < nbkv; ++i) base.push_back(cta_cost(G * tiles[kt], false));
  }
  double best = 0.98 * dispatch_end(base, sms);
  bool found = false;
  struct Unit { int kt, part, nparts, t0, t1; };
  std::vector<Unit> units;
  std::vector<std::pair<double, int>> items;   // (cost, unit), one per CTA
  std::vector<double> cost;
  std::vector<int> sm_of, best_sm;
  for (int cap = most - 1; cap >= std::max(1, most / 2); --cap) {
    units.clear();
    bool fits = true;
    for (int kt = 0; kt < nkt && fits; ++kt) {
      const int np = tiles[kt] > cap ? (tiles[kt] + cap - 1) / cap : 1;
      if (np > kMaxParts) fits = false;
      for (int q = 0; q < np; ++q) units.push_back({kt, q, np, q * cap, np > 1 ? std::min(tiles[kt], (q + 1) * cap) : 0});
    }
    if (!fits || (int)units.size() > kMaxUnits || (long long)units.size() * nbkv > kMaxCtas) continue;
    items.clear();
    for (int u = 0; u < (int)units.size(); ++u) {
      const Unit& x = units[u];
      const int steps = G * (x.nparts > 1 ? x.t1 - x.t0 : tiles[x.kt]);
      for (int i = 0; i < nbkv; ++i) items.push_back({cta_cost(steps, x.nparts > 1), u});
    }
    std::stable_sort(items.begin(), items.end(), [](const std::pair<double, int>& a, const std::pair<double, int>& b) {
      return a.first > b.first;
    });
    cost.resize(items.size());
    double total = 0.0;
    for (size_t k = 0; k < items.size(); ++k) total += (cost[k] = items[k].first);
    sm_of.assign(items.size(), 0);
    double lo = std::max(total / sms, cost[0]), hi = dispatch_end(cost, sms) + 1.0;
    if (!best_fit(cost, sms, hi, sm_of)) continue;
    std::vector<int> fit = sm_of;
    for (int it = 0; it < 24 && hi - lo > 0.05; ++it) {
      const double mid = 0.5 * (lo + hi);
      if (best_fit(cost, sms, mid, sm_of)) {
        hi = mid;
        fit = sm_of;
      } else {
        lo = mid;
      }
    }
    // planned start of each CTA: on its SM, after the larger ones packed there before it
    std::vector<double> start(items.size()), used(sms, 0.0);
    for (size_t k = 0; k < items.size(); ++k) {
      start[k] = used[fit[k]];
      used[fit[k]] += cost[k];
    }
    std::vector<int> order(items.size());
    for (size_t k = 0; k < order.size(); ++k) order[k] = (int)k;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
      return start[a] < start[b] || (start[a] == start[b] && fit[a] < fit[b]);
    });
    std::vector<double> ordered(order.size());
    for (size_t k = 0; k < order.size(); ++k) ordered[k] = cost[order[k]];
    const double end = dispatch_end(ordered, sms);
    if (end >= best) continue;
    best = end;
    found = true;
    // the plan: units (slots of the split tiles' parts in key-tile order), then the launch order
    int slots = 0;
    for (int u = 0; u < (int)units.size(); ++u) {
      const Unit& x = units[u];
      const uint32_t slot = x.nparts > 1 ? (uint32_t)slots++ : 0u;
      out.units[u] = (uint32_t)x.kt | (uint32_t)x.part << 12 | (uint32_t)x.nparts << 16 | slot << 20;
      out.range[u] = (uint32_t)x.t0 | (uint32_t)x.t1 << 16;
    }
    std::vector<int> next_bkv(units.size(), 0);
    for (size_t k = 0; k < order.size(); ++k) {
      const int u = items[order[k]].second;
      out.ctas[k] = (uint32_t)u | (uint32_t)next_bkv[u]++ << 16;
    }
    out.n_units = (int)units.size();
    out.n_slots = slots;
    out.n_ctas = (int)order.size();
  }
  return found;
}

struct PlanKey {
  int B, Hq, Hkv, Sq, Sk, causal, window, deterministic;
  long long q_offset;
  bool operator==(const PlanKey& o) const { return memcmp(this, &o, sizeof(PlanKey)) == 0; }
};

void plan_split_uncached(const Shape& s, BwdSplit& out) {
  out.n_units = out.n_slots = out.n_ctas = 0;
  constexpr int BQ = 128;   // the query tile of both configurations
  const int sms = sm_count();
  const int nkt = (s.Sk + kBN - 1) / kBN, G = s.Hq / s.Hkv;
  const long long nbkv = (long long)s.B * s.Hkv;
  // Never with deterministic dQ, whose turns need the key tiles dispatched in ascending order.
  if (s.deterministic || nkt > kMaxUnits || nkt > 4095 || nbkv > 0xffff) return;
  int tiles[kMaxUnits];
  long long total = 0, heaviest = 0;
  for (int kt = 0; kt < nkt; ++kt) {
    int ib, ie;
    key_tile_rows(s, kt, BQ, ib, ie);
    tiles[kt] = ib < ie ? (ie - ib + BQ - 1) / BQ : 0;
    total += (long long)G * tiles[kt];
    heaviest = std::max(heaviest, (long long)G * tiles[kt]);
  }
  // the per-SM share of all steps
  const double share = (double)(total * nbkv) / sms;
  if (share <= 0 || heaviest <= share) return;
  if ((long long)nkt * nbkv >= sms) {
    if ((long long)nkt * nbkv <= kMaxCtas) plan_full_grid(tiles, nkt, G, (int)nbkv, sms, out);
    return;
  }
  // under-filled grid: key tiles above the share are cut into even parts of about that size
  int nparts[kMaxUnits];
  int units = 0, split = 0;
  for (int kt = 0; kt < nkt; ++kt) {
    const long long steps = (long long)G * tiles[kt];
    int np = 1;
    // parts of at least 4 steps: shorter CTAs spend most of their time filling and draining
    if (steps > share)
      np = (int)std::min<long long>({kMaxParts, tiles[kt], steps / 4, (long long)std::ceil(steps / share)});
    nparts[kt] = std::max(1, np);
    units += nparts[kt];
    split += nparts[kt] > 1;
  }
  if (split == 0 || units > kMaxUnits) return;
  // slots of the split tiles' parts, then the units sorted heaviest first (ties in key-tile order)
  int slot_of[kMaxUnits];
  int slots = 0;
  for (int kt = 0; kt < nkt; ++kt) {
    slot_of[kt] = slots;
    if (nparts[kt] > 1) slots += nparts[kt];
  }
  if (slots >= 4096) return;
  struct U { double work; int kt, part; };
  U list[kMaxUnits];
  int n = 0;
  for (int kt = 0; kt < nkt; ++kt)
    for (int q = 0; q < nparts[kt]; ++q)
      list[n++] = U{(double)G * tiles[kt] / nparts[kt], kt, q};
  std::stable_sort(list, list + n, [](const U& a, const U& b) { return a.work > b.work; });
  for (int i = 0; i < n; ++i) {
    const int kt = list[i].kt, q = list[i].part, np = nparts[kt];
    const uint32_t slot = np > 1 ? (uint32_t)(slot_of[kt] + q) : 0u;
    out.units[i] = (uint32_t)kt | (uint32_t)q << 12 | (uint32_t)np << 16 | slot << 20;
    out.range[i] = (uint32_t)(q * tiles[kt] / np) | (uint32_t)((q + 1) * tiles[kt] / np) << 16;
  }
  out.n_units = n;
  out.n_slots = slots;
}

}  // namespace

int sm_count() {
  static const int n = [] {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        v > 0)
      return v;
    cudaGetLastError();
    return 152;
  }();
  return n;
}

void plan_bwd_split(const Shape& s, BwdSplit& out) {
  // the full-grid plan searches a few dozen packings: plans are kept for the last few shapes
  constexpr int kCache = 4;
  struct Entry { PlanKey key; BwdSplit plan; bool used; };
  static thread_local Entry cache[kCache];
  static thread_local int next = 0;
  PlanKey key;
  memset(&key, 0, sizeof(key));
  key.B = s.B; key.Hq = s.Hq; key.Hkv = s.Hkv; key.Sq = s.Sq; key.Sk = s.Sk;
  key.causal = s.causal; key.window = s.window; key.deterministic = s.deterministic; key.q_offset = s.q_offset;
  for (Entry& e : cache)
    if (e.used && e.key == key) {
      out = e.plan;
      return;
    }
  plan_split_uncached(s, out);
  Entry& e = cache[next];
  next = (next + 1) % kCache;
  e.key = key;
  e.plan = out;
  e.used = true;
}

int bwd_plan_records(const Shape& s, int32_t* rec, int cap) {
  static thread_local BwdSplit split;
  plan_bwd_split(s, split);
  const int nbkv = s.B * s.Hkv, nkt = (s.Sk + kBN - 1) / kBN;
  const long long n = split.n_ctas > 0 ? split.n_ctas : (long long)nbkv * (split.n_units > 0 ? split.n_units : nkt);
  for (long long i = 0; i < n && i < cap; ++i) {
    int unit = (int)(i / nbkv), bkv = (int)(i % nbkv);
    if (split.n_ctas > 0) {
      unit = (int)(split.ctas[i] & 0xffffu);
      bkv = (int)(split.ctas[i] >> 16);
    }
    int kt = unit, part = 0, nparts = 1;
    if (split.n_units > 0) {
      kt = (int)(split.units[unit] & 0xfffu);
      part = (int)((split.units[unit] >> 12) & 0xfu);
      nparts = (int)((split.units[unit] >> 16) & 0xfu);
    }
    int ib, ie;
    key_tile_rows(s, kt, 128, ib, ie);
    if (nparts > 1) {
      const int base = ib;
      ib = base + (int)(split.range[unit] & 0xffffu) * 128;
      ie = std::min(ie, base + (int)(split.range[unit] >> 16) * 128);
    }
    int32_t* r = rec + 6 * i;
    r[0] = kt;
    r[1] = bkv;
    r[2] = part;
    r[3] = nparts;
    r[4] = ib;
    r[5] = ie;
  }
  return (int)n;
}

template <int D>
static cudaError_t tc_bwd_t(const BwdArgs& a, const BwdPlan& plan, char* ws, unsigned* status) {
  using C = BwdCfg<D>;
  const Shape& s = a.s;
  BwdTcParams p;
  memset(&p, 0, sizeof(p));
  cudaError_t e;
  if ((e = make_tmap_4d(&p.tm_q, a.q, s.layout, s.B, s.Hq, s.Sq, D, C::BQ)) != cudaSuccess) return e;
  if ((e = make_tmap_4d(&p.tm_do, a.dO, s.layout, s.B, s.Hq, s.Sq, D, C::BQ)) != cudaSuccess) return e;
  p.q8 = a.kq != nullptr ? 1 : 0;
  if (p.q8) {
    p.kq = a.kq;
    p.kd = static_cast<const __half*>(a.kd);
    p.vq = a.vq;
    p.vd = static_cast<const __half*>(a.vd);
  } else {
    if ((e = make_tmap_4d(&p.tm_k, a.k, s.layout, s.B, s.Hkv, s.Sk, D, kBN)) != cudaSuccess) return e;
    if ((e = make_tmap_4d(&p.tm_v, a.v, s.layout, s.B, s.Hkv, s.Sk, D, kBN)) != cudaSuccess) return e;
  }
  float* dq_acc = reinterpret_cast<float*>(ws + plan.dqacc_off);
  const int groups = dq_groups(s);
  if ((e = make_tmap_f32_bhsd_sw128(&p.tm_dq, dq_acc, s.Sq, groups * s.B * s.Hq, D, C::BQ)) != cudaSuccess) return e;
  p.s = s;
  p.mask = a.mask;
  p.nqt = (s.Sq + 127) / 128;
  p.nkt = (s.Sk + kBN - 1) / kBN;
  p.tilemap = nullptr;
  if (s.mask_kind != MK_NONE) {
    uint8_t* tm = reinterpret_cast<uint8_t*>(ws + plan.tilemap_off);
    if ((e = launch_mask_classify(s, a.mask, tm, a.stream)) != cudaSuccess) return e;
    p.tilemap = tm;
  }
  float* dsum = reinterpret_cast<float*>(ws + plan.dsum_off);
  static thread_local BwdSplit split;
  plan_bwd_split(s, split);
  int* part_sync = nullptr;
  int n_sync = 0;
  if (split.n_units > 0) {   // the split key tiles' counters start at zero, set by the D pass
    part_sync = reinterpret_cast<int*>(ws + plan.cnt_off);
    n_sync = (int)(plan.cnt_bytes / 4);
  }
  if ((e = launch_dsum(a, dsum, dq_acc, groups, reinterpret_cast<uint32_t*>(part_sync), n_sync)) != cudaSuccess)
    return e;
  p.lse = a.lse;
  p.dsum = dsum;
  p.dq_acc = dq_acc;
  p.dk = a.dk;
  p.dv = a.dv;
  p.accum = a.accum ? 1 : 0;
  p.rows_begin = a.rows_begin;
  p.n_rows = a.accum ? a.n_rows : 0;
  p.dk_rows = static_cast<__nv_bfloat16*>(a.dk_rows);
  p.dv_rows = static_cast<__nv_bfloat16*>(a.dv_rows);
  p.status = status;
  p.turn = nullptr;
  if (s.deterministic) {
    p.turn = reinterpret_cast<int*>(ws + plan.turn_off);
    if ((e = cudaMemsetAsync(p.turn, 0, plan.turn_bytes, a.stream)) != cudaSuccess) return e;
  }
  p.n_units = split.n_units;
  p.n_slots = split.n_slots;
  p.n_ctas = split.n_ctas;
  p.part = split.n_units > 0 ? reinterpret_cast<float*>(ws + plan.part_off) : nullptr;
  p.part_sync = part_sync;
  memcpy(p.units, split.units, sizeof(uint32_t) * split.n_units);
  memcpy(p.range, split.range, sizeof(uint32_t) * split.n_units);
  memcpy(p.ctas, split.ctas, sizeof(uint32_t) * split.n_ctas);
  const int smem = C::BYTES;
  auto kernel = s.mask_kind != MK_NONE ? (s.deterministic ? bwd_tc_kernel<D, true, true> : bwd_tc_kernel<D, true, false>)
                                       : (s.deterministic ? bwd_tc_kernel<D, false, true> : bwd_tc_kernel<D, false, false>);
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
    return e;
  const long long ctas = split.n_ctas > 0 ? split.n_ctas : (long long)s.B * s.Hkv * (split.n_units > 0 ? split.n_units : p.nkt);
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if ((e = prof_begin(KID_BWD_MAIN, a.stream)) != cudaSuccess) return e;
  kernel<<<(unsigned)ctas, kThreads, smem, a.stream>>>(p);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = prof_end(KID_BWD_MAIN, a.stream)) != cudaSuccess) return e;
  return launch_dq_convert(a, dq_acc, groups);
}

cudaError_t tc_bwd(const BwdArgs& a, const BwdPlan& plan, char* ws) {
  unsigned* status = device_status_ptr();
  if (status == nullptr) return cudaErrorUnknown;
  return a.s.D == 64 ? tc_bwd_t<64>(a, plan, ws, status) : tc_bwd_t<128>(a, plan, ws, status);
}

}  // namespace fa
