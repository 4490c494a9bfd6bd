// Internal interface between the C-ABI layer (fa_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fa {

enum : int { DT_F32 = 0, DT_BF16 = 1 };
enum : int { MK_NONE = 0, MK_ADD = 1, MK_BOOL = 2 };

// Tile-map codes produced by the mask classifier (one byte per 128x128 tile).
enum : uint8_t { TILE_SKIP = 0, TILE_OPEN = 1, TILE_MIXED = 2 };

struct Shape {
  int B, Hq, Hkv, Sq, Sk, D;
  int dtype;
  float scale;
  int causal;
  int mask_kind;
  int mask_batch;
  int window;          // sliding-window half-width, 0 = none
  long long q_offset;  // key position of query row 0 (0 unless causal or windowed)
  int deterministic;   // the backward adds dQ partials in a fixed order
  int kv_format;       // fa_kv_format of the call (read by the host side only)
  int layout;          // 0: [B, H, S, D]; 1: [B, S, H, D] (Q, K, V, O, dO, dQ, dK, dV)
};

// Offset (elements) of row 0 of head h of batch b, and the distance between consecutive rows of
// one head, in a [B, H, S, D] or [B, S, H, D] tensor with D = s.D.
__host__ __device__ inline size_t head_base(const Shape& s, int b, int h, int H, long long S) {
  return s.layout ? ((size_t)b * (size_t)S * H + h) * (size_t)s.D : ((size_t)b * H + h) * (size_t)S * s.D;
}
__host__ __device__ inline size_t row_stride(const Shape& s, int H) {
  return s.layout ? (size_t)H * s.D : (size_t)s.D;
}

struct FwdArgs {
  Shape s;
  const void* q;
  const void* k;
  const void* v;
  const void* mask;
  void* o;
  float* lse;
  cudaStream_t stream;
  int kv_layout = -1;   // layout of k, v when it differs from s.layout (a dequantized q8_0 cache)
};

struct BwdArgs {
  Shape s;
  const void* q;
  const void* k;
  const void* v;
  const void* mask;
  const void* o;
  const float* lse;
  const void* dO;
  void* dq;
  void* dk;  // dtype when !accum, fp32 accumulator when accum
  void* dv;
  bool accum;
  cudaStream_t stream;
  // accumulate only: keys [rows_begin, rows_begin + n_rows) are also written, after the add, to
  // dk_rows / dv_rows [B, Hkv, n_rows, D] in dtype (n_rows == 0: none)
  long long rows_begin = 0;
  int n_rows = 0;
  void* dk_rows = nullptr;
  void* dv_rows = nullptr;
  // q8_0 K/V cache (k, v unused when kq != nullptr): int8 [B, Hkv, Sk, D] + fp16 [B, Hkv, Sk, D / 32]
  const int8_t* kq = nullptr;
  const void* kd = nullptr;
  const int8_t* vq = nullptr;
  const void* vd = nullptr;
};

// Carve-up of the caller's workspace. Offsets are 256-byte aligned.
struct FwdPlan {
  bool tensor_core;   // tcgen05 path (bf16) vs SIMT fp32 path
  int kv_splits;      // > 1: split-KV partials + combine
  size_t tilemap_off, tilemap_bytes;
  size_t part_o_off, part_o_bytes;     // fp32 [splits, B, Hq, Sq, D]
  size_t part_ml_off, part_ml_bytes;   // fp32 [splits, B, Hq, Sq, 2]
  size_t kvbf_off, kvbf_bytes;         // q8_0 or f16 cache: bf16 K then V (q8_0: [B, Hkv, Sk, D]; f16: the layout)
  size_t total;
};

struct BwdPlan {
  bool tensor_core;
  size_t tilemap_off, tilemap_bytes;
  size_t dsum_off, dsum_bytes;   // fp32 [B, Hq, Sq]
  size_t dqacc_off, dqacc_bytes; // fp32 [groups, B, Hq, Sq, D]
  size_t turn_off, turn_bytes;   // deterministic: int32 [groups, B, Hq, ceil(Sq / 128)] dQ turn counters
  size_t part_off, part_bytes;   // split key tiles: fp32 dV/dK partials [B * Hkv, slots, 2, D / 4, 128] float4
  size_t cnt_off, cnt_bytes;     // split key tiles: int32 [B * Hkv, slots, 2] part tickets / partials written
  size_t kvbf_off, kvbf_bytes;   // f16 cache: bf16 K then V, in the call's layout
  size_t total;
};

// Sets the calling thread's fa_last_error() text.
void set_error_message(const char* msg);

// Device status word the kernels' bounded waits report into (nullptr if unavailable).
unsigned* device_status_ptr();

// Self-test of the kernels' bounded waits (see fa_train_selftest_wait).
constexpr unsigned kSelfTestSite = 900;
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t st);

// Tracing hooks (fa_profile_set_events): per-thread events recorded around a
// kernel family, and a per-thread launch counter.
enum : int { KID_FWD = 0, KID_BWD_MAIN = 1, KID_BWD_DSUM = 2, KID_BWD_DQCONV = 3, KID_MASK = 4, KID_COUNT = 5 };
cudaError_t prof_begin(int kid, cudaStream_t st);
cudaError_t prof_end(int kid, cudaStream_t st);
void count_launches(int n);

// Deterministic dQ: the key tiles form groups of det_group(s) consecutive 128-key tiles; each group
// adds its partials in key-tile order into its own fp32 dQ accumulator, and the dQ convert pass
// sums the groups' accumulators in group order. Without it there is one accumulator. Every group
// costs the D pass and the convert pass one more accumulator to zero and read; a longer group
// chains more ordered adds per query tile. Groups of 32 (measured: causal S = 4096 step 0.737 ->
// 0.658 ms against groups of 8) unless the keys far outnumber the query tiles, where every key
// tile adds to the same few query tiles and the chains are the bound (the 67,584-key window over
// 4 query tiles: 1.62 ms with groups of 8, 1.69 with 32).
__host__ __device__ inline int det_group(const Shape& s) {
  const int nkt = (s.Sk + 127) / 128, nqt = (s.Sq + 127) / 128;
  return nkt <= 4 * nqt ? 32 : 8;
}
inline int dq_groups(const Shape& s) { return s.deterministic ? ((s.Sk + 127) / 128 + det_group(s) - 1) / det_group(s) : 1; }

// Backward work split (tensor-core path). A key tile's query steps may be cut into up to kMaxParts
// parts (consecutive query tiles), each a CTA of its own that writes fp32 dK/dV partials; the
// part that finishes last sums all of them in part order and writes dK/dV. Two cases:
//  - the key tiles of all (batch, key/value head) pairs are fewer than the SMs: key tiles well
//    above the per-SM share are cut into even parts, units run heaviest first;
//  - a full grid whose heaviest key tiles are longer than the per-SM share (the causal rule): the
//    heavy tiles shed their last query tiles into a second part, and the CTAs are packed onto the
//    SMs ahead of time (best-fit decreasing on a cost per step and per CTA); the launch order is
//    the packing's planned start order, so the block scheduler, which hands the next block to the
//    first SM that frees up, reproduces it.
constexpr int kMaxUnits = 512;
constexpr int kMaxParts = 8;
constexpr int kMaxCtas = 1024;
struct BwdSplit {
  int n_units = 0;        // 0: no split, one CTA per key tile in key-tile order
  int n_slots = 0;        // partial slots per (batch, key/value head)
  int n_ctas = 0;         // 0: CTA i runs unit i / (B * Hkv) for (batch, kv head) i % (B * Hkv)
  uint32_t units[kMaxUnits];   // kt | part << 12 | nparts << 16 | slot << 20
  uint32_t range[kMaxUnits];   // the part's query tiles, from the key tile's first: first | end << 16
  uint32_t ctas[kMaxCtas];     // launch order: unit | (batch * Hkv + kv head) << 16
};
void plan_bwd_split(const Shape& s, BwdSplit& out);
// The plan as records (see fa_train_bwd_plan): returns the CTA count, writes at most `cap` records.
int bwd_plan_records(const Shape& s, int32_t* rec, int cap);

// Streaming multiprocessors of the current device (queried once).
int sm_count();

FwdPlan plan_fwd(const Shape& s);
BwdPlan plan_bwd(const Shape& s);

// SIMT fp32 kernels (any dtype, D in {64, 128}).
cudaError_t simt_fwd(const FwdArgs& a);
cudaError_t simt_bwd(const BwdArgs& a, float* dsum);

// Helper passes shared by both paths.
// dsum also zeroes `groups` fp32 dQ accumulators (none when dq_acc_to_zero is null) and n_zero
// words at zero_words; dq_convert sums the groups in order, scales and converts to the dtype.
cudaError_t launch_dsum(const BwdArgs& a, float* dsum, float* dq_acc_to_zero, int groups = 1,
                        uint32_t* zero_words = nullptr, int n_zero = 0);
cudaError_t launch_dq_convert(const BwdArgs& a, const float* dq_acc, int groups = 1);
cudaError_t launch_mask_classify(const Shape& s, const void* mask, uint8_t* tilemap, cudaStream_t st);

// q8_0 cache -> bf16 [B, Hkv, Sk, D] (x = scale[d / 32] * q[d], rounded to nearest even).
cudaError_t launch_q8_dequant(const Shape& s, const int8_t* xq, const void* xd, void* out, cudaStream_t st);
// fp16 -> bf16, n elements (a multiple of 8; 16-byte aligned buffers), rounded to nearest even.
cudaError_t launch_f16_to_bf16(const void* x, void* out, long long n, cudaStream_t st);

// SET_ROWS backward gather (fa_set_rows_backward): out[bh, r, :] = acc[bh, idx[r], :].
constexpr unsigned kSiteRowIndex = 950;
cudaError_t launch_set_rows_backward(const float* acc, int heads, int S, int D, const int64_t* idx, int n_rows,
                                     void* out, int out_dtype, unsigned* status, cudaStream_t st);
// The same gather for the contiguous keys [row0, row0 + n_rows) of dK / dV accumulators (in s.dtype).
cudaError_t launch_rows_copy(const Shape& s, const float* dk_acc, const float* dv_acc, long long row0, int n_rows,
                             void* dk_rows, void* dv_rows, cudaStream_t st);

// tcgen05 paths (bf16, D in {64, 128}).
bool tc_fwd_supported(const Shape& s);
bool tc_bwd_supported(const Shape& s);
// bf16 tensor of B x H heads of S rows of D features ([B, H, S, D] when layout == 0, [B, S, H, D]
// when 1) viewed as (D, S, H, B) with 64 x box_rows x 1 x 1 boxes and the 128-byte swizzle.
cudaError_t make_tmap_4d(struct CUtensorMap_st* map, const void* base, int layout, int B, int H, int S, int D,
                         int box_rows);
cudaError_t make_tmap_f32_bhsd(struct CUtensorMap_st* map, const void* base, int S, int heads, int D, int box_rows);
cudaError_t make_tmap_f32_bhsd_sw128(struct CUtensorMap_st* map, const void* base, int S, int heads, int D,
                                     int box_rows);
int tc_fwd_kv_splits(const Shape& s);
// Launch shape of the tensor-core forward: CTAs and whether they are persistent (each chains the
// key tiles of several 256-row units: more units than SMs, no mask, no key split).
struct FwdLaunch {
  long long ctas;
  bool persistent;
};
FwdLaunch tc_fwd_launch(const Shape& s, int kv_splits);
cudaError_t tc_fwd(const FwdArgs& a, const FwdPlan& plan, char* ws);
cudaError_t tc_bwd(const BwdArgs& a, const BwdPlan& plan, char* ws);

}  // namespace fa
