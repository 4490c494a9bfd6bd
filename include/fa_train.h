/*
 * fa_train.h — C ABI of the fused flash-attention training op for one GB300 (sm_103a).
 *
 * What the op computes (flash-attn-training skill, trap list items 5, 8 and 9;
 * llama.cpp PR #57 "train: the exact walk at her real window", commit 86c140d
 * "tiled flash-attention backward"):
 *
 *   forward   s_ij = scale * <q_i, k_j> + mask_ij ; P = softmax over the visible
 *             keys of row i ; O_i = sum_j P_ij v_j ; LSE_i = ln sum_vis exp(s_ij).
 *             A query row with no visible key gets O_i = 0 and LSE_i = 0.
 *   backward  P is recomputed from LSE ; D_i = <dO_i, O_i> ;
 *             dS_ij = P_ij (<dO_i, v_j> - D_i) ; dQ = scale dS K ;
 *             dK = scale dS^T Q ; dV = P^T dO, with dK/dV summed over the query
 *             heads that share a key/value head (native GQA, no head expansion).
 *   accumulate variant: dK/dV are added into caller-owned fp32 buffers
 *             (PR #57, commit 86c140d: a node's gradient is added into an
 *             existing tensor instead of being returned).
 *
 * Conventions (the pages leave these open; these are the plain readings):
 *   - Layout: every tensor is contiguous row-major. Q, O, dO, dQ: [B, Hq, Sq, D];
 *     K, V, dK, dV: [B, Hkv, Sk, D] (or, with p->layout == FA_LAYOUT_BSHD, [B, Sq, Hq, D]
 *     and [B, Sk, Hkv, D]); LSE: [B, Hq, Sq] fp32; mask: [mask_batch, Sq, Sk].
 *   - GQA: query head h reads key/value head h / (Hq / Hkv).
 *   - Additive mask (FA_MASK_ADD_F32): a value <= -1e9 (or -inf) hides the pair
 *     (its probability is exactly 0); any larger value is a bias added after scaling.
 *   - Boolean mask (FA_MASK_BOOL_U8): 1 = attend, 0 = hidden.
 *   - Causal: key j is visible to query i iff j <= q_offset + i (a query chunk
 *     sitting at positions q_offset.. of a longer cached window).
 *   - Sliding window w > 0 (HOT-Step TRAINING.md, "DiT micro-batching": the DiT
 *     self-attention mask is a sliding window plus padded key columns; the page
 *     gives no width convention, so w is the half-width): key j is visible to
 *     query i iff |q_offset + i - j| <= w. With causal only the left half remains
 *     (q_offset + i - w <= j <= q_offset + i). The band is analytic: no mask
 *     tensor is read for it, and key tiles outside it are never loaded.
 *   - Mask, causal rule and window combine: a pair must pass all that are set.
 *   - LSE is a natural logarithm. O, dQ, dK, dV have the input element type;
 *     bf16 results are rounded to nearest even from fp32 accumulators.
 *
 * Ownership and execution:
 *   - All data pointers are DEVICE pointers (CUDA global memory) owned by the caller.
 *     The library never allocates, frees or synchronises; all work is enqueued on
 *     `stream` (a cudaStream_t; NULL = the legacy default stream) and returns
 *     before the GPU has finished.
 *   - `ws` is caller-owned device scratch of at least the size the matching
 *     *_workspace_size() query returns (ws may be NULL when that size is 0). Its
 *     contents need no initialisation and are garbage afterwards. Two calls in
 *     flight at once must not share a workspace.
 *   - Outputs must not alias inputs or each other.
 *
 * Limits: B and Hq at most 65535, Sq and Sk at most 2^24, D 64 or 128, and no tensor of the call
 * (Q, K, V, the mask, the gradients) above 2^40 elements.
 *
 * Errors: parameters are validated before anything is enqueued. A rejected call
 * returns FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED / FA_ERR_WORKSPACE and leaves
 * every buffer untouched. A failed launch returns FA_ERR_CUDA. fa_last_error()
 * gives a one-line description of the most recent failure on the calling thread.
 */
#ifndef FA_TRAIN_H
#define FA_TRAIN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* a shape, pointer, alignment or enum value is invalid */
  FA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. D not in {64, 128}) */
  FA_ERR_WORKSPACE = 3,   /* ws_bytes is smaller than the size query returns */
  FA_ERR_CUDA = 4         /* a CUDA launch or runtime call failed */
} fa_status;

typedef enum fa_dtype { FA_F32 = 0, FA_BF16 = 1 } fa_dtype;

typedef enum fa_mask_kind {
  FA_MASK_NONE = 0,
  FA_MASK_ADD_F32 = 1, /* float32 additive mask, <= -1e9 hides a pair */
  FA_MASK_BOOL_U8 = 2  /* uint8 boolean mask, nonzero = attend */
} fa_mask_kind;

typedef enum fa_kv_format {
  FA_KV_DTYPE = 0, /* K and V are tensors in p->dtype */
  FA_KV_Q8_0 = 1,  /* K and V are a q8_0 cache (fa_kv_q8, the _q8 entry points) */
  FA_KV_F16 = 2    /* K and V are an fp16 cache (IEEE binary16) in p->layout, passed to the plain
                      entry points; needs p->dtype == FA_BF16. llama.cpp PR #57, commit 2394a4c:
                      attention reads the cache in place, in the cache's own type (f16 or q8_0).
                      The library rounds K and V to bf16 (to nearest even) into its workspace
                      ahead of the kernels, since the tensor cores multiply bf16 by bf16; the
                      op then computes as on that bf16 K/V, and dK / dV (bf16, or added into the
                      fp32 accumulators) are the gradients with respect to it. The workspace-size
                      queries include the copy: 2 x B x Hkv x Sk x D x 2 bytes. */
} fa_kv_format;

typedef enum fa_layout {
  FA_LAYOUT_BHSD = 0, /* [B, H, S, D]: each head's rows contiguous */
  FA_LAYOUT_BSHD = 1  /* [B, S, H, D]: each position's heads contiguous (PyTorch's [B, S, H, D]
                         activations, no transpose copy); a row of one head is strided by H * D */
} fa_layout;

typedef struct fa_params {
  int32_t B;          /* batch, >= 1 */
  int32_t Hq;         /* query heads, a multiple of Hkv */
  int32_t Hkv;        /* key/value heads, >= 1 */
  int32_t Sq;         /* query rows per head, >= 0 (0 makes every call a no-op) */
  int32_t Sk;         /* keys per head, >= 1 */
  int32_t D;          /* head dimension: 64 or 128 */
  int32_t dtype;      /* fa_dtype of Q, K, V, O, dO, dQ, dK, dV */
  float scale;        /* softmax scale, finite */
  int32_t causal;     /* 0 or 1 */
  int32_t mask_kind;  /* fa_mask_kind */
  int32_t mask_batch; /* 1 (broadcast over batch) or B; ignored without a mask */
  int32_t window;     /* sliding-window half-width w >= 0; 0 = no window */
  int64_t q_offset;   /* causal or window > 0: key position of query row 0; needs 0 <= q_offset and
                         q_offset + Sq <= Sk. Ignored (taken as 0) when neither is set. */
  int32_t deterministic; /* 0 or 1. 1: the backward's dQ is bitwise reproducible from run to run
                            (its per-key-tile partials are added in a fixed order); dK/dV always are.
                            Costs some backward speed and workspace. */
  int32_t kv_format;  /* fa_kv_format: FA_KV_DTYPE or FA_KV_F16 for the plain entry points,
                         FA_KV_Q8_0 for the _q8 ones (it sizes the workspace) */
  int32_t layout;     /* fa_layout of Q, K, V, O, dO, dQ, dK, dV (and of dk_acc / dv_acc, dk_rows /
                         dv_rows); LSE is always [B, Hq, Sq] and a q8_0 cache's planes always
                         [B, Hkv, Sk, ...] */
  int32_t reserved;   /* must be 0 */
} fa_params;

/* Bytes of scratch the forward needs for these parameters (0 when none). */
FA_API size_t fa_train_fwd_workspace_size(const fa_params* p);

/* Bytes of scratch the backward (both variants) needs for these parameters. */
FA_API size_t fa_train_bwd_workspace_size(const fa_params* p);

/*
 * Forward: writes O [B,Hq,Sq,D] (dtype) and LSE [B,Hq,Sq] (fp32).
 * mask may be NULL only when p->mask_kind == FA_MASK_NONE.
 * Every pointer must be 16-byte aligned.
 */
FA_API fa_status fa_train_fwd(const fa_params* p, const void* q, const void* k, const void* v,
                       const void* mask, void* o, float* lse, void* ws, size_t ws_bytes,
                       void* stream);

/*
 * Backward: from Q, K, V, mask, the forward's O and LSE and the upstream
 * gradient dO, writes (overwrites) dQ [B,Hq,Sq,D], dK and dV [B,Hkv,Sk,D], all
 * in dtype. O and LSE must be the forward's outputs for the same inputs.
 */
FA_API fa_status fa_train_bwd(const fa_params* p, const void* q, const void* k, const void* v,
                       const void* mask, const void* o, const float* lse, const void* dO,
                       void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, void* stream);

/*
 * Accumulating backward: as fa_train_bwd, but dK and dV are ADDED into the
 * caller's fp32 buffers dk_acc/dv_acc [B,Hkv,Sk,D] (fp32 sums, no bf16 rounding
 * of the increment). dQ is overwritten in dtype. Rows of dk_acc/dv_acc whose key
 * is visible to no query receive +0.
 */
FA_API fa_status fa_train_bwd_accum(const fa_params* p, const void* q, const void* k, const void* v,
                             const void* mask, const void* o, const float* lse, const void* dO,
                             void* dq, float* dk_acc, float* dv_acc, void* ws, size_t ws_bytes,
                             void* stream);

/*
 * A q8_0-style quantized K/V cache, read in place (llama.cpp PR #57, commit 2394a4c: a q8_0
 * cache trains in place; the backward admits a quantized source where it only casts a tile).
 * Per (batch, key/value head, key) the cache holds D signed 8-bit values and one fp16 scale per
 * block of 32 consecutive features; the value is x[d] = scale[d / 32] * q[d] (the layout of
 * ggml's q8_0 blocks, split into a value plane and a scale plane). This struct lives in host
 * memory; its pointers are DEVICE pointers, 16-byte aligned:
 *   k_q, v_q: int8 [B, Hkv, Sk, D]; k_d, v_d: fp16 (IEEE binary16 bits) [B, Hkv, Sk, D / 32].
 */
typedef struct fa_kv_q8 {
  const int8_t* k_q;
  const uint16_t* k_d;
  const int8_t* v_q;
  const uint16_t* v_d;
} fa_kv_q8;

/*
 * The op with K and V read from a q8_0 cache (the _q8 entry points): as fa_train_fwd /
 * fa_train_bwd / fa_train_bwd_accum with `k`, `v` replaced by `kv`, and p->kv_format ==
 * FA_KV_Q8_0. The values are rounded to bf16 (x = scale * q, to nearest even) and the op then
 * computes exactly as on a bf16 K/V: the backward dequantizes each CTA's key tile on chip, in
 * place; the forward, whose key tiles are read by every query tile, first dequantizes the cache
 * once into a bf16 copy in its workspace (2 x B x Hkv x Sk x D x 2 bytes, included in
 * fa_train_fwd_workspace_size). dK and dV are the gradients with respect to the dequantized
 * values (bf16 [B, Hkv, Sk, D] for fa_train_bwd_q8, added into fp32 buffers for
 * fa_train_bwd_accum_q8). Needs p->dtype == FA_BF16 (else FA_ERR_UNSUPPORTED).
 */
FA_API fa_status fa_train_fwd_q8(const fa_params* p, const void* q, const fa_kv_q8* kv, const void* mask,
                                 void* o, float* lse, void* ws, size_t ws_bytes, void* stream);
FA_API fa_status fa_train_bwd_q8(const fa_params* p, const void* q, const fa_kv_q8* kv, const void* mask,
                                 const void* o, const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                 void* ws, size_t ws_bytes, void* stream);
FA_API fa_status fa_train_bwd_accum_q8(const fa_params* p, const void* q, const fa_kv_q8* kv, const void* mask,
                                       const void* o, const float* lse, const void* dO, void* dq, float* dk_acc,
                                       float* dv_acc, void* ws, size_t ws_bytes, void* stream);

/*
 * SET_ROWS backward: the gradient of the rows a chunk wrote into its cached K/V window
 * (llama.cpp PR #57, commit 2394a4c: the written source's gradient is the result's
 * gradient at the written rows; the destination, a cache, carries none). With the
 * window's dL/dK or dL/dV accumulated in `acc`, this reads the written rows back out:
 *     out[b, h, r, :] = acc[b, h, idx[r], :]      for r < n_rows,
 * converted to out_dtype (fa_dtype; bf16 rounds to nearest even). acc: fp32 [B, H, S, D];
 * idx: int64 [n_rows] (device memory, shared by every (b, h); repeats allowed); out:
 * [B, H, n_rows, D] in out_dtype. D must be a multiple of 4 in [4, 1024]; acc and out
 * 16-byte aligned, idx 8-byte aligned; out must not overlap acc or idx. An index outside
 * [0, S) cannot be checked before launch: that row of out is written as zeros and
 * 0x40000000 | 950 is recorded in the status word read by fa_device_status().
 * n_rows == 0 is a no-op. Asynchronous on `stream`.
 */
FA_API fa_status fa_set_rows_backward(const float* acc, int32_t B, int32_t H, int32_t S, int32_t D,
                                      const int64_t* idx, int32_t n_rows, void* out, int32_t out_dtype,
                                      void* stream);

/*
 * Accumulating backward fused with the SET_ROWS backward of the chunk's own rows: as
 * fa_train_bwd_accum, and in the same kernel, once a key row's dK/dV sum is complete in
 * dk_acc/dv_acc, the keys rows_begin .. rows_begin + n_rows - 1 are also written, in the
 * input dtype p->dtype, to dk_rows / dv_rows [B, Hkv, n_rows, D]:
 *     dk_rows[b, h, r, :] = dk_acc[b, h, rows_begin + r, :] (after the add), likewise dv.
 * This is the chunk's K/V gradient read back from the window accumulator (the exact walk of
 * PR #57 writes the chunk's K/V at the end of the cached window: rows_begin = q_offset,
 * n_rows = Sq). Needs 0 <= rows_begin and rows_begin + n_rows <= Sk, n_rows >= 0; dk_rows
 * and dv_rows 16-byte aligned and overlapping no other buffer. n_rows == 0 makes this
 * fa_train_bwd_accum. Same workspace as fa_train_bwd_accum.
 */
FA_API fa_status fa_train_bwd_accum_rows(const fa_params* p, const void* q, const void* k, const void* v,
                                         const void* mask, const void* o, const float* lse, const void* dO,
                                         void* dq, float* dk_acc, float* dv_acc, int64_t rows_begin,
                                         int32_t n_rows, void* dk_rows, void* dv_rows, void* ws,
                                         size_t ws_bytes, void* stream);

/*
 * Tracing (optional). Kernels of the op, as named for fa_profile_set_events.
 * FA_KERNEL_FWD: the forward main kernel (plus the split-KV combine when used);
 * FA_KERNEL_BWD_MAIN: the backward main kernel(s) that form dQ/dK/dV;
 * FA_KERNEL_BWD_DSUM: the D = rowsum(dO*O) pass; FA_KERNEL_BWD_DQ_CONVERT: the
 * fp32 -> dtype dQ pass; FA_KERNEL_MASK_CLASSIFY: the mask tile classifier.
 */
typedef enum fa_kernel_id {
  FA_KERNEL_FWD = 0,
  FA_KERNEL_BWD_MAIN = 1,
  FA_KERNEL_BWD_DSUM = 2,
  FA_KERNEL_BWD_DQ_CONVERT = 3,
  FA_KERNEL_MASK_CLASSIFY = 4,
  FA_KERNEL_COUNT = 5
} fa_kernel_id;

/*
 * Make later calls on the calling thread record `start_event` just before and
 * `stop_event` just after the given kernel(s), on the stream they launch on.
 * Both are cudaEvent_t handles owned by the caller (NULL, NULL clears the hook).
 * Returns FA_ERR_INVALID_ARG for an unknown kernel id. Recording errors are
 * reported by the op call that records them (FA_ERR_CUDA).
 */
FA_API fa_status fa_profile_set_events(int kernel, void* start_event, void* stop_event);

/* Number of CUDA kernels the library has launched from the calling thread so far. */
FA_API uint64_t fa_profile_launch_count(void);

/*
 * Allocation-free backward (no counterpart in the pages; an addition for callers of this
 * library that cannot allocate device memory: a framework pool or plugin host that owns all of
 * the GPU's memory and hands over only its tensors, or a loop where a cudaMalloc and the
 * device synchronisation it can imply are not allowed). Same arguments, results and errors as
 * fa_train_bwd without ws / ws_bytes: the scratch lives in one static device array of
 * 16 MiB (16777216 bytes) inside the library, which every GPU that loads the library holds
 * until the process exits. Shapes whose fa_train_bwd_workspace_size() exceeds 16 MiB are
 * rejected with FA_ERR_WORKSPACE (and a message in fa_last_error()) before anything runs.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress, once
 * per device, with that device current); make that first call before any stream capture. The
 * address is kept for the life of the process: after cudaDeviceReset (or anything else that
 * tears down and recreates the device's primary context) the array may move, and this entry
 * point must not be called again in that process. The tensors and the stream must belong to
 * the current device: the array is looked up, and the kernels launched, on that device.
 * The library allocates and frees nothing in this call. Every call shares the one array and
 * the kernels re-initialise what must start at zero, so back-to-back calls on one stream are
 * fine, but calls that overlap on the GPU (other streams, other host threads) race.
 */
FA_API fa_status fa_train_bwd_noalloc(const fa_params* p, const void* q, const void* k, const void* v,
                                      const void* mask, const void* o, const float* lse, const void* dO,
                                      void* dq, void* dk, void* dv, void* stream);

/*
 * Reads and clears the status word of the current device's kernels: 0 when
 * every wait inside a kernel completed and no kernel found bad data; otherwise
 * the first problem recorded since the last read: 0x80000000 | site when the wait
 * `site` ran out of its time limit (the kernel then stopped early and its outputs
 * are invalid), 0x40000000 | site when a kernel met a device-side argument it
 * could not use (site 950: a row index of fa_set_rows_backward outside [0, S)).
 * Synchronous (waits for the device to finish the copy). Returns FA_ERR_CUDA if
 * no device is usable.
 */
FA_API fa_status fa_device_status(uint32_t* out);

/*
 * Self-test of the failure detection: launches one thread that waits on an mbarrier nothing ever
 * arrives on, with the given limit (1..10000 ms). The wait gives up, writes 0x80000000 | 900 into
 * the status word that fa_device_status() reads, and the kernel returns normally (the CUDA
 * context stays usable). Asynchronous on `stream` like the op calls.
 */
FA_API fa_status fa_train_selftest_wait(uint32_t limit_ms, void* stream);

/*
 * The backward's work plan on the tensor-core path, for inspection (host only: no GPU work, no
 * device needed). One record per CTA of the main kernel, in launch order, 6 int32 each: key tile
 * (128 keys), batch * Hkv + key/value head, part, number of parts of that key tile (1: not split),
 * and the query rows [first, end) the CTA walks (for every query head of the GQA group). A key
 * tile cut into parts has its rows partitioned by them; the last part to finish sums the parts'
 * fp32 partials in part order. Writes min(*n_ctas, cap) records to `records` (may be NULL when
 * cap is 0) and the CTA count to *n_ctas. FA_ERR_UNSUPPORTED when the call would not take the
 * tensor-core path.
 */
FA_API fa_status fa_train_bwd_plan(const fa_params* p, int32_t* records, int32_t cap, int32_t* n_ctas);

/*
 * The forward's launch on the tensor-core path, for inspection (host only: no GPU work; without
 * a device the SM count is taken as 152). A work unit is 256 query rows (two 128-row tiles) of
 * one (batch, query head). Writes the main kernel's CTA count to *ctas, the key splits per unit
 * to *kv_splits (> 1 when the units are fewer than the SMs and the keys are long enough: each CTA
 * then takes one split, and a combine kernel merges the partial outputs), and 1 to *persistent
 * when the CTAs are persistent (one per SM, each running several units in sequence: more units
 * than SMs, no mask and no key split), else 0 (one unit, or one split of it, per CTA). All three
 * pointers must be non-null. FA_ERR_UNSUPPORTED when the call would not take the tensor-core
 * path (fp32, or D outside {64, 128}).
 */
FA_API fa_status fa_train_fwd_plan(const fa_params* p, int32_t* ctas, int32_t* kv_splits, int32_t* persistent);

/* Static description of a status code. */
FA_API const char* fa_status_str(fa_status s);

/* One-line description of the most recent failure on the calling thread ("" if none). */
FA_API const char* fa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_TRAIN_H */
