// C-ABI layer of the fused attention training op: parameter validation,
// workspace planning and dispatch to the kernels. Nothing here allocates,
// frees or synchronises; every launch goes on the caller's stream.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "fa_train.h"
#include "fa_internal.h"

namespace fa {
namespace {

thread_local char g_last_error[256] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

constexpr int kMaxSeq = 1 << 24;
// Largest element count of one tensor (2^40: terabytes, more than a GB300 holds). Keeps every byte
// count of the validation and every 64-bit offset in the kernels far from overflow.
constexpr double kMaxElems = 1099511627776.0;

bool too_large(double a, double b, double c, double d) { return a * b * c * d > kMaxElems; }

fa_status check_params(const fa_params* p, Shape& s) {
  g_last_error[0] = '\0';
  if (p == nullptr) { set_error("params is NULL"); return FA_ERR_INVALID_ARG; }
  if (p->B < 1 || p->B > 65535) { set_error("B=%d outside [1, 65535]", p->B); return FA_ERR_INVALID_ARG; }
  if (p->Hkv < 1 || p->Hq < 1 || p->Hq > 65535) {
    set_error("Hq=%d, Hkv=%d: need 1 <= Hkv, 1 <= Hq <= 65535", p->Hq, p->Hkv); return FA_ERR_INVALID_ARG;
  }
  if (p->Hq % p->Hkv != 0) { set_error("Hq=%d is not a multiple of Hkv=%d", p->Hq, p->Hkv); return FA_ERR_INVALID_ARG; }
  if (p->Sq < 0 || p->Sq > kMaxSeq) { set_error("Sq=%d outside [0, %d]", p->Sq, kMaxSeq); return FA_ERR_INVALID_ARG; }
  if (p->Sk < 1 || p->Sk > kMaxSeq) { set_error("Sk=%d outside [1, %d]", p->Sk, kMaxSeq); return FA_ERR_INVALID_ARG; }
  if (p->D <= 0) { set_error("D=%d must be positive", p->D); return FA_ERR_INVALID_ARG; }
  if (p->D != 64 && p->D != 128) { set_error("D=%d unsupported (64 or 128)", p->D); return FA_ERR_UNSUPPORTED; }
  if (p->dtype != FA_F32 && p->dtype != FA_BF16) { set_error("dtype=%d invalid", p->dtype); return FA_ERR_INVALID_ARG; }
  if (!std::isfinite(p->scale)) { set_error("scale is not finite"); return FA_ERR_INVALID_ARG; }
  if (p->causal != 0 && p->causal != 1) { set_error("causal=%d must be 0 or 1", p->causal); return FA_ERR_INVALID_ARG; }
  if (p->mask_kind < FA_MASK_NONE || p->mask_kind > FA_MASK_BOOL_U8) {
    set_error("mask_kind=%d invalid", p->mask_kind); return FA_ERR_INVALID_ARG;
  }
  if (p->mask_kind != FA_MASK_NONE && p->mask_batch != 1 && p->mask_batch != p->B) {
    set_error("mask_batch=%d must be 1 or B=%d", p->mask_batch, p->B); return FA_ERR_INVALID_ARG;
  }
  if (p->window < 0) { set_error("window=%d must be >= 0 (0 = no window)", p->window); return FA_ERR_INVALID_ARG; }
  if (p->deterministic != 0 && p->deterministic != 1) {
    set_error("deterministic=%d must be 0 or 1", p->deterministic); return FA_ERR_INVALID_ARG;
  }
  if (p->kv_format != FA_KV_DTYPE && p->kv_format != FA_KV_Q8_0 && p->kv_format != FA_KV_F16) {
    set_error("kv_format=%d invalid", p->kv_format); return FA_ERR_INVALID_ARG;
  }
  if (p->kv_format == FA_KV_F16 && p->dtype != FA_BF16) {
    set_error("an f16 K/V cache needs bf16 queries (dtype=%d)", p->dtype); return FA_ERR_UNSUPPORTED;
  }
  if (p->layout != FA_LAYOUT_BHSD && p->layout != FA_LAYOUT_BSHD) {
    set_error("layout=%d invalid", p->layout); return FA_ERR_INVALID_ARG;
  }
  if (p->reserved != 0) { set_error("reserved field must be 0"); return FA_ERR_INVALID_ARG; }
  if (too_large(p->B, p->Hq, p->Sq, p->D) || too_large(p->B, p->Hkv, p->Sk, p->D) ||
      (p->mask_kind != FA_MASK_NONE && too_large(p->mask_batch, p->Sq, p->Sk, 1))) {
    set_error("a tensor of these shapes would hold more than 2^40 elements"); return FA_ERR_INVALID_ARG;
  }
  const bool positioned = p->causal || p->window > 0;
  if (positioned && (p->q_offset < 0 || p->q_offset + p->Sq > p->Sk)) {
    set_error("q_offset=%lld with Sq=%d needs 0 <= q_offset and q_offset + Sq <= Sk=%d",
              (long long)p->q_offset, p->Sq, p->Sk);
    return FA_ERR_INVALID_ARG;
  }
  s.B = p->B; s.Hq = p->Hq; s.Hkv = p->Hkv; s.Sq = p->Sq; s.Sk = p->Sk; s.D = p->D;
  s.dtype = p->dtype; s.scale = p->scale; s.causal = p->causal; s.mask_kind = p->mask_kind;
  s.mask_batch = p->mask_kind == FA_MASK_NONE ? 1 : p->mask_batch;
  // with q_offset + Sq <= Sk no pair is further apart than Sk - 1, so a window of Sk or more hides
  // nothing: drop it so no kernel pays for it
  s.window = (p->window > 0 && p->window < p->Sk) ? p->window : 0;
  s.q_offset = (p->causal || s.window > 0) ? (long long)p->q_offset : 0;
  s.deterministic = p->deterministic;
  s.kv_format = p->kv_format;
  s.layout = p->layout;
  return FA_OK;
}

size_t elem_size(const Shape& s) { return s.dtype == DT_BF16 ? 2 : 4; }
size_t q_bytes(const Shape& s) { return (size_t)s.B * s.Hq * s.Sq * s.D * elem_size(s); }
size_t kv_bytes(const Shape& s, size_t es) { return (size_t)s.B * s.Hkv * s.Sk * s.D * es; }
size_t mask_bytes(const Shape& s) {
  if (s.mask_kind == MK_NONE) return 0;
  return (size_t)s.mask_batch * s.Sq * s.Sk * (s.mask_kind == MK_ADD ? 4 : 1);
}

struct Span { const void* p; size_t n; const char* name; };

bool overlaps(const Span& a, const Span& b) {
  if (a.p == nullptr || b.p == nullptr || a.n == 0 || b.n == 0) return false;
  const uintptr_t a0 = (uintptr_t)a.p, b0 = (uintptr_t)b.p;
  return a0 < b0 + b.n && b0 < a0 + a.n;
}

fa_status check_buffers(const Span* in, int nin, const Span* out, int nout) {
  for (int i = 0; i < nin + nout; ++i) {
    const Span& x = i < nin ? in[i] : out[i - nin];
    if (x.n == 0) continue;
    if (x.p == nullptr) { set_error("%s is NULL", x.name); return FA_ERR_INVALID_ARG; }
    if ((uintptr_t)x.p % 16 != 0) { set_error("%s is not 16-byte aligned", x.name); return FA_ERR_INVALID_ARG; }
  }
  for (int o = 0; o < nout; ++o) {
    for (int i = 0; i < nin; ++i)
      if (overlaps(out[o], in[i])) { set_error("output %s overlaps input %s", out[o].name, in[i].name); return FA_ERR_INVALID_ARG; }
    for (int o2 = o + 1; o2 < nout; ++o2)
      if (overlaps(out[o], out[o2])) { set_error("outputs %s and %s overlap", out[o].name, out[o2].name); return FA_ERR_INVALID_ARG; }
  }
  return FA_OK;
}

fa_status check_ws(void* ws, size_t ws_bytes, size_t need, const Span* bufs, int n) {
  if (ws_bytes < need) { set_error("workspace %zu bytes < %zu needed", ws_bytes, need); return FA_ERR_WORKSPACE; }
  if (need == 0) return FA_OK;
  if (ws == nullptr) { set_error("workspace is NULL"); return FA_ERR_WORKSPACE; }
  if ((uintptr_t)ws % kAlign != 0) { set_error("workspace is not %zu-byte aligned", kAlign); return FA_ERR_INVALID_ARG; }
  const Span w{ws, need, "workspace"};
  for (int i = 0; i < n; ++i)
    if (overlaps(w, bufs[i])) { set_error("workspace overlaps %s", bufs[i].name); return FA_ERR_INVALID_ARG; }
  return FA_OK;
}

fa_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return FA_OK;
  set_error("%s: %s", what, cudaGetErrorString(e));
  return FA_ERR_CUDA;
}

// The tcgen05 path takes bf16 inputs; fp32 inputs stay on the SIMT fp32 path.
bool use_tc_fwd(const Shape& s) { return s.dtype == DT_BF16 && tc_fwd_supported(s); }
bool use_tc_bwd(const Shape& s) { return s.dtype == DT_BF16 && tc_bwd_supported(s); }

// Status word of the bounded device waits (0 = fine; 0x80000000 | site = a wait ran out).
__device__ unsigned int g_fa_device_status = 0;
constexpr int kMaxDevices = 64;
unsigned* g_status_ptr[kMaxDevices] = {};

thread_local cudaEvent_t g_prof_start[KID_COUNT] = {};
thread_local cudaEvent_t g_prof_stop[KID_COUNT] = {};
thread_local uint64_t g_launches = 0;

}  // namespace

cudaError_t prof_begin(int kid, cudaStream_t st) {
  return g_prof_start[kid] ? cudaEventRecord(g_prof_start[kid], st) : cudaSuccess;
}
cudaError_t prof_end(int kid, cudaStream_t st) {
  return g_prof_stop[kid] ? cudaEventRecord(g_prof_stop[kid], st) : cudaSuccess;
}
void count_launches(int n) { g_launches += (uint64_t)n; }

void set_error_message(const char* msg) { set_error("%s", msg); }

unsigned* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  // host threads making their first call at the same time fill the per-device cache under a lock
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_device_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_status_ptr[dev];
}

FwdPlan plan_fwd(const Shape& s) {
  FwdPlan p{};
  p.tensor_core = use_tc_fwd(s);
  p.kv_splits = p.tensor_core ? tc_fwd_kv_splits(s) : 1;
  size_t off = 0;
  if (p.tensor_core && s.mask_kind != MK_NONE) {
    p.tilemap_off = off;
    p.tilemap_bytes = (size_t)s.mask_batch * ((s.Sq + 127) / 128) * ((s.Sk + 127) / 128);
    off = align_up(off + p.tilemap_bytes);
  }
  if (p.tensor_core && s.kv_format != FA_KV_DTYPE) {
    // the q8_0 or f16 cache as bf16 K then V (read by every query tile of the forward)
    p.kvbf_off = off;
    p.kvbf_bytes = 2 * (size_t)s.B * s.Hkv * s.Sk * s.D * 2;
    off = align_up(off + p.kvbf_bytes);
  }
  if (p.kv_splits > 1) {
    const size_t rows = (size_t)s.B * s.Hq * s.Sq;
    p.part_o_off = off;
    p.part_o_bytes = (size_t)p.kv_splits * rows * s.D * 4;
    off = align_up(off + p.part_o_bytes);
    p.part_ml_off = off;
    p.part_ml_bytes = (size_t)p.kv_splits * rows * 2 * 4;
    off = align_up(off + p.part_ml_bytes);
  }
  p.total = off;
  return p;
}

BwdPlan plan_bwd(const Shape& s) {
  BwdPlan p{};
  p.tensor_core = use_tc_bwd(s);
  size_t off = 0;
  const size_t rows = (size_t)s.B * s.Hq * s.Sq;
  if (p.tensor_core && s.mask_kind != MK_NONE) {
    p.tilemap_off = off;
    p.tilemap_bytes = (size_t)s.mask_batch * ((s.Sq + 127) / 128) * ((s.Sk + 127) / 128);
    off = align_up(off + p.tilemap_bytes);
  }
  p.dsum_off = off;
  p.dsum_bytes = rows * 4;
  off = align_up(off + p.dsum_bytes);
  if (p.tensor_core) {
    p.dqacc_off = off;
    p.dqacc_bytes = (size_t)dq_groups(s) * rows * s.D * 4;
    off = align_up(off + p.dqacc_bytes);
    if (s.deterministic) {
      // one turn counter per (key-tile group, batch, query head, 128-row query tile)
      p.turn_off = off;
      p.turn_bytes = (size_t)dq_groups(s) * s.B * s.Hq * ((s.Sq + 127) / 128) * 4;
      off = align_up(off + p.turn_bytes);
    }
    static thread_local BwdSplit split;   // large; planned again at launch
    plan_bwd_split(s, split);
    if (split.n_units > 0) {
      p.part_off = off;
      p.part_bytes = (size_t)s.B * s.Hkv * split.n_slots * 2 * 128 * s.D * 4;
      off = align_up(off + p.part_bytes);
      p.cnt_off = off;
      p.cnt_bytes = (size_t)s.B * s.Hkv * split.n_slots * 2 * 4;
      off = align_up(off + p.cnt_bytes);
    }
    if (s.kv_format == FA_KV_F16) {
      p.kvbf_off = off;
      p.kvbf_bytes = 2 * (size_t)s.B * s.Hkv * s.Sk * s.D * 2;
      off = align_up(off + p.kvbf_bytes);
    }
  }
  p.total = off;
  return p;
}

}  // namespace fa

using namespace fa;

extern "C" {

size_t fa_train_fwd_workspace_size(const fa_params* p) {
  Shape s;
  if (check_params(p, s) != FA_OK) return 0;
  return plan_fwd(s).total;
}

size_t fa_train_bwd_workspace_size(const fa_params* p) {
  Shape s;
  if (check_params(p, s) != FA_OK) return 0;
  return plan_bwd(s).total;
}

// The K/V inputs of a call: tensors in the params' dtype or fp16, or a q8_0 cache (value and scale planes).
struct KvIn {
  const void* k;
  const void* v;
  const fa_kv_q8* q8;
};

// Appends the K/V input spans to `in` (2 for tensors, 4 for a q8_0 cache).
static fa_status kv_spans(const Shape& s, const KvIn& kv, Span* in, int& n) {
  const bool q8 = s.kv_format == FA_KV_Q8_0;
  if ((kv.q8 != nullptr) != q8) {
    set_error(q8 ? "kv_format is FA_KV_Q8_0: use the _q8 entry points" : "the _q8 entry points need kv_format FA_KV_Q8_0");
    return FA_ERR_INVALID_ARG;
  }
  if (kv.q8 == nullptr) {
    const size_t es = s.kv_format == FA_KV_F16 ? 2 : elem_size(s);
    in[n++] = {kv.k, kv_bytes(s, es), "k"};
    in[n++] = {kv.v, kv_bytes(s, es), "v"};
    return FA_OK;
  }
  if (s.dtype != DT_BF16) { set_error("a q8_0 K/V cache needs bf16 queries (dtype=%d)", s.dtype); return FA_ERR_UNSUPPORTED; }
  const size_t scales = (size_t)s.B * s.Hkv * s.Sk * (s.D / 32) * 2;
  in[n++] = {kv.q8->k_q, kv_bytes(s, 1), "k_q"};
  in[n++] = {kv.q8->k_d, scales, "k_d"};
  in[n++] = {kv.q8->v_q, kv_bytes(s, 1), "v_q"};
  in[n++] = {kv.q8->v_d, scales, "v_d"};
  return FA_OK;
}

// An fp16 cache rounded to bf16 K then V at `dst` (2 x B x Hkv x Sk x D x 2 bytes of workspace), in the
// call's layout: the tensor cores multiply bf16 by bf16. Points k, v at the copies.
static fa_status cast_f16_cache(const Shape& s, const KvIn& kv, char* dst, cudaStream_t st, const void*& k,
                                const void*& v) {
  const long long n = (long long)s.B * s.Hkv * s.Sk * s.D;
  char* vdst = dst + (size_t)n * 2;
  cudaError_t e = launch_f16_to_bf16(kv.k, dst, n, st);
  if (e == cudaSuccess) e = launch_f16_to_bf16(kv.v, vdst, n, st);
  if (e != cudaSuccess) return cuda_status(e, "f16 cache cast launch");
  k = dst;
  v = vdst;
  return FA_OK;
}

static fa_status fwd_common(const fa_params* p, const void* q, const KvIn& kv, const void* mask, void* o, float* lse,
                            void* ws, size_t ws_bytes, void* stream) {
  Shape s;
  fa_status st = check_params(p, s);
  if (st != FA_OK) return st;
  Span in[7];
  int nin = 0;
  in[nin++] = {q, q_bytes(s), "q"};
  if ((st = kv_spans(s, kv, in, nin)) != FA_OK) return st;
  in[nin++] = {mask, mask_bytes(s), "mask"};
  const Span out[] = {{o, q_bytes(s), "o"}, {lse, (size_t)s.B * s.Hq * s.Sq * 4, "lse"}};
  if ((st = check_buffers(in, nin, out, 2)) != FA_OK) return st;
  const FwdPlan plan = plan_fwd(s);
  Span all[9];
  for (int i = 0; i < nin; ++i) all[i] = in[i];
  all[nin] = out[0];
  all[nin + 1] = out[1];
  if ((st = check_ws(ws, ws_bytes, plan.total, all, nin + 2)) != FA_OK) return st;
  if (s.Sq == 0) return FA_OK;
  if (s.kv_format != FA_KV_DTYPE && !plan.tensor_core) {
    set_error("a quantized or f16 K/V cache needs the tensor-core path"); return FA_ERR_UNSUPPORTED;
  }

  FwdArgs a{s, q, kv.k, kv.v, mask, o, lse, (cudaStream_t)stream};
  cudaError_t e = cudaSuccess;
  if (s.kv_format == FA_KV_F16 && (st = cast_f16_cache(s, kv, (char*)ws + plan.kvbf_off, a.stream, a.k, a.v)) != FA_OK)
    return st;
  if (kv.q8 != nullptr) {
    // every query tile reads every key tile: dequantize the cache once, then run the bf16 kernel on it
    char* kbf = (char*)ws + plan.kvbf_off;
    char* vbf = kbf + plan.kvbf_bytes / 2;
    e = launch_q8_dequant(s, kv.q8->k_q, kv.q8->k_d, kbf, a.stream);
    if (e == cudaSuccess) e = launch_q8_dequant(s, kv.q8->v_q, kv.q8->v_d, vbf, a.stream);
    if (e != cudaSuccess) return cuda_status(e, "q8_0 dequantize launch");
    a.k = kbf;
    a.v = vbf;
    a.kv_layout = 0;   // the copy is [B, Hkv, Sk, D] like the cache's planes
  }
  e = plan.tensor_core ? tc_fwd(a, plan, (char*)ws) : simt_fwd(a);
  return cuda_status(e, "forward launch");
}

fa_status fa_train_fwd(const fa_params* p, const void* q, const void* k, const void* v, const void* mask, void* o,
                       float* lse, void* ws, size_t ws_bytes, void* stream) {
  return fwd_common(p, q, KvIn{k, v, nullptr}, mask, o, lse, ws, ws_bytes, stream);
}

fa_status fa_train_fwd_q8(const fa_params* p, const void* q, const fa_kv_q8* kv, const void* mask, void* o,
                          float* lse, void* ws, size_t ws_bytes, void* stream) {
  if (kv == nullptr) { g_last_error[0] = '\0'; set_error("kv is NULL"); return FA_ERR_INVALID_ARG; }
  return fwd_common(p, q, KvIn{nullptr, nullptr, kv}, mask, o, lse, ws, ws_bytes, stream);
}

// Rows of the accumulator written back out by the fused SET_ROWS backward (n_rows == 0: none).
struct RowsOut {
  long long begin = 0;
  int n = 0;
  void* dk = nullptr;
  void* dv = nullptr;
};

static fa_status bwd_common(const fa_params* p, const void* q, const KvIn& kv, const void* mask,
                            const void* o, const float* lse, const void* dO, void* dq, void* dk, void* dv,
                            bool accum, void* ws, size_t ws_bytes, void* stream, const RowsOut& rb = RowsOut{}) {
  Shape s;
  fa_status st = check_params(p, s);
  if (st != FA_OK) return st;
  const size_t es = elem_size(s);
  const size_t rows = (size_t)s.B * s.Hq * s.Sq;
  Span in[10];
  int nin = 0;
  in[nin++] = {q, q_bytes(s), "q"};
  if ((st = kv_spans(s, kv, in, nin)) != FA_OK) return st;
  in[nin++] = {mask, mask_bytes(s), "mask"};
  in[nin++] = {o, q_bytes(s), "o"};
  in[nin++] = {lse, rows * 4, "lse"};
  in[nin++] = {dO, q_bytes(s), "dO"};
  const size_t gk = accum ? kv_bytes(s, 4) : kv_bytes(s, es);
  if (rb.n < 0 || rb.begin < 0 || rb.begin + rb.n > s.Sk) {
    set_error("rows [%lld, %lld) outside the %d keys", rb.begin, rb.begin + rb.n, s.Sk);
    return FA_ERR_INVALID_ARG;
  }
  const size_t gr = (size_t)s.B * s.Hkv * rb.n * s.D * es;
  const Span out[] = {{dq, q_bytes(s), "dq"}, {dk, gk, accum ? "dk_acc" : "dk"}, {dv, gk, accum ? "dv_acc" : "dv"},
                      {rb.dk, gr, "dk_rows"}, {rb.dv, gr, "dv_rows"}};
  const int n_out = rb.n > 0 ? 5 : 3;
  if ((st = check_buffers(in, nin, out, n_out)) != FA_OK) return st;
  const BwdPlan plan = plan_bwd(s);
  Span all[15];
  for (int i = 0; i < nin; ++i) all[i] = in[i];
  for (int i = 0; i < n_out; ++i) all[nin + i] = out[i];
  if ((st = check_ws(ws, ws_bytes, plan.total, all, nin + n_out)) != FA_OK) return st;

  cudaStream_t cs = (cudaStream_t)stream;
  if (s.Sq == 0) {
    // No query rows: the gradient of every key is zero (the accumulator keeps its contents,
    // and the read-back rows are those contents).
    if (accum) {
      if (rb.n == 0) return FA_OK;
      cudaError_t e = launch_rows_copy(s, static_cast<const float*>(dk), static_cast<const float*>(dv), rb.begin,
                                       rb.n, rb.dk, rb.dv, cs);
      return cuda_status(e, "rows read-back");
    }
    cudaError_t e = cudaMemsetAsync(dk, 0, gk, cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, gk, cs);
    return cuda_status(e, "zero dK/dV");
  }
  if (s.kv_format != FA_KV_DTYPE && !plan.tensor_core) {
    set_error("a quantized or f16 K/V cache needs the tensor-core path"); return FA_ERR_UNSUPPORTED;
  }
  BwdArgs a{s, q, kv.k, kv.v, mask, o, lse, dO, dq, dk, dv, accum, cs};
  if (s.kv_format == FA_KV_F16 && (st = cast_f16_cache(s, kv, (char*)ws + plan.kvbf_off, cs, a.k, a.v)) != FA_OK)
    return st;
  if (kv.q8 != nullptr) {
    a.kq = kv.q8->k_q;
    a.kd = kv.q8->k_d;
    a.vq = kv.q8->v_q;
    a.vd = kv.q8->v_d;
  }
  a.rows_begin = rb.begin;
  a.n_rows = rb.n;
  a.dk_rows = rb.dk;
  a.dv_rows = rb.dv;
  cudaError_t e = plan.tensor_core ? tc_bwd(a, plan, (char*)ws)
                                   : simt_bwd(a, reinterpret_cast<float*>((char*)ws + plan.dsum_off));
  return cuda_status(e, "backward launch");
}

fa_status fa_train_bwd(const fa_params* p, const void* q, const void* k, const void* v, const void* mask,
                       const void* o, const float* lse, const void* dO, void* dq, void* dk, void* dv, void* ws,
                       size_t ws_bytes, void* stream) {
  return bwd_common(p, q, KvIn{k, v, nullptr}, mask, o, lse, dO, dq, dk, dv, false, ws, ws_bytes, stream);
}

fa_status fa_train_bwd_accum(const fa_params* p, const void* q, const void* k, const void* v, const void* mask,
                             const void* o, const float* lse, const void* dO, void* dq, float* dk_acc,
                             float* dv_acc, void* ws, size_t ws_bytes, void* stream) {
  return bwd_common(p, q, KvIn{k, v, nullptr}, mask, o, lse, dO, dq, dk_acc, dv_acc, true, ws, ws_bytes, stream);
}

fa_status fa_train_bwd_q8(const fa_params* p, const void* q, const fa_kv_q8* kv, const void* mask, const void* o,
                          const float* lse, const void* dO, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                          void* stream) {
  if (kv == nullptr) { g_last_error[0] = '\0'; set_error("kv is NULL"); return FA_ERR_INVALID_ARG; }
  return bwd_common(p, q, KvIn{nullptr, nullptr, kv}, mask, o, lse, dO, dq, dk, dv, false, ws, ws_bytes, stream);
}

fa_status fa_train_bwd_accum_q8(const fa_params* p, const void* q, const fa_kv_q8* kv, const void* mask,
                                const void* o, const float* lse, const void* dO, void* dq, float* dk_acc,
                                float* dv_acc, void* ws, size_t ws_bytes, void* stream) {
  if (kv == nullptr) { g_last_error[0] = '\0'; set_error("kv is NULL"); return FA_ERR_INVALID_ARG; }
  return bwd_common(p, q, KvIn{nullptr, nullptr, kv}, mask, o, lse, dO, dq, dk_acc, dv_acc, true, ws, ws_bytes,
                    stream);
}

fa_status fa_train_bwd_accum_rows(const fa_params* p, const void* q, const void* k, const void* v, const void* mask,
                                  const void* o, const float* lse, const void* dO, void* dq, float* dk_acc,
                                  float* dv_acc, int64_t rows_begin, int32_t n_rows, void* dk_rows, void* dv_rows,
                                  void* ws, size_t ws_bytes, void* stream) {
  RowsOut rows;
  rows.begin = rows_begin;
  rows.n = n_rows;
  rows.dk = dk_rows;
  rows.dv = dv_rows;
  return bwd_common(p, q, KvIn{k, v, nullptr}, mask, o, lse, dO, dq, dk_acc, dv_acc, true, ws, ws_bytes, stream,
                    rows);
}

fa_status fa_set_rows_backward(const float* acc, int32_t B, int32_t H, int32_t S, int32_t D, const int64_t* idx,
                               int32_t n_rows, void* out, int32_t out_dtype, void* stream) {
  g_last_error[0] = '\0';
  if (B < 1 || H < 1 || S < 1 || (long long)B * H > 0x7fffffffLL) {
    set_error("B=%d, H=%d, S=%d: each must be >= 1", B, H, S);
    return FA_ERR_INVALID_ARG;
  }
  if (D < 4 || D > 1024 || D % 4 != 0) { set_error("D=%d: a multiple of 4 in [4, 1024]", D); return FA_ERR_INVALID_ARG; }
  if (n_rows < 0) { set_error("n_rows=%d must be >= 0", n_rows); return FA_ERR_INVALID_ARG; }
  if (out_dtype != FA_F32 && out_dtype != FA_BF16) { set_error("out_dtype=%d invalid", out_dtype); return FA_ERR_INVALID_ARG; }
  if (too_large(B, H, S, D) || too_large(B, H, n_rows, D)) {
    set_error("acc or out would hold more than 2^40 elements"); return FA_ERR_INVALID_ARG;
  }
  if (n_rows == 0) return FA_OK;
  if (acc == nullptr || idx == nullptr || out == nullptr) { set_error("acc, idx and out must be non-NULL"); return FA_ERR_INVALID_ARG; }
  if ((uintptr_t)acc % 16 != 0 || (uintptr_t)out % 16 != 0 || (uintptr_t)idx % 8 != 0) {
    set_error("acc and out must be 16-byte aligned, idx 8-byte aligned");
    return FA_ERR_INVALID_ARG;
  }
  const size_t heads = (size_t)B * H;
  const Span in[] = {{acc, heads * S * D * 4, "acc"}, {idx, (size_t)n_rows * 8, "idx"}};
  const Span outs[] = {{out, heads * n_rows * D * (out_dtype == FA_BF16 ? 2 : 4), "out"}};
  for (const Span& a : in)
    if (overlaps(outs[0], a)) { set_error("out overlaps %s", a.name); return FA_ERR_INVALID_ARG; }
  return cuda_status(launch_set_rows_backward(acc, (int)heads, S, D, idx, n_rows, out, out_dtype,
                                              device_status_ptr(), (cudaStream_t)stream),
                     "set_rows backward launch");
}

fa_status fa_train_bwd_plan(const fa_params* p, int32_t* records, int32_t cap, int32_t* n_ctas) {
  Shape s;
  fa_status st = check_params(p, s);
  if (st != FA_OK) return st;
  if (n_ctas == nullptr || cap < 0 || (cap > 0 && records == nullptr)) {
    set_error("n_ctas must be non-null, cap >= 0, records non-null when cap > 0");
    return FA_ERR_INVALID_ARG;
  }
  if (!plan_bwd(s).tensor_core) {
    set_error("this backward does not take the tensor-core path");
    return FA_ERR_UNSUPPORTED;
  }
  *n_ctas = bwd_plan_records(s, records, cap);
  return FA_OK;
}

fa_status fa_train_fwd_plan(const fa_params* p, int32_t* ctas, int32_t* kv_splits, int32_t* persistent) {
  Shape s;
  fa_status st = check_params(p, s);
  if (st != FA_OK) return st;
  if (ctas == nullptr || kv_splits == nullptr || persistent == nullptr) {
    set_error("ctas, kv_splits and persistent must be non-null");
    return FA_ERR_INVALID_ARG;
  }
  const FwdPlan plan = plan_fwd(s);
  if (!plan.tensor_core) {
    set_error("this forward does not take the tensor-core path");
    return FA_ERR_UNSUPPORTED;
  }
  const FwdLaunch l = tc_fwd_launch(s, plan.kv_splits);
  *ctas = (int32_t)l.ctas;
  *kv_splits = plan.kv_splits;
  *persistent = l.persistent ? 1 : 0;
  return FA_OK;
}

fa_status fa_train_selftest_wait(uint32_t limit_ms, void* stream) {
  if (limit_ms == 0 || limit_ms > 10000) {
    set_error("limit_ms=%u outside [1, 10000]", limit_ms);
    return FA_ERR_INVALID_ARG;
  }
  return cuda_status(launch_wait_selftest((unsigned long long)limit_ms * 1000000ull, (cudaStream_t)stream),
                     "wait self-test launch");
}

const char* fa_status_str(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_WORKSPACE: return "workspace too small";
    case FA_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

const char* fa_last_error(void) { return g_last_error; }

fa_status fa_profile_set_events(int kernel, void* start_event, void* stop_event) {
  if (kernel < 0 || kernel >= KID_COUNT) {
    set_error("unknown kernel id %d", kernel);
    return FA_ERR_INVALID_ARG;
  }
  g_prof_start[kernel] = (cudaEvent_t)start_event;
  g_prof_stop[kernel] = (cudaEvent_t)stop_event;
  return FA_OK;
}

uint64_t fa_profile_launch_count(void) { return g_launches; }

fa_status fa_device_status(uint32_t* out) {
  if (out == nullptr) { set_error("out is NULL"); return FA_ERR_INVALID_ARG; }
  unsigned* p = device_status_ptr();
  if (p == nullptr) { set_error("no CUDA device"); return FA_ERR_CUDA; }
  unsigned v = 0;
  cudaError_t e = cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && v != 0) e = cudaMemset(p, 0, sizeof(v));
  *out = v;
  return cuda_status(e, "read device status");
}

}  // extern "C"
