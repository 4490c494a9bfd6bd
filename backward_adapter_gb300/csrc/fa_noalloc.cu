// Allocation-free backward: fa_train_bwd with its scratch in a fixed device array.
//
// Some callers cannot hand the library a workspace: their device memory is owned
// by another allocator (a framework pool that has reserved the GPU, or a plugin
// host that passes in only its own tensors), or they run in a loop where a
// cudaMalloc, with the device synchronisation it can imply, is not acceptable.
// For them this entry point keeps the backward's scratch (D = rowsum(dO * O),
// the fp32 dQ accumulator and the mask tile map) in one file-scope __device__
// array of kNoAllocScratchBytes, which every GPU that loads the library holds
// until the process exits. Nothing here allocates or frees.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "fa_internal.h"
#include "fa_train.h"

namespace fa {
namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

// Device address of g_bwd_scratch per device. In host code the symbol name is only a host-side
// stand-in, so its device address is looked up once per device, with that device current.
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace fa

extern "C" {

FA_API fa_status fa_train_bwd_noalloc(const fa_params* p, const void* q, const void* k, const void* v,
                                      const void* mask, const void* o, const float* lse, const void* dO, void* dq,
                                      void* dk, void* dv, void* stream) {
  // Shapes are checked by the size query (0 = invalid parameters, reported by fa_train_bwd below).
  const size_t need = fa_train_bwd_workspace_size(p);
  if (need > fa::kNoAllocScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "these shapes need %zu bytes of backward scratch; fa_train_bwd_noalloc has a fixed %zu bytes",
             need, fa::kNoAllocScratchBytes);
    fa::set_error_message(msg);
    return FA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  if (need > 0) {
    cudaError_t e = fa::scratch_address(&scratch);
    if (e != cudaSuccess) {
      char msg[200];
      snprintf(msg, sizeof(msg), "locating the static backward scratch: %s", cudaGetErrorString(e));
      fa::set_error_message(msg);
      return FA_ERR_CUDA;
    }
  }
  return fa_train_bwd(p, q, k, v, mask, o, lse, dO, dq, dk, dv, scratch, fa::kNoAllocScratchBytes, stream);
}

}  // extern "C"
