// qkv_prologue_bwd_noalloc: the backward for callers that cannot allocate.
//
// Some callers of this library may not allocate device memory at all and have
// no spare buffer to lend us: a plugin inside an engine whose device memory
// belongs entirely to the engine's own pool, or a latency-critical loop in
// which a cudaMalloc (it can synchronise the whole device) is not allowed.
// The regular backward needs a caller-provided workspace for its per-CTA
// weight-gradient partial sums. This entry point instead uses one fixed
// array in the library's own device memory, declared below, and otherwise
// runs the regular backward unchanged.
//
// Costs and limits:
//  * every GPU that loads this library holds the array (kScratchBytes) until
//    the process exits;
//  * all calls share the one array: two calls whose work overlaps on the GPU
//    (different streams, no ordering between them) race on it and give wrong
//    weight gradients; calls on one stream, or otherwise ordered, are fine;
//  * the array keeps whatever the last call left in it. Nothing has to start
//    at zero: the backward writes every partial row before it reads it;
//  * the array's device address is cached per device index for the life of
//    the process, so the call must not be used on a device after a
//    cudaDeviceReset in the same process (the module, and the array with it,
//    is then reloaded at another address).
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "qkv_prologue.h"

namespace {

// 520 KiB: up to 512 KiB of partial rows (head_dim 64 always fits: at most
// 1024 rows of 512 bytes) and, after them, the 4112 bytes of arrival and
// election words of the weight-gradient fold.
constexpr size_t kScratchBytes = 520 * 1024;
constexpr int kMaxDevices = 64;

// Weight-gradient partial sums of qkv_prologue_bwd_noalloc. In host code this
// name is only a host-side stand-in; kernels get the device address below.
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device, looked up once per
// device (with that device current) and cached; nullptr on failure.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (err != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" int qkv_prologue_bwd_noalloc(const qkvp_layout* layout, int64_t T, const void* dq, const void* dk,
                                        const void* dv, const void* q_pre, const void* k_pre, const int32_t* pos,
                                        const float* w_q, const float* w_k, float eps, double rope_base,
                                        uint32_t flags, void* dpacked, float* dw_q, float* dw_k, void* stream) {
  if (!layout) return QKVP_ERR_NULL;
  // Without the norm there are no weight-gradient partial sums: no scratch.
  const size_t need = (flags & QKVP_NORM_OFF) ? 0 : qkv_prologue_bwd_workspace_size(layout, T);
  if (need > kScratchBytes) return QKVP_ERR_WORKSPACE;  // too many partial rows for the fixed array
  if (T == 0 || need == 0) {
    // an empty batch needs no scratch; an invalid layout gets the regular checks' answer
    return qkv_prologue_bwd(layout, T, dq, dk, dv, q_pre, k_pre, pos, w_q, w_k, eps, rope_base, flags, dpacked,
                            dw_q, dw_k, nullptr, 0, stream);
  }
  void* scratch = scratch_on_current_device();
  if (!scratch) return QKVP_ERR_ARCH;
  return qkv_prologue_bwd(layout, T, dq, dk, dv, q_pre, k_pre, pos, w_q, w_k, eps, rope_base, flags, dpacked,
                          dw_q, dw_k, scratch, kScratchBytes, stream);
}
