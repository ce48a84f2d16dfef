// Pipelined backward kernel instances with the norm, and the library's device
// error word.
#include <mutex>

#include "instances.cuh"

namespace qkvp {

// Set (atomic OR) by a streaming kernel whose bounded wait gave up.
__device__ int g_qkvp_device_error = 0;

namespace {
constexpr int kMaxDev = 64;
std::mutex g_err_mutex;
int* g_err_ptr[kMaxDev] = {};
}  // namespace

const void* bwd_stream_kernel_norm(const BwdVariant& v) { return inst::BwdPick<true, true>::pick(v); }

int* device_error_word() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_err_mutex);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_qkvp_device_error) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  return g_err_ptr[dev];
}

int read_device_error(bool clear, int* value) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_qkvp_device_error, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (clear && v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_qkvp_device_error, &zero, sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      return -1;
    }
  }
  *value = v;
  return 0;
}

}  // namespace qkvp
