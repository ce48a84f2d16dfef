// Backward kernel instances and the float64 weight-grad finalize kernel.
#include "gqa_kernels.cuh"

namespace qkvp {

// dw[j] = sum over partial rows b of partials[b][j], j over [dw_q | dw_k],
// added in float64 in a fixed order (deterministic), then rounded to float32.
// CTA x owns kFinalizeOutputsPerCta consecutive outputs; its threads split
// the rows into kFinalizeThreads / kFinalizeOutputsPerCta interleaved slices
// and a fixed-shape tree adds the slices.
__global__ void __launch_bounds__(kFinalizeThreads) qkvp_dw_finalize_kernel(const FinalizeArgs a) {
  griddep_wait();
  constexpr int K = kFinalizeOutputsPerCta, SLICES = kFinalizeThreads / K;
  __shared__ double s_sum[SLICES][K];
  const int jj = threadIdx.x % K, slice = threadIdx.x / K;
  const int j = blockIdx.x * K + jj;
  const int n_out = 2 * a.head_dim;
  double acc = 0.0;
  if (j < n_out) {
#pragma unroll 4
    for (int b = slice; b < a.nparts; b += SLICES) acc += (double)a.partials[(int64_t)b * n_out + j];
  }
  s_sum[slice][jj] = acc;
  __syncthreads();
  for (int width = SLICES / 2; width > 0; width /= 2) {
    if (slice < width) s_sum[slice][jj] += s_sum[slice + width][jj];
    __syncthreads();
  }
  if (slice == 0 && j < n_out) {
    float* dst = j < a.head_dim ? a.dw_q + j : a.dw_k + (j - a.head_dim);
    const double total = s_sum[0][jj];
    *dst = a.accumulate ? (float)(total + (double)*dst) : (float)total;
  }
}

namespace {
template <int HD, bool S, bool R>
const void* bwd_ptr() {
  return reinterpret_cast<const void*>(&qkvp_bwd_kernel<HD, S, R>);
}
template <int HD>
const void* bwd_pick(bool sectioned, bool rope) {
  if (sectioned) return rope ? bwd_ptr<HD, true, true>() : bwd_ptr<HD, true, false>();
  return rope ? bwd_ptr<HD, false, true>() : bwd_ptr<HD, false, false>();
}
}  // namespace

const void* bwd_kernel(int head_dim, bool sectioned, bool rope) {
  return head_dim == 64 ? bwd_pick<64>(sectioned, rope) : bwd_pick<128>(sectioned, rope);
}

const void* dw_finalize_kernel() { return reinterpret_cast<const void*>(&qkvp_dw_finalize_kernel); }

}  // namespace qkvp
