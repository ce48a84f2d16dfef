// General backward kernel instances with the norm, and the float64 finalize
// kernel of the weight and bias gradients.
#include "instances.cuh"

namespace qkvp {

// Outputs: [dw_q | dw_k] (2 * head_dim, when dw_q is set), then db (n_bias,
// when db is set). Output j = sum over partial rows b of its column, added in
// float64 in a fixed order (deterministic), then rounded to float32. CTA x
// owns kFinalizeOutputsPerCta consecutive outputs; its threads split the rows
// into kFinalizeThreads / kFinalizeOutputsPerCta interleaved slices and a
// fixed-shape tree adds the slices. (Many small CTAs: the float64 adds spread
// over every SM; 32 outputs per CTA measured slower on GB300.)
__global__ void __launch_bounds__(kFinalizeThreads) qkvp_dw_finalize_kernel(const FinalizeArgs a) {
  griddep_wait();
  constexpr int K = kFinalizeOutputsPerCta, SLICES = kFinalizeThreads / K;
  __shared__ double s_sum[SLICES][K];
  const int jj = threadIdx.x % K, slice = threadIdx.x / K;
  const int j = blockIdx.x * K + jj;
  const int n_dw = a.dw_q ? 2 * a.head_dim : 0;
  const int n_out = n_dw + (a.db ? a.n_bias : 0);
  const bool is_dw = j < n_dw;
  const float* col = is_dw ? a.partials + j : a.db_partials + (j - n_dw);
  const int64_t stride = is_dw ? 2 * a.head_dim : a.n_bias;
  double acc = 0.0;
  if (j < n_out) {
#pragma unroll 4
    for (int b = slice; b < a.nparts; b += SLICES) acc += (double)col[(int64_t)b * stride];
  }
  s_sum[slice][jj] = acc;
  __syncthreads();
  for (int width = SLICES / 2; width > 0; width /= 2) {
    if (slice < width) s_sum[slice][jj] += s_sum[slice + width][jj];
    __syncthreads();
  }
  if (slice == 0 && j < n_out) {
    float* dst = is_dw ? (j < a.head_dim ? a.dw_q + j : a.dw_k + (j - a.head_dim)) : a.db + (j - n_dw);
    const double total = s_sum[0][jj];
    *dst = a.accumulate ? (float)(total + (double)*dst) : (float)total;
  }
}

const void* bwd_kernel_norm(const BwdVariant& v) { return inst::BwdPick<true, false>::pick(v); }

const void* dw_finalize_kernel() { return reinterpret_cast<const void*>(&qkvp_dw_finalize_kernel); }

}  // namespace qkvp
