// General backward kernel instances with the norm, and the finalize kernel of
// the weight and bias gradients.
#include "instances.cuh"

namespace qkvp {

// Outputs: [dw_q | dw_k] (2 * head_dim, when dw_q is set), then db (n_bias,
// when db is set). Output j = sum over partial rows b of its column, in a
// fixed order (deterministic): CTA x owns kFinalizeOutputsPerCta consecutive
// outputs (a warp reads 32 consecutive outputs of one row: 128 contiguous
// bytes per load); its threads split the rows into kFinalizeThreads /
// kFinalizeOutputsPerCta interleaved slices, each thread fetches its rows in
// batches of independent loads and adds row i of its slice into running sum
// i % 4, the four sums are combined in order, and a fixed-shape tree adds the
// slices. Float32 throughout: float64 adds are slow on this part, and a float32
// sum over at most 1024 rows is far inside the weight-gradient tolerance.
__global__ void __launch_bounds__(kFinalizeThreads) qkvp_dw_finalize_kernel(const FinalizeArgs a) {
  griddep_wait();
  constexpr int K = kFinalizeOutputsPerCta, SLICES = kFinalizeThreads / K, kBatch = 20;
  __shared__ float s_sum[SLICES][K];
  const int jj = threadIdx.x % K, slice = threadIdx.x / K;
  const int j = blockIdx.x * K + jj;
  const int n_dw = a.dw_q ? 2 * a.head_dim : 0;
  const int n_out = n_dw + (a.db ? a.n_bias : 0);
  const bool is_dw = j < n_dw;
  const float* col = is_dw ? a.partials + j : a.db_partials + (j - n_dw);
  const int64_t stride = is_dw ? 2 * a.head_dim : a.n_bias;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (j < n_out) {
    for (int i0 = 0; slice + SLICES * i0 < a.nparts; i0 += kBatch) {
      float v[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int b = slice + SLICES * (i0 + k);
        v[k] = b < a.nparts ? __ldcg(col + (int64_t)b * stride) : 0.f;
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) acc[k & 3] += v[k];  // kBatch is a multiple of 4: row i into sum i % 4
    }
  }
  s_sum[slice][jj] = ((acc[0] + acc[1]) + acc[2]) + acc[3];
  __syncthreads();
  for (int width = SLICES / 2; width > 0; width /= 2) {
    if (slice < width) s_sum[slice][jj] += s_sum[slice + width][jj];
    __syncthreads();
  }
  if (slice == 0 && j < n_out) {
    float* dst = is_dw ? (j < a.head_dim ? a.dw_q + j : a.dw_k + (j - a.head_dim)) : a.db + (j - n_dw);
    const float total = s_sum[0][jj];
    *dst = a.accumulate ? total + *dst : total;
  }
}

const void* bwd_kernel_norm(const BwdVariant& v) { return inst::BwdPick<true, false>::pick(v); }

const void* dw_finalize_kernel() { return reinterpret_cast<const void*>(&qkvp_dw_finalize_kernel); }

}  // namespace qkvp
