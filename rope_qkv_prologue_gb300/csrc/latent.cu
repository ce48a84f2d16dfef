// MLA kv latent rows (RMSNorm over the first norm_dim values, rotate-half RoPE
// over the last 64, no norm on the rope part) with a contiguous or a paged-pool
// destination, and the staged path's scatter kernel.
//
// One warp handles one token row at a time (kLatentTokensPerWarp rows per
// iteration, all loads issued before any arithmetic). Lane l holds norm chunks
// l, l + 32, ... (8 values each) and lanes 0..7 hold the 8 rope chunks; the
// rope partner of chunk c is chunk c ^ 4 (lane ^ 4). Lane l computes cos/sin of
// frequency l once per token; lanes 0..7 fetch the 8 they need by shuffle.
#include "common.cuh"
#include "qkv_prologue.h"

namespace qkvp {

template <bool POOL, bool ROPE, int NCL>
__global__ void __launch_bounds__(kLatentWarps * 32) qkvp_latent_kernel(const LatentArgs a) {
  griddep_wait();
  constexpr int TPW = kLatentTokensPerWarp;
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = (int64_t)blockIdx.x * kLatentWarps + (threadIdx.x >> 5);
  const int64_t n_warps = (int64_t)gridDim.x * kLatentWarps;
  const bool rope_lane = lane < 8;
  const bool lo = (lane & 7) < 4;
  const int f0 = (lane & 3) * 8;

  float2 w[NCL][4];
#pragma unroll
  for (int m = 0; m < NCL; ++m) {
    const int chunk = lane + 32 * m;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[m][i] = chunk < a.norm_chunks ? f2(__ldg(a.w + chunk * 8 + 2 * i), __ldg(a.w + chunk * 8 + 2 * i + 1))
                                      : f2(0.f, 0.f);
  }

  for (int64_t t0 = warp_id * TPW; t0 < a.T; t0 += n_warps * TPW) {
    uint4 xn[TPW][NCL], xr[TPW];
    int32_t p[TPW];
#pragma unroll
    for (int k = 0; k < TPW; ++k) {
      const int64_t t = t0 + k;
      const bool vt = t < a.T;
      const uint4* row = a.rows + t * a.row_stride16;
#pragma unroll
      for (int m = 0; m < NCL; ++m) {
        const int chunk = lane + 32 * m;
        xn[k][m] = (vt && chunk < a.norm_chunks) ? ld_stream(row + chunk) : make_uint4(0u, 0u, 0u, 0u);
      }
      xr[k] = (vt && rope_lane) ? ld_stream(row + a.norm_chunks + lane) : make_uint4(0u, 0u, 0u, 0u);
      p[k] = (ROPE && vt) ? a.pos[t] : 0;
    }

#pragma unroll
    for (int k = 0; k < TPW; ++k) {
      const int64_t t = t0 + k;
      if (t >= a.T) break;  // warp-uniform
      float2 x[NCL][4];
      const float ss = latent_sum_sq<NCL>(xn[k], x);
      const float r = rsqrtf(fmaf(ss, a.inv_norm_dim, a.eps));

      float xq[8], o8[8];
      unpack8(xr[k], xq);
      if (ROPE) {
        float cl, sl;
        rope_cos_sin(p[k], a.rope.turns[lane], a.rope.scale, &cl, &sl);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float c = __shfl_sync(0xffffffffu, cl, f0 + i);
          const float s = __shfl_sync(0xffffffffu, sl, f0 + i);
          const float xp = __shfl_xor_sync(0xffffffffu, xq[i], 4);
          o8[i] = fmaf(xq[i], c, xp * (lo ? -s : s));
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) o8[i] = xq[i];
      }

      uint4* dst;
      if (POOL) {
        const int32_t pg = a.page[t], of = a.offset[t];
        int bad = 0;
        if (pg < 0 || pg >= a.num_pages) bad |= QKVP_DEV_BAD_PAGE;
        if (of < 0 || of >= a.page_size) bad |= QKVP_DEV_BAD_OFFSET;
        if (bad) {
          if (lane == 0 && a.dev_status) atomicOr(a.dev_status, bad);
          continue;  // warp-uniform: page/offset are per token
        }
        dst = a.pool + ((int64_t)pg * a.page_size + of) * a.row_chunks;
      } else {
        dst = a.out + t * a.row_chunks;
      }
#pragma unroll
      for (int m = 0; m < NCL; ++m) {
        const int chunk = lane + 32 * m;
        if (chunk < a.norm_chunks) st_keep(dst + chunk, latent_norm_chunk(x[m], r, w[m]));
      }
      if (rope_lane) st_keep(dst + a.norm_chunks + lane, ROPE ? pack8(o8) : xr[k]);
    }
  }
}

// Staged write: copy contiguous rows [T, row_chunks] into pool slots.
__global__ void __launch_bounds__(256) qkvp_scatter_kernel(const ScatterArgs a) {
  griddep_wait();
  const int64_t total = a.T * a.row_chunks;
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < total; i += (int64_t)gridDim.x * 256) {
    const int64_t t = i / a.row_chunks;
    const int64_t c = i - t * a.row_chunks;
    const int32_t pg = a.page[t], of = a.offset[t];
    int bad = 0;
    if (pg < 0 || pg >= a.num_pages) bad |= QKVP_DEV_BAD_PAGE;
    if (of < 0 || of >= a.page_size) bad |= QKVP_DEV_BAD_OFFSET;
    if (bad) {
      if (c == 0 && a.dev_status) atomicOr(a.dev_status, bad);
      continue;
    }
    const int64_t dst = ((int64_t)pg * a.page_size + of) * a.row_chunks + c;
    a.pool_a[dst] = a.src_a[i];
    if (a.src_b) a.pool_b[dst] = a.src_b[i];
  }
}

namespace {
template <bool P, bool R, int N>
const void* latent_ptr() {
  return reinterpret_cast<const void*>(&qkvp_latent_kernel<P, R, N>);
}
template <int N>
const void* latent_pick(bool pool, bool rope) {
  if (pool) return rope ? latent_ptr<true, true, N>() : latent_ptr<true, false, N>();
  return rope ? latent_ptr<false, true, N>() : latent_ptr<false, false, N>();
}
}  // namespace

const void* latent_kernel(bool pool, bool rope, int ncl) {
  switch (ncl) {
    case 1: return latent_pick<1>(pool, rope);
    case 2: return latent_pick<2>(pool, rope);
    default: return latent_pick<4>(pool, rope);
  }
}

const void* scatter_kernel() { return reinterpret_cast<const void*>(&qkvp_scatter_kernel); }

}  // namespace qkvp
