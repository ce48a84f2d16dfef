// Pipelined MLA kv latent kernel: the same arithmetic as qkvp_latent_kernel
// (so both give identical bits), fed by the shared-memory pipeline of
// gqa_stream.cuh.
//
// A tile is kLatentTileTokens consecutive rows. The producer warp bulk-copies
// the tile's rows into a stage and writes the tile's positions and checked
// pool slots beside it. Each consumer warp takes groups of 8 consecutive rows:
//   * norm part, row by row: lane l holds norm chunks l, l + 32, ... of the
//     row, the whole warp reduces its sum of squares;
//   * rope part, all 8 rows at once: lane l takes row l / 4 and its rope chunk
//     pair (e, e + 4), e = l % 4 (values 8e .. 8e+7 and their rotate-half
//     partners), and computes the 8 angles it needs itself.
#include "gqa_stream.cuh"

namespace qkvp {

template <bool POOL, bool ROPE, int NCL, int NCW, int CPS>
__global__ void __maxnreg__(stream_max_regs(NCW, CPS)) qkvp_latent_stream_kernel(const LatentArgs a) {
  griddep_wait();
  constexpr int HD = 2;  // table layout: positions in the "cos" slots, pool slots after them
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + StreamSmem::kBarriers);
  uint64_t* empty = full + kMaxStages;
  const int tpt = a.sg.tpt, stages = a.sg.stages, stage_bytes = a.sg.stage_bytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    mbar_init_fence();
  }
  __syncthreads();

  if (threadIdx.x >= NCW * 32) {
    const uint32_t row_bytes = (uint32_t)a.row_chunks * 16u;
    const bool dense = a.sg.dense != 0;
    auto load = [&](unsigned char* dst, int64_t t0, int ntok, uint64_t* bar, uint64_t pol) {
      mbar_expect_tx(bar, (uint32_t)ntok * row_bytes);
      if (dense) {
        bulk_load(dst, a.rows + t0 * a.row_stride16, (uint32_t)ntok * row_bytes, bar, pol);
      } else {
        for (int i = 0; i < ntok; ++i)
          bulk_load(dst + (size_t)i * row_bytes, a.rows + (t0 + i) * a.row_stride16, row_bytes, bar, pol);
      }
    };
    stream_producer<HD / 2, false, POOL, decltype(load), ROPE>(smem, HD, tpt, stages, stage_bytes, a.sg.n_tiles,
                                                              a.T, a.pos, a.rope, a.page, a.offset, a.num_pages,
                                                              a.page_size, a.dev_status, a.err, load);
    return;
  }

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int kr = lane >> 2, e = lane & 3;  // rope part: row of the group, chunk pair
  float2 w[NCL][4];
#pragma unroll
  for (int m = 0; m < NCL; ++m) {
    const int chunk = lane + 32 * m;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[m][i] = chunk < a.norm_chunks ? f2(__ldg(a.w + chunk * 8 + 2 * i), __ldg(a.w + chunk * 8 + 2 * i + 1))
                                      : f2(0.f, 0.f);
  }
  const unsigned char* data = smem + StreamSmem::data(HD, tpt, stages);

  int s = 0;
  uint32_t phase = 0;
  for (int64_t tile = blockIdx.x; tile < a.sg.n_tiles; tile += gridDim.x) {
    const bool got = mbar_wait(&full[s], phase, a.err);
    if (!__all_sync(0xffffffffu, got)) break;
    const int64_t t0 = tile * tpt;
    const uint4* sx = reinterpret_cast<const uint4*>(data + (size_t)s * stage_bytes);
    const int32_t* spos = reinterpret_cast<const int32_t*>(smem + StreamSmem::tables(HD) +
                                                           s * StreamSmem::table_stride(HD, tpt));
    const int32_t* slots = spos + 2 * tpt * (HD / 2);

    for (int g0 = 8 * warp; g0 < tpt; g0 += 8 * NCW) {
      // norm part, row by row (two rows interleaved)
#pragma unroll 2
      for (int k = 0; k < 8; ++k) {
        const int tl = g0 + k;
        const int64_t t = t0 + tl;
        const uint4* row = sx + tl * a.row_chunks;
        uint4 xr[NCL];
#pragma unroll
        for (int m = 0; m < NCL; ++m) {
          const int chunk = lane + 32 * m;
          xr[m] = chunk < a.norm_chunks ? row[chunk] : make_uint4(0u, 0u, 0u, 0u);
        }
        float2 x[NCL][4];
        const float r = rsqrtf(fmaf(latent_sum_sq<NCL>(xr, x), a.inv_norm_dim, a.eps));
        if (t >= a.T) continue;  // warp-uniform
        uint4* dst;
        if (POOL) {
          const int32_t slot = slots[tl];
          if (slot < 0) continue;  // bad page / offset: reported by the producer, store skipped
          dst = a.pool + (int64_t)slot * a.row_chunks;
        } else {
          dst = a.out + t * a.row_chunks;
        }
#pragma unroll
        for (int m = 0; m < NCL; ++m) {
          const int chunk = lane + 32 * m;
          if (chunk < a.norm_chunks) st_keep(dst + chunk, latent_norm_chunk(x[m], r, w[m]));
        }
      }
      // rope part: lane -> (row g0 + kr, chunk pair e)
      {
        const int tl = g0 + kr;
        const int64_t t = t0 + tl;
        const uint4* row = sx + tl * a.row_chunks;
        const uint4 rlo = row[a.norm_chunks + e], rhi = row[a.norm_chunks + e + 4];
        uint4 olo = rlo, ohi = rhi;
        if (ROPE) {
          float c[8], sn[8];
          const int32_t p = spos[tl];
#pragma unroll
          for (int i = 0; i < 8; ++i) rope_cos_sin(p, a.rope.turns[8 * e + i], &c[i], &sn[i]);
          latent_rope_pair(rlo, rhi, c, sn, olo, ohi);
        }
        uint4* dst = nullptr;
        if (t < a.T) {
          if (POOL) {
            const int32_t slot = slots[tl];
            if (slot >= 0) dst = a.pool + (int64_t)slot * a.row_chunks;
          } else {
            dst = a.out + t * a.row_chunks;
          }
        }
        if (dst) {
          st_keep(dst + a.norm_chunks + e, olo);
          st_keep(dst + a.norm_chunks + e + 4, ohi);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (++s == stages) {
      s = 0;
      phase ^= 1;
    }
  }
}

namespace {
template <bool P, bool R, int N>
const void* ptr() {
  return reinterpret_cast<const void*>(
      &qkvp_latent_stream_kernel<P, R, N, kLatentStreamWarps, kLatentStreamCtasPerSm>);
}
template <int N>
const void* pick(bool pool, bool rope) {
  if (pool) return rope ? ptr<true, true, N>() : ptr<true, false, N>();
  return rope ? ptr<false, true, N>() : ptr<false, false, N>();
}
}  // namespace

const void* latent_stream_kernel(bool pool, bool rope, int ncl) {
  switch (ncl) {
    case 1: return pick<1>(pool, rope);
    case 2: return pick<2>(pool, rope);
    default: return pick<4>(pool, rope);
  }
}

}  // namespace qkvp
