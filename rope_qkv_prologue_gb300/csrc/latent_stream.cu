// Pipelined MLA kv latent kernel: the same arithmetic as qkvp_latent_kernel
// (so both give identical bits), fed by the shared-memory pipeline of
// gqa_stream.cuh.
//
// A tile is kLatentTileTokens consecutive rows. The producer warp bulk-copies
// the tile's rows into a stage and writes the tile's positions and checked
// pool slots beside it. Each consumer warp takes groups of 4 consecutive rows:
//   * norm part, 4 / NCL rows at a time (32 values per lane, NCL = norm chunks
//     per lane): lane l holds norm chunks l, l + 32, ... of each row, and one
//     row-trading butterfly reduces the rows' sums of squares together;
//   * rope part, all four rows at once: lane l takes row l / 8, rope chunk pair
//     (e, e + 4) with e = (l / 2) % 4, and half h = l % 2 of it (values
//     8e + 4h .. 8e + 4h + 3 and their rotate-half partners), and computes the
//     4 angles it needs itself.
#include "gqa_stream.cuh"

namespace qkvp {

template <bool POOL, bool ROPE, int NCL, int NCW, int CPS>
__global__ void __maxnreg__(stream_max_regs(NCW, CPS)) qkvp_latent_stream_kernel(const LatentArgs a) {
  griddep_wait();
  constexpr int HD = 2;  // table layout: positions in the "cos" slots, pool slots after them
  constexpr int RB = 4 / NCL;  // norm rows per reduction: 32 values per lane in flight (register budget)
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
    stream_producer<HD / 2, false, POOL, ROPE>(smem, HD, tpt, stages, stage_bytes, a.sg.n_tiles,
                                                              a.T, a.pos, a.rope, a.page, a.offset, a.num_pages,
                                                              a.page_size, a.dev_status, a.err, true, load);
    return;
  }

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int kr = lane >> 3, e = (lane >> 1) & 3, hh = lane & 1;  // rope part: row of the group, pair, half
  float2 w[NCL][4];
#pragma unroll
  for (int m = 0; m < NCL; ++m) {
    const int chunk = lane + 32 * m;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[m][i] = chunk < a.norm_chunks ? f2(__ldg(a.w + chunk * 8 + 2 * i), __ldg(a.w + chunk * 8 + 2 * i + 1))
                                      : f2(0.f, 0.f);
  }
  uint64_t turns[4];  // this lane's four rope frequencies (fixed for the whole kernel)
#pragma unroll
  for (int i = 0; i < 4; ++i) turns[i] = ROPE ? a.rope.turns[8 * e + 4 * hh + i] : 0;
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

    for (int g0 = 4 * warp; g0 < tpt; g0 += 4 * NCW) {
      // norm part: the group's rows, RB at a time (one shared reduction for all of them)
#pragma unroll 1
      for (int k0 = 0; k0 < 4; k0 += RB) {
        float2 x[RB][NCL][4];
        float ss[RB], r[RB];
#pragma unroll
        for (int j = 0; j < RB; ++j) {
          const uint4* row = sx + (g0 + k0 + j) * a.row_chunks;
          ss[j] = 0.f;
#pragma unroll
          for (int m = 0; m < NCL; ++m) {
            const int chunk = lane + 32 * m;
            unpack_pairs(chunk < a.norm_chunks ? row[chunk] : make_uint4(0u, 0u, 0u, 0u), x[j][m]);
            ss[j] += chunk_partial_sq(x[j][m]);  // the per-lane partial of latent_sum_sq
          }
        }
        latent_rsqrt_rows<RB>(ss, a.inv_norm_dim, a.eps, r);
#pragma unroll
        for (int j = 0; j < RB; ++j) {
          const int tl = g0 + k0 + j;
          const int64_t t = t0 + tl;
          if (t >= a.T) break;  // warp-uniform; the rows after it are past the end too
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
            if (chunk < a.norm_chunks) st_keep(dst + chunk, latent_norm_chunk(x[j][m], r[j], w[m]));
          }
        }
      }
      // rope part: lane -> (row g0 + kr, chunk pair e, half hh)
      {
        const int tl = g0 + kr;
        const int64_t t = t0 + tl;
        const uint2* row = reinterpret_cast<const uint2*>(sx + tl * a.row_chunks + a.norm_chunks);
        const uint2 rlo = row[2 * e + hh], rhi = row[2 * (e + 4) + hh];
        uint2 olo = rlo, ohi = rhi;
        if (ROPE) {
          float c[4], sn[4];
          const int32_t p = spos[tl];
#pragma unroll
          for (int i = 0; i < 4; ++i) rope_cos_sin(p, turns[i], a.rope.scale, &c[i], &sn[i]);
          latent_rope_quad(rlo, rhi, c, sn, olo, ohi);
        }
        uint2* dst = nullptr;
        if (t < a.T) {
          if (POOL) {
            const int32_t slot = slots[tl];
            if (slot >= 0) dst = reinterpret_cast<uint2*>(a.pool + (int64_t)slot * a.row_chunks + a.norm_chunks);
          } else {
            dst = reinterpret_cast<uint2*>(a.out + t * a.row_chunks + a.norm_chunks);
          }
        }
        if (dst) {
          dst[2 * e + hh] = olo;
          dst[2 * (e + 4) + hh] = ohi;
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
