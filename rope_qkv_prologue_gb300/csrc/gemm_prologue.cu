// The wqkv projection with the prologue in its epilogue: packed = x . W^T on
// the tensor cores (tcgen05, bf16 in, fp32 accumulator in tensor memory), and
// each finished accumulator tile is rounded to bf16 (the packed tensor of the
// unfused path) and then split, normed and roped straight into q, k and v, so
// the packed tensor never goes to HBM.
//
// Persistent CTAs, one per SM, in clusters of two that work on the same W
// tile for two neighbouring 128-token tiles at the same time (the second read
// of each W tile is an L2 hit); 10 warps per CTA:
//   warp 0       TMA producer: its own x tile [128 x 64] and the W tile
//                [256 x 64] per K step into a ring of 128B-swizzled
//                shared-memory stages; a stage is reused once this CTA's MMAs
//                have read it;
//   warp 1       MMA issuer: four 128x256x16 MMAs per stage into one of two
//                TMEM accumulators (2 x 256 columns), then a commit that frees
//                the stage; a commit after the tile's last K step hands the
//                accumulator to the epilogue;
//   warps 2-9    epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 for
//                half of the tile's head blocks, so thread i owns token row i
//                of the tile and holds every value of a head itself: the
//                RMSNorm sum and the rotate-half pairs need no shuffles. While
//                they work on one accumulator the MMAs fill the other.
// Work items (pairs of M tiles x one N tile) go M-fastest inside groups of 8
// pairs, so the x rows of a group stay in L2 while W tiles stream past. Every
// wait is bounded (see pipeline.cuh).
#include "gqa_kernels.cuh"
#include "tcgen05.cuh"

namespace qkvp {

namespace {

constexpr int kGemmStages = 4;
constexpr int kGemmStageBytes = kGemmBM * kGemmBK * 2 + kGemmBN * kGemmBK * 2;
constexpr int kGemmGroupPairs = 8;
constexpr int kGemmEpiWarps = 8;            // two per TMEM lane quarter
constexpr int kGemmThreads = (2 + kGemmEpiWarps) * 32;

__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// One head block of the tile for this thread's token row: the head's fp32
// accumulator columns are loaded once, rounded to bf16 (the packed value),
// and the norm sum, the scaling and the rotation run on registers.
template <int HD, bool SECTIONED, bool ROPE, bool SAVE>
__device__ __forceinline__ void gemm_epilogue_head(const GemmArgs& a, const float* s_w, uint32_t col0, int64_t t,
                                                   bool valid, int32_t p, int hb) {
  constexpr int HALF = HD / 2;
  int role;
  uint32_t oh;
  classify<SECTIONED>((uint32_t)hb, a.n_q, a.n_kv, a.group, a.gs_magic, role, oh);
  float x[HD];
#pragma unroll
  for (int c = 0; c < HD; c += 32) tmem_ld32(col0 + c, x + c);  // every lane: warp-wide loads
#pragma unroll
  for (int i = 0; i < HD; ++i) x[i] = round_bf16(x[i]);
  if (!valid) return;
  const int heads_out = role == kRoleQ ? a.n_q : a.n_kv;
  const int64_t base = (t * heads_out + oh) * HD;  // element offset of this row's output head
  uint4* out = role == kRoleQ ? a.q : (role == kRoleK ? a.k : a.v);
  uint4* pre = (SAVE && role == kRoleQ) ? a.q_pre : ((SAVE && role == kRoleK) ? a.k_pre : nullptr);
  if (role == kRoleV || pre) {
    uint4* dst = (role == kRoleV ? out : pre) + base / 8;
#pragma unroll
    for (int c = 0; c < HD; c += 8) {
      float f[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = x[c + i];
      dst[c / 8] = pack8(f);
    }
    if (role == kRoleV) return;
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < HD; ++i) ss = fmaf(x[i], x[i], ss);
  const float r = rsqrtf(fmaf(ss, a.inv_head_dim, a.eps));
  const float* w = s_w + (role == kRoleK ? HD : 0);
  uint4* dst = out + base / 8;
#pragma unroll
  for (int i0 = 0; i0 < HALF; i0 += 8) {
    float lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float ylo = x[i0 + i] * r * w[i0 + i];
      const float yhi = x[HALF + i0 + i] * r * w[HALF + i0 + i];
      if (ROPE) {
        float c, s;
        rope_cos_sin(p, a.rope.turns[i0 + i], a.rope.scale, &c, &s);
        lo[i] = fmaf(ylo, c, yhi * -s);
        hi[i] = fmaf(yhi, c, ylo * s);
      } else {
        lo[i] = ylo;
        hi[i] = yhi;
      }
    }
    dst[i0 / 8] = pack8(lo);
    dst[(HALF + i0) / 8] = pack8(hi);
  }
}

}  // namespace

template <int HD, bool SECTIONED, bool ROPE, bool SAVE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    qkvp_gemm_fwd_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                         const GemmArgs a) {
  griddep_wait();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* ring = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[kGemmStages], empty[kGemmStages], tfull[2], tempty[2];
  __shared__ uint32_t s_tmem;
  __shared__ float s_w[2 * HD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);  // this CTA's MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kGemmEpiWarps);  // one arrive per epilogue warp
    }
    mbar_init_fence();
  }
  for (int i = threadIdx.x; i < 2 * HD; i += blockDim.x) s_w[i] = i < HD ? a.w_q[i] : a.w_k[i - HD];
  if (warp == 1) tmem_alloc(&s_tmem, 2 * kGemmBN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();  // both CTAs of the pair start together
  const uint32_t tmem = s_tmem;
  const uint32_t rank = cluster_ctarank();
  const int64_t cluster = blockIdx.x >> 1, clusters = gridDim.x >> 1;
  const int kb_count = (a.hidden + kGemmBK - 1) / kGemmBK;
  const int64_t group = (int64_t)kGemmGroupPairs * a.n_tiles;

  // work item w -> (pair of M tiles, N tile); this CTA takes M tile 2 pair + rank
  auto tile_of = [&](int64_t w, int& mt, int& nt) {
    const int64_t g = w / group, r = w - g * group;
    const int64_t gm = min((int64_t)kGemmGroupPairs, (int64_t)a.m_pairs - g * kGemmGroupPairs);
    nt = (int)(r / gm);
    mt = (int)(2 * (g * kGemmGroupPairs + (r - (int64_t)nt * gm)) + rank);
  };

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int64_t w = cluster; w < a.n_work && ok; w += clusters) {
        int mt, nt;
        tile_of(w, mt, nt);
        for (int kb = 0; kb < kb_count; ++kb, ++it) {
          const int s = (int)(it % kGemmStages);
          if (it >= (uint32_t)kGemmStages && !mbar_wait(&empty[s], ((it / kGemmStages) - 1) & 1, a.err)) {
            ok = false;
            break;
          }
          unsigned char* st = ring + (size_t)s * kGemmStageBytes;
          mbar_arrive_expect_tx(&full[s], kGemmStageBytes);  // x tile + both W halves
          tma_load_2d(st, &tmap_x, kb * kGemmBK, mt * kGemmBM, &full[s]);
          for (int h = 0; h < 2; ++h)
            tma_load_2d(st + kGemmBM * kGemmBK * 2 + h * (kGemmBN / 2) * kGemmBK * 2, &tmap_w, kb * kGemmBK,
                        nt * kGemmBN + h * (kGemmBN / 2), &full[s]);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(kGemmBM, kGemmBN);
      uint32_t it = 0, local = 0;
      bool ok = true;
      for (int64_t w = cluster; w < a.n_work && ok; w += clusters, ++local) {
        const uint32_t b = local & 1;
        if (local >= 2 && !mbar_wait(&tempty[b], ((local >> 1) - 1) & 1, a.err)) break;
        tc_fence_after();
        const uint32_t d = tmem + b * kGemmBN;
        for (int kb = 0; kb < kb_count; ++kb, ++it) {
          const int s = (int)(it % kGemmStages);
          if (!mbar_wait(&full[s], (it / kGemmStages) & 1, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          unsigned char* st = ring + (size_t)s * kGemmStageBytes;
          const uint64_t ad = umma_desc_sw128(st), bd = umma_desc_sw128(st + kGemmBM * kGemmBK * 2);
#pragma unroll
          for (int k = 0; k < kGemmBK / 16; ++k) umma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0);
          umma_commit(&empty[s]);  // frees the stage once these MMAs have read it
        }
        if (ok) umma_commit(&tfull[b]);
      }
    }
  } else {
    // epilogue warps 2 .. 2 + kGemmEpiWarps - 1: TMEM lane quarter warp % 4,
    // and one half of the tile's head blocks
    constexpr int HEADS = kGemmBN / HD, PER = HEADS / 2;
    const int qtr = warp & 3, part = (warp - 2) >> 2;
    const uint32_t lane_base = (uint32_t)(qtr * 32) << 16;
    uint32_t local = 0;
    for (int64_t w = cluster; w < a.n_work; w += clusters, ++local) {
      int mt, nt;
      tile_of(w, mt, nt);
      const uint32_t b = local & 1;
      const bool got = mbar_wait(&tfull[b], (local >> 1) & 1, a.err);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const int64_t t = (int64_t)mt * kGemmBM + qtr * 32 + lane;
      const bool valid = t < a.T;
      const int32_t p = (ROPE && valid) ? a.pos[t] : 0;
#pragma unroll 1
      for (int j = part * PER; j < (part + 1) * PER; ++j) {
        const int hb = nt * HEADS + j;
        if (hb >= a.n_blocks) break;  // the same for the whole warp
        gemm_epilogue_head<HD, SECTIONED, ROPE, SAVE>(a, s_w, tmem + b * kGemmBN + lane_base + (uint32_t)(j * HD),
                                                      t, valid, p, hb);
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[b]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 2 * kGemmBN);
  cluster_sync_all();
}

namespace {
template <int HD, bool S, bool R, bool SV>
const void* gptr() {
  return reinterpret_cast<const void*>(&qkvp_gemm_fwd_kernel<HD, S, R, SV>);
}
template <int HD>
const void* gpick(bool sectioned, bool rope, bool save) {
  if (sectioned)
    return rope ? (save ? gptr<HD, true, true, true>() : gptr<HD, true, true, false>())
                : (save ? gptr<HD, true, false, true>() : gptr<HD, true, false, false>());
  return rope ? (save ? gptr<HD, false, true, true>() : gptr<HD, false, true, false>())
              : (save ? gptr<HD, false, false, true>() : gptr<HD, false, false, false>());
}
}  // namespace

const void* gemm_fwd_kernel(int head_dim, bool sectioned, bool rope, bool save) {
  return head_dim == 64 ? gpick<64>(sectioned, rope, save) : gpick<128>(sectioned, rope, save);
}

int gemm_fwd_smem_bytes() { return kGemmStages * kGemmStageBytes + 1024; }
int gemm_fwd_threads() { return kGemmThreads; }

}  // namespace qkvp
