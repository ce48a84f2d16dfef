// The wqkv projection with the prologue in its epilogue: packed = x . W^T on
// the tensor cores (tcgen05, bf16 in, fp32 accumulator in tensor memory), and
// each finished accumulator tile is rounded to bf16 (the packed tensor of the
// unfused path) and then split, normed and roped straight into q, k and v, so
// the packed tensor never goes to HBM.
//
// Persistent CTA pairs (thread-block clusters of two, one CTA per SM), each
// pair computing 256-token x 256-column tiles with the 2-SM MMA (cta_group::2):
// CTA r of the pair holds tokens [128 r, 128 r + 128) of the tile's A operand
// (x) and packed columns [128 r, 128 r + 128) of its B operand (W) in its own
// shared memory, the leader (r = 0) issues the MMAs for both, and each CTA's
// tensor memory receives its own 128 token rows of the 256 x 256 accumulator.
// Each SM thus reads half of the B tile it would need alone, which halves the
// shared-memory operand traffic of a 128 x 256 single-SM MMA. 10 warps per CTA:
//   warp 0       TMA producer: per K step its x half [128 x 64] and W half
//                [128 x 64] into a ring of 128B-swizzled stages, counted on
//                the leader's "full" barrier; the leader's producer also
//                announces both CTAs' bytes, and after each wait for a free
//                stage passes the "stage free" event on to the peer;
//   warp 1       (leader) MMA issuer: four 256x256x16 MMAs per stage into one
//                of two accumulators (2 x 256 TMEM columns in each CTA), a
//                commit that frees the stage, and a commit after the tile's
//                last K step that hands the accumulator to the epilogues;
//                in both CTAs warp 1 allocates and frees the tensor memory
//                together with its peer;
//   warps 2-9    epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 of this
//                CTA for half of the tile's head blocks, so thread i owns
//                token row i and holds every value of a head itself: the
//                RMSNorm sum and the rotate-half pairs need no shuffles. The
//                values are rounded to bf16 as they leave tensor memory (kept
//                as bf16 pairs) and, for head_dim 64, the accumulator is
//                handed back before any arithmetic; results leave through a
//                per-warp 128B-swizzled buffer as TMA stores of 32-token x
//                64-value boxes. The leader's epilogue passes "accumulator
//                ready" on to the peer; both CTAs' epilogue warps report
//                "accumulator drained" to the leader's MMA issuer. While they
//                work on one accumulator the MMAs fill the other.
// Work items (256-token M tiles x 256-column N tiles) go M-fastest inside
// groups of 16 M tiles, so the 4096 x rows of a group stay in L2 while the W
// tiles stream past (W is read from DRAM once per group). Every wait is
// bounded (see pipeline.cuh). No multicast: every load and every signal names
// one CTA of this GPU's own cluster.
#include "gqa_kernels.cuh"
#include "tcgen05.cuh"

namespace qkvp {

namespace {

constexpr int kGemmKBoxes = 2;                               // 64-wide K boxes per stage
constexpr int kGemmStages = 3;
constexpr int kGemmBoxBytes = kGemmBM * kGemmBK * 2;        // one 128 x 64 bf16 box (128B-swizzled)
constexpr int kGemmHalfBytes = kGemmKBoxes * kGemmBoxBytes;  // one operand half of a stage
constexpr int kGemmStageBytes = 2 * kGemmHalfBytes;          // this CTA's x half + W half
constexpr int kGemmKStage = kGemmKBoxes * kGemmBK;          // K per stage
constexpr int kGemmGroupM = 16;
constexpr int kGemmEpiWarps = 8;            // two per TMEM lane quarter
constexpr int kGemmUnitBytes = 32 * 128;    // an epilogue warp's staging buffer: 32 rows x 64 bf16
constexpr int kGemmThreads = (2 + kGemmEpiWarps) * 32;

// Bounded wait with cluster-scope acquire (the phase may be completed by
// arrivals from the other CTA of the pair).
__device__ __forceinline__ bool mbar_wait_cl(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, kErrWaitTimeout);
      return false;
    }
  }
  return true;
}

// The epilogue's output path: a unit is 64 consecutive values of one head for
// the warp's 32 token rows. Lane i writes its row's 8 chunks of 16 bytes into
// the warp's 4 KiB buffer with the 128-byte swizzle (chunk c of row r at slot
// c ^ (r % 8): the 8 lanes of a shared-memory wavefront hit 8 different slots,
// no bank conflicts), and one lane stores the [32 x 64] box with TMA. Full
// 128-byte lines leave the SM, instead of 32 scattered 16-byte pieces per
// store instruction (measured: those cost the projection ~130 us at T = 16384,
// taking the shared-memory / L1 data path from the MMA operands).
struct UnitStore {
  uint4* buf;   // this warp's buffer, 1024-byte aligned
  int lane;
  int row0;     // the warp's first token (the box's row coordinate)

  // Before writing the buffer: the previous store has read it.
  __device__ __forceinline__ void acquire() const {
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
  }
  __device__ __forceinline__ void put(int c, const uint4& v) const { buf[lane * 8 + (c ^ (lane & 7))] = v; }
  __device__ __forceinline__ void put8(int c, const float (&f)[8]) const { put(c, pack8(f)); }
  __device__ __forceinline__ void issue(const CUtensorMap* map, int col) const {
    fence_proxy_async_cta();  // the chunks written above, before the copy engine reads them
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(map, buf, col, row0);
      bulk_commit();
    }
  }
};

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// One head block of the tile for this thread's token row, from its rounded
// packed values (gemm_load_head): the norm sum, the scaling and the rotation
// run on registers; the results go out through the warp's staging buffer
// (UnitStore). Rows past T are clipped by the tensor maps.
// The head's fp32 accumulator columns for this thread's token row, rounded to
// bf16 pairs: element 2i in the low half of xb[i], 2i + 1 in the high half.
template <int HD>
__device__ __forceinline__ void gemm_load_head(uint32_t col0, uint32_t (&xb)[HD / 2]) {
#pragma unroll
  for (int c = 0; c < HD; c += 32) {
    float v[32];
    tmem_ld32(col0 + c, v);  // every lane: warp-wide loads
#pragma unroll
    for (int i = 0; i < 16; ++i) xb[c / 2 + i] = pack2(v[2 * i], v[2 * i + 1]);
  }
}

template <int HD, bool SECTIONED, bool ROPE, bool SAVE>
__device__ __forceinline__ void gemm_epilogue_head(const GemmArgs& a, const GemmOutMaps& m, const float* s_w,
                                                   const uint32_t (&xb)[HD / 2], int32_t p, int hb,
                                                   const UnitStore& st) {
  constexpr int HALF = HD / 2, UNITS = HD / 64;
  int role;
  uint32_t oh;
  classify<SECTIONED>((uint32_t)hb, a.n_q, a.n_kv, a.group, a.gs_magic, role, oh);
  auto xv = [&](int e) { return (e & 1) ? bf_hi(xb[e >> 1]) : bf_lo(xb[e >> 1]); };
  const int col = (int)oh * HD;  // the head's first column in its output's 2-D view
  if (role == kRoleV || SAVE) {  // the packed values themselves: v, or the pre-norm save
    const CUtensorMap* map = role == kRoleV ? &m.v : (role == kRoleQ ? &m.q_pre : &m.k_pre);
#pragma unroll
    for (int u = 0; u < UNITS; ++u) {
      st.acquire();
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int w0 = 32 * u + 4 * c;
        st.put(c, make_uint4(xb[w0], xb[w0 + 1], xb[w0 + 2], xb[w0 + 3]));
      }
      st.issue(map, col + 64 * u);
    }
    if (role == kRoleV) return;
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < HD; ++i) ss = fmaf(xv(i), xv(i), ss);
  const float r = rsqrtf(fmaf(ss, a.inv_head_dim, a.eps));
  const float* w = s_w + (role == kRoleK ? HD : 0);
  const CUtensorMap* map = role == kRoleQ ? &m.q : &m.k;
  // unit u holds elements [64 u, 64 u + 64): for head_dim 64 the rotate-half
  // pairs (i, i + 32) are both in unit 0; for head_dim 128 unit 0 is the low
  // half and unit 1 the high half of every pair, the high half waiting in
  // registers (bf16 pairs) while unit 0 is stored
  uint32_t hib[UNITS == 2 ? 32 : 1];
  st.acquire();
#pragma unroll
  for (int i0 = 0; i0 < HALF; i0 += 8) {
    float lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = i0 + i;  // frequency index
      const float ylo = xv(e) * r * w[e];
      const float yhi = xv(HALF + e) * r * w[HALF + e];
      if (ROPE) {
        float c, s;
        rope_cos_sin(p, a.rope.turns[e], a.rope.scale, &c, &s);
        lo[i] = fmaf(ylo, c, yhi * -s);
        hi[i] = fmaf(yhi, c, ylo * s);
      } else {
        lo[i] = ylo;
        hi[i] = yhi;
      }
    }
    st.put8(i0 / 8, lo);
    if (UNITS == 1) {
      st.put8((HALF + i0) / 8, hi);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) hib[(UNITS == 2 ? i0 / 2 : 0) + i] = pack2(hi[2 * i], hi[2 * i + 1]);
    }
  }
  st.issue(map, col);
  if (UNITS == 2) {
    st.acquire();
#pragma unroll
    for (int c = 0; c < 8; ++c) st.put(c, make_uint4(hib[4 * c], hib[4 * c + 1], hib[4 * c + 2], hib[4 * c + 3]));
    st.issue(map, col + 64);
  }
}

}  // namespace

template <int HD, bool SECTIONED, bool ROPE, bool SAVE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    qkvp_gemm_fwd_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                         const __grid_constant__ GemmOutMaps maps, const GemmArgs a) {
  griddep_wait();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* ring = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[kGemmStages], empty[kGemmStages], tfull[2], tempty[2], tdone;
  __shared__ uint32_t s_tmem;
  __shared__ float s_w[2 * HD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(&full[s], 1);   // (leader) its producer's arrive; both CTAs' bytes
      mbar_init(&empty[s], 1);  // the leader's MMA commit, or its producer's relay (peer)
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);                   // the leader's MMA commit, or its epilogue's relay (peer)
      mbar_init(&tempty[b], 2 * kGemmEpiWarps);  // (leader) every epilogue warp of both CTAs
    }
    mbar_init(&tdone, 1);  // (leader) the last commit: every MMA it issued is complete
    mbar_init_fence();
  }
  for (int i = threadIdx.x; i < 2 * HD; i += blockDim.x) s_w[i] = i < HD ? a.w_q[i] : a.w_k[i - HD];
  if (warp == 1) tmem_alloc_pair(&s_tmem, 2 * kGemmBN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();  // both CTAs' barriers exist before any load or arrival names them
  const uint32_t tmem = s_tmem;
  const int64_t cluster = blockIdx.x >> 1, clusters = gridDim.x >> 1;
  const int kb_count = (a.hidden + kGemmKStage - 1) / kGemmKStage;
  const int64_t group = (int64_t)kGemmGroupM * a.n_tiles;
  const uint32_t peer = rank ^ 1u;

  // work item w -> (M tile of 256 tokens, N tile of 256 packed columns)
  auto tile_of = [&](int64_t w, int& mt, int& nt) {
    const int64_t g = w / group, r = w - g * group;
    const int64_t gm = min((int64_t)kGemmGroupM, (int64_t)a.m_tiles - g * kGemmGroupM);
    nt = (int)(r / gm);
    mt = (int)(g * kGemmGroupM + (r - (int64_t)nt * gm));
  };

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t full0 = cluster_map(smem_addr(&full[0]), 0);  // the leader's full barriers
      uint32_t it = 0;
      bool ok = true;
      for (int64_t w = cluster; w < a.n_work && ok; w += clusters) {
        int mt, nt;
        tile_of(w, mt, nt);
        for (int kb = 0; kb < kb_count; ++kb, ++it) {
          const int s = (int)(it % kGemmStages);
          if (it >= (uint32_t)kGemmStages) {
            const uint32_t par = ((it / kGemmStages) - 1) & 1;
            if (!(leader ? mbar_wait(&empty[s], par, a.err) : mbar_wait_cl(&empty[s], par, a.err))) {
              ok = false;
              break;
            }
            // the stage is free in the peer too: the MMAs that read both halves are done
            if (leader) mbar_arrive_cluster(cluster_map(smem_addr(&empty[s]), peer));
          }
          unsigned char* st = ring + (size_t)s * kGemmStageBytes;
          if (leader) mbar_arrive_expect_tx(&full[s], 2 * kGemmStageBytes);  // both CTAs' halves
          const uint32_t bar = full0 + (uint32_t)s * 8u;
#pragma unroll
          for (int x = 0; x < kGemmKBoxes; ++x) {
            const int k0 = kb * kGemmKStage + x * kGemmBK;
            tma_load_2d_pair(st + x * kGemmBoxBytes, &tmap_x, k0, mt * 2 * kGemmBM + (int)rank * kGemmBM, bar);
            tma_load_2d_pair(st + kGemmHalfBytes + x * kGemmBoxBytes, &tmap_w, k0,
                             nt * kGemmBN + (int)rank * (kGemmBN / 2), bar);
          }
        }
      }
      // Before the pair may exit, every copy into either CTA must have landed:
      // the leader waits (bounded) for the latest fill of each stage, whose
      // phase counts both CTAs' bytes (the peer never fills a stage the leader
      // has not). Phases that the MMAs already consumed return at once.
      if (leader) {
        const uint32_t last = it;
        for (uint32_t k = last > (uint32_t)kGemmStages ? last - kGemmStages : 0; k < last; ++k)
          mbar_wait(&full[k % kGemmStages], (k / kGemmStages) & 1, a.err);
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(2 * kGemmBM, kGemmBN);
      uint32_t it = 0, local = 0;
      bool ok = true;
      for (int64_t w = cluster; w < a.n_work && ok; w += clusters, ++local) {
        const uint32_t b = local & 1;
        if (local >= 2 && !mbar_wait_cl(&tempty[b], ((local >> 1) - 1) & 1, a.err)) break;
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
#pragma unroll
          for (int x = 0; x < kGemmKBoxes; ++x) {
            const uint64_t ad = umma_desc_sw128(st + x * kGemmBoxBytes);
            const uint64_t bd = umma_desc_sw128(st + kGemmHalfBytes + x * kGemmBoxBytes);
#pragma unroll
            for (int k = 0; k < kGemmBK / 16; ++k)
              umma_bf16_pair(d, ad + 2 * k, bd + 2 * k, idesc, (kb | x | k) != 0);
          }
          umma_commit_pair(&empty[s]);  // frees the stage once these MMAs have read both CTAs' halves
        }
        if (ok) umma_commit_pair(&tfull[b]);
      }
      umma_commit_pair(&tdone);  // nothing it issued may still run when the pair exits
      mbar_wait(&tdone, 0, a.err);
    }
  } else {
    // epilogue warps 2 .. 2 + kGemmEpiWarps - 1: TMEM lane quarter warp % 4,
    // and one half of the tile's head blocks
    constexpr int HEADS = kGemmBN / HD, PER = HEADS / 2;
    const int qtr = warp & 3, part = (warp - 2) >> 2;
    const uint32_t lane_base = (uint32_t)(qtr * 32) << 16;
    const uint32_t tempty0 = cluster_map(smem_addr(&tempty[0]), 0);
    UnitStore st;
    st.buf = reinterpret_cast<uint4*>(ring + (size_t)kGemmStages * kGemmStageBytes) + (warp - 2) * (kGemmUnitBytes / 16);
    st.lane = lane;
    uint32_t local = 0;
    for (int64_t w = cluster; w < a.n_work; w += clusters, ++local) {
      int mt, nt;
      tile_of(w, mt, nt);
      const uint32_t b = local & 1;
      const bool got = leader ? mbar_wait(&tfull[b], (local >> 1) & 1, a.err)
                              : mbar_wait_cl(&tfull[b], (local >> 1) & 1, a.err);
      if (!__all_sync(0xffffffffu, got)) break;
      // the peer's half of the accumulator is complete too (one MMA wrote both)
      if (leader && warp == 2 && lane == 0) mbar_arrive_cluster(cluster_map(smem_addr(&tfull[b]), peer));
      tc_fence_after();
      st.row0 = mt * 2 * kGemmBM + (int)rank * kGemmBM + qtr * 32;
      const int64_t t = (int64_t)st.row0 + lane;
      const int32_t p = (ROPE && t < a.T) ? a.pos[t] : 0;
      if constexpr (PER > 1) {
        // Take this warp's columns out of tensor memory first and hand the
        // accumulator back at once: the MMAs of the tile after next never
        // wait for the epilogue's arithmetic and stores.
        uint32_t xb[PER][HD / 2];
#pragma unroll
        for (int j = 0; j < PER; ++j)
          if (nt * HEADS + part * PER + j < a.n_blocks)  // the same for the whole warp
            gemm_load_head<HD>(tmem + b * kGemmBN + lane_base + (uint32_t)((part * PER + j) * HD), xb[j]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty0 + b * 8u);  // this warp is done with accumulator b
#pragma unroll
        for (int j = 0; j < PER; ++j) {
          const int hb = nt * HEADS + part * PER + j;
          if (hb < a.n_blocks) gemm_epilogue_head<HD, SECTIONED, ROPE, SAVE>(a, maps, s_w, xb[j], p, hb, st);
          __syncwarp();
        }
      } else {
        // one head of 128 per warp: its 64 packed registers stay live through
        // the arithmetic, so the accumulator is handed back after it (holding
        // the loads in registers across the hand-back spilled)
        const int hb = nt * HEADS + part;
        if (hb < a.n_blocks) {
          uint32_t xb[HD / 2];
          gemm_load_head<HD>(tmem + b * kGemmBN + lane_base + (uint32_t)(part * HD), xb);
          gemm_epilogue_head<HD, SECTIONED, ROPE, SAVE>(a, maps, s_w, xb, p, hb, st);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty0 + b * 8u);  // this warp is done with accumulator b
      }
    }
    if (lane == 0) bulk_wait_all();  // this warp's output stores are complete
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // every load, MMA, relay and arrival of the pair is done
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, 2 * kGemmBN);
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

int gemm_fwd_smem_bytes() { return kGemmStages * kGemmStageBytes + kGemmEpiWarps * kGemmUnitBytes + 1024; }
int gemm_fwd_threads() { return kGemmThreads; }

}  // namespace qkvp
