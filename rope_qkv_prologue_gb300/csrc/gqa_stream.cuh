// Streaming (shared-memory staged) forward and backward kernels of the
// packed-QKV prologue: the fast path for the common head layouts.
//
// Pipeline. A persistent CTA = NCW consumer warps + 1
// producer warp. The batch is cut into tiles of `tpt` consecutive tokens; CTA b
// takes tiles b, b + grid, ... The producer warp waits for a free stage of the
// shared-memory ring, issues bulk copies of the tile's source rows into it
// (one copy per source tensor when rows are dense), writes the tile's cos/sin
// table (and, for pool writes, the checked page slots) next to it, and arrives
// on the stage's "full" mbarrier, which also waits for the copied bytes.
// Consumers wait on "full", compute from shared memory, store results straight
// to HBM with 16-byte stores, and arrive on the stage's "empty" mbarrier.
//
// Work mapping. A token row of cpt 16-byte chunks is cut into cpt / 2 units:
// unit (h, e) = chunk e of head h together with its rotate-half partner chunk
// e + CPH/2, so the rotation needs no data from other lanes and a head is
// spread over CPH/2 lanes (its RMSNorm sum: two xor-shuffle rounds for
// head_dim 64). The consumer threads are split into tpt groups of tpg =
// consumers / tpt threads; group g owns token g of every tile, and thread i of
// a group owns units j = i + tpg * m (m < steps, j < cpt / 2), steps =
// ceil(cpt / 2 / tpg) (the last step may cover only part of the group; the
// host keeps that waste small). So across all tiles a thread always sees the
// same head positions: their role (q / k / v), output head and weight rows
// are worked out once, before the tile loop, and it needs the cos/sin of one
// token per tile (loaded once per tile, reused for every step).
// Element-wise float math uses Blackwell's paired fp32 instructions
// (__ffma2_rn / __fmul2_rn: two IEEE float operations per instruction, each
// rounded exactly like the scalar one).
#pragma once

#include "common.cuh"
#include "gqa_kernels.cuh"
#include "pipeline.cuh"
#include "qkv_prologue.h"

namespace qkvp {

// Norm weights in shared memory, laid out so that the CPH lanes of a head read
// them without bank conflicts: for role r (q, k), half h of a lane's 8 values
// and lane position e, the 4 floats w_r[8e + 4h .. 8e + 4h + 3] sit at
// r * HD + h * 4 * CPH + 4 * e. One 16-byte read per lane and half then covers
// 8 consecutive 16-byte words across the head's lanes.
template <int HD>
__device__ __forceinline__ void fill_split_weights(const float* w_q, const float* w_k, float* s_w) {
  constexpr int CPH = HD / 8;
  for (int i = threadIdx.x; i < 2 * HD; i += blockDim.x) {
    const int r = i / HD, rem = i % HD;
    const int h = rem / (4 * CPH), e = (rem % (4 * CPH)) / 4, k = rem % 4;
    s_w[i] = (r == 0 ? w_q : w_k)[8 * e + 4 * h + k];
  }
}

template <int HD>
__device__ __forceinline__ void load_split_weights(const float* s_w, int role, int e, float2 (&w)[4]) {
  constexpr int CPH = HD / 8;
  const float* p = s_w + (role == kRoleQ ? 0 : HD) + 4 * e;
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4 * CPH);
  w[0] = f2(a.x, a.y); w[1] = f2(a.z, a.w); w[2] = f2(b.x, b.y); w[3] = f2(b.z, b.w);
}

// Register cap of a streaming kernel: as many registers per thread as let
// CPS CTAs of NCW + 1 warps stay resident on an SM. The register file is
// split over the SM's 4 schedulers (16384 registers each) and a warp lives on
// one of them, so the cap is 16384 / (ceil(warps / 4) * 32), in steps of 8,
// at most 255. Without it the compiler can stop short of the budget and spill
// inside the tile loop.
constexpr int stream_max_regs_raw(int ncw, int cps) { return 16384 / (((cps * (ncw + 1) + 3) / 4) * 32) / 8 * 8; }
constexpr int stream_max_regs(int ncw, int cps) {
  return stream_max_regs_raw(ncw, cps) > 255 ? 255 : stream_max_regs_raw(ncw, cps);
}

// The producer warp of a streaming CTA: fills stages, writes tables, and (on a
// wait that timed out) drains the copies it issued before returning.
// `load(stage_ptr, t0, ntok, bar, policy)` (run by lane 0 only) announces the
// tile's byte count on `bar` and issues its bulk copies, with the L2 policy
// evict-first (`evict_first`) or normal. POS_AHEAD: the RoPE positions of the
// next tile (up to 32 tokens, token l in lane l) are loaded one tile ahead,
// so a tile's table never waits for a global load under the stream's traffic.
// The backward with the norm takes it (T = 16384: 155.1 -> 152.7 us on GB300),
// its consumers being slow enough that the producer's own latency showed. The
// forward and the norm-off backward do not: there the position load paces the
// reads, and without it they go out in bursts that interleave worse with the
// writes (forward 147 -> 162 us; Llama 3 backward 67.5 -> 70.1 us).
template <int HALF, bool ROPE, bool POOL, bool STAGE_POS = false, bool POS_AHEAD = false, class LoadTile>
__device__ __forceinline__ void stream_producer(unsigned char* smem, int hd, int tpt, int stages,
                                                int stage_bytes, int64_t n_tiles, int64_t T,
                                                const int32_t* pos, const RopeTable& rope,
                                                const int32_t* page, const int32_t* offset,
                                                int32_t num_pages, int32_t page_size,
                                                int32_t* dev_status, int* err, bool evict_first,
                                                LoadTile load) {
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + StreamSmem::kBarriers);
  uint64_t* empty = full + kMaxStages;
  unsigned char* data = smem + StreamSmem::data(hd, tpt, stages);
  const int lane = threadIdx.x & 31;
  const uint64_t policy = evict_first ? policy_evict_first() : policy_evict_normal();
  int s = 0;
  uint32_t phase = 0;
  int64_t issued = 0;
  bool ok = true;
  static_assert(!ROPE || HALF % 32 == 0, "a tile's table is whole warp-rows");
  auto tile_pos = [&](int64_t tile) -> int32_t {
    const int64_t t = tile * tpt + lane;
    return (lane < tpt && tile < n_tiles && t < T) ? pos[t] : 0;
  };
  const bool pos_ahead = POS_AHEAD && ROPE && tpt <= 32;
  int32_t pos_next = pos_ahead ? tile_pos(blockIdx.x) : 0;
  for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int32_t pos_cur = pos_next;
    if (pos_ahead) pos_next = tile_pos(tile + gridDim.x);
    if (issued >= stages) {
      const bool freed = mbar_wait(&empty[s], phase ^ 1, err);
      if (!__all_sync(0xffffffffu, freed)) {
        ok = false;
        break;
      }
    }
    const int64_t t0 = tile * tpt;
    const int ntok = (int)min((int64_t)tpt, T - t0);
    if (lane == 0) load(data + (size_t)s * stage_bytes, t0, ntok, &full[s], policy);
    float* tab = reinterpret_cast<float*>(smem + StreamSmem::tables(hd) + s * StreamSmem::table_stride(hd, tpt));
    if (ROPE) {
      // Unrolled: the position loads and sincospif chains of several entries
      // are in flight together (for head_dim 128 a tile's 64 frequencies per
      // token otherwise hold the ring back; measured on GB300). HALF is a
      // multiple of 32, so every lane runs every iteration (the shuffle of
      // POS_AHEAD is whole-warp).
#pragma unroll 4
      for (int i = lane; i < ntok * HALF; i += 32) {
        const int tl = i / HALF, f = i - (i / HALF) * HALF;
        const int32_t pt = pos_ahead ? __shfl_sync(0xffffffffu, pos_cur, tl) : pos[t0 + tl];
        float c, sn;
        rope_cos_sin(pt, rope.turns[f], rope.scale, &c, &sn);
        tab[i] = c;
        tab[tpt * HALF + i] = sn;
      }
    }
    if (STAGE_POS) {  // positions only (the consumers compute the angles)
      int32_t* sp = reinterpret_cast<int32_t*>(tab);
      for (int i = lane; i < ntok; i += 32) sp[i] = pos[t0 + i];
    }
    if (POOL) {
      int32_t* slot = reinterpret_cast<int32_t*>(tab + 2 * tpt * HALF);
      for (int i = lane; i < ntok; i += 32) {
        const int32_t pg = page[t0 + i], of = offset[t0 + i];
        int bad = 0;
        if (pg < 0 || pg >= num_pages) bad |= QKVP_DEV_BAD_PAGE;
        if (of < 0 || of >= page_size) bad |= QKVP_DEV_BAD_OFFSET;
        if (bad && dev_status) atomicOr(dev_status, bad);
        slot[i] = bad ? -1 : pg * page_size + of;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&full[s]);
    ++issued;
    if (++s == stages) {
      s = 0;
      phase ^= 1;
    }
  }
  griddep_launch_dependents();  // every load of this CTA is issued
  if (!ok && lane == 0) {
    // Let the copies already issued land before this CTA can exit.
    const int64_t first = issued > stages ? issued - stages : 0;
    for (int64_t k = first; k < issued; ++k) mbar_wait(&full[k % stages], (uint32_t)((k / stages) & 1), err);
  }
}

// ------------------------------------------------------------- forward ----

// The qkv bias in shared memory, laid out by unit: unit j (chunk pair lo =
// chunk e of packed head h, hi = chunk e + PPH; j = h * PPH + e) has four
// float4 pieces (lo values 0-3, lo 4-7, hi 0-3, hi 4-7), piece k at
// s_b[k * upt + j]. A warp's lanes hold consecutive units, so each 16-byte
// read covers consecutive words (no bank conflicts).
template <int HD>
__device__ __forceinline__ void fill_bias(const float* bias, int upt, float4* s_b) {
  constexpr int CPH = HD / 8, PPH = CPH / 2;
  for (int i = threadIdx.x; i < 4 * upt; i += blockDim.x) {
    const int k = i / upt, j = i - k * upt;
    const int chunk = (j / PPH) * CPH + (j % PPH) + (k >= 2 ? PPH : 0);
    s_b[i] = reinterpret_cast<const float4*>(bias)[2 * chunk + (k & 1)];
  }
}

// The bias pairs of unit j (lo and hi chunk).
__device__ __forceinline__ void load_bias_unit(const float4* s_b, int upt, int j, float2 (&lo)[4],
                                               float2 (&hi)[4]) {
  const float4 a = s_b[j], b = s_b[upt + j], c = s_b[2 * upt + j], d = s_b[3 * upt + j];
  lo[0] = f2(a.x, a.y); lo[1] = f2(a.z, a.w); lo[2] = f2(b.x, b.y); lo[3] = f2(b.z, b.w);
  hi[0] = f2(c.x, c.y); hi[1] = f2(c.z, c.w); hi[2] = f2(d.x, d.y); hi[3] = f2(d.z, d.w);
}

// NORM: RMSNorm of q and k (off: split -> RoPE only). BIAS: the qkv bias,
// staged in shared memory after the ring, is added to every input chunk first;
// v then stores the rounded biased value instead of a copy of the input.
template <int HD, bool SECTIONED, bool ROPE, bool SAVE, bool POOL, bool NORM, bool BIAS, int NCW, int CPS>
__global__ void __maxnreg__(stream_max_regs(NCW, CPS)) qkvp_fwd_stream_kernel(const FwdArgs a) {
  griddep_wait();
  using G = Geom<HD>;
  constexpr int CPH = G::CPH, HALF = G::HALF, NCT = NCW * 32, MAXM = kStreamMaxSteps;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + StreamSmem::kBarriers);
  uint64_t* empty = full + kMaxStages;
  float* s_w = reinterpret_cast<float*>(smem + StreamSmem::kWeights);
  const int tpt = a.sg.tpt, stages = a.sg.stages, steps = a.sg.steps, stage_bytes = a.sg.stage_bytes;
  float4* s_b = reinterpret_cast<float4*>(smem + StreamSmem::bias(HD, tpt, stages, stage_bytes));

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    mbar_init_fence();
  }
  if (NORM) fill_split_weights<HD>(a.w_q, a.w_k, s_w);
  if (BIAS) fill_bias<HD>(a.bias, a.cpt / 2, s_b);
  __syncthreads();

  if (threadIdx.x >= NCT) {
    const uint32_t row_bytes = (uint32_t)a.cpt * 16u;
    const bool dense = a.sg.dense != 0;
    stream_producer<HALF, ROPE, POOL>(
        smem, HD, tpt, stages, stage_bytes, a.sg.n_tiles, a.T, a.pos, a.rope, a.page, a.offset, a.num_pages,
        // L2 policy of the loads, measured at T = 16384: with the pre-norm save
        // normal aging is faster (149.2 -> 147.8 us), without it evict-first
        // (prefill 117.5 -> 106.4 us; Llama 3 and GPT-OSS steps 7-8 us)
        a.page_size, a.dev_status, a.err, !SAVE,
        [&](unsigned char* dst, int64_t t0, int ntok, uint64_t* bar, uint64_t pol) {
          mbar_expect_tx(bar, (uint32_t)ntok * row_bytes);
          if (dense) {
            bulk_load(dst, a.packed + t0 * a.row_stride16, (uint32_t)ntok * row_bytes, bar, pol);
          } else {
            for (int i = 0; i < ntok; ++i)
              bulk_load(dst + (size_t)i * row_bytes, a.packed + (t0 + i) * a.row_stride16, row_bytes, bar, pol);
          }
        });
    return;
  }

  // ---- consumers ----
  // Unit j of a token = chunk pair (lo = chunk e of head h, hi = chunk e + PPH)
  // with h = j / PPH, e = j % PPH; PPH = CPH / 2 lanes share a head.
  constexpr int PPH = CPH / 2, LOG_PPH = G::LOG_CPH - 1;
  const int ct = threadIdx.x, lane = ct & 31;
  const int upt = a.cpt / 2;            // units per token
  const int tpg = NCT / tpt;            // threads per token
  const int tl = ct / tpg;              // token of the tile this thread works on
  const int ig = ct - tl * tpg;         // index inside the group
  const int e = ig & (PPH - 1);         // the same for every step (tpg is a multiple of PPH)
  // Per step: output head, role and packed-head parity, fixed for the whole kernel.
  uint32_t info[MAXM];
#pragma unroll
  for (int m = 0; m < MAXM; ++m) {
    int role = kRoleV;
    uint32_t oh = 0, h = 0;
    if (m < steps && ig + tpg * m < upt) {
      h = (uint32_t)(ig + tpg * m) >> LOG_PPH;
      classify<SECTIONED>(h, a.n_q, a.n_kv, a.group, a.gs_magic, role, oh);
    }
    info[m] = oh | ((uint32_t)role << 16) | ((h & 1u) << 18);
  }
  const unsigned char* data = smem + StreamSmem::data(HD, tpt, stages);

  int s = 0;
  uint32_t phase = 0;
  for (int64_t tile = blockIdx.x; tile < a.sg.n_tiles; tile += gridDim.x) {
    const bool got = mbar_wait(&full[s], phase, a.err);
    if (!__all_sync(0xffffffffu, got)) break;
    const int64_t t0 = tile * tpt;
    const int64_t t = t0 + tl;
    const bool valid = t < a.T;
    const uint4* sx = reinterpret_cast<const uint4*>(data + (size_t)s * stage_bytes) + tl * a.cpt;
    const float* tab = reinterpret_cast<const float*>(smem + StreamSmem::tables(HD) + s * StreamSmem::table_stride(HD, tpt));
    float2 c2[4], s2[4];
    if (ROPE) {
      load_pairs(tab + tl * HALF + 8 * e, c2);
      load_pairs(tab + tpt * HALF + tl * HALF + 8 * e, s2);
    }
    int32_t slot = -1;
    if (POOL) slot = reinterpret_cast<const int32_t*>(tab + 2 * tpt * HALF)[tl];
    uint4* qrow = a.q + t * a.n_q * CPH;
    uint4* krow = POOL ? a.k_pool + (int64_t)slot * a.n_kv * CPH : a.k + t * a.n_kv * CPH;
    uint4* vrow = POOL ? a.v_pool + (int64_t)slot * a.n_kv * CPH : a.v + t * a.n_kv * CPH;
    uint4* qprow = SAVE ? a.q_pre + t * a.n_q * CPH : nullptr;
    uint4* kprow = SAVE ? a.k_pre + t * a.n_kv * CPH : nullptr;

#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
      if (m >= steps) break;
      const int j = ig + tpg * m;
      const bool in_row = j < upt;
      // stage chunks of the pair; odd heads read hi first so that the two heads a
      // quarter-warp covers fall in different shared-memory banks
      const int clo = in_row ? ((j >> LOG_PPH) * CPH + e) : 0;
      const bool odd = (info[m] >> 18) & 1u;
      const uint4 first = sx[odd ? clo + PPH : clo];
      const uint4 second = sx[odd ? clo : clo + PPH];
      const uint4 xlo = odd ? second : first, xhi = odd ? first : second;
      const int role = (int)((info[m] >> 16) & 3u);
      const int olo = (int)(info[m] & 0xffffu) * CPH + e;
      float2 lo[4], hi[4], wlo[4], whi[4], ylo[4], yhi[4];
      unpack_pairs(xlo, lo);
      unpack_pairs(xhi, hi);
      if (BIAS) {
        float2 blo[4], bhi[4];
        load_bias_unit(s_b, upt, in_row ? j : 0, blo, bhi);
        add_bias_pairs(lo, blo);
        add_bias_pairs(hi, bhi);
      }
      if (NORM) {
        load_split_weights<HD>(s_w, role, e, wlo);
        load_split_weights<HD>(s_w, role, e + PPH, whi);
      }
      pair_forward<CPH, ROPE, NORM>(lo, hi, wlo, whi, a.eps, a.inv_head_dim, c2, s2, ylo, yhi);
      if (!valid || !in_row) continue;
      // Plain contiguous forward: cache-streaming stores (measured faster on GB300
      // at every size tried); with the pre-norm save, or into a pool that
      // attention reads next, write-back stores.
      constexpr bool STREAM_OUT = !SAVE && !POOL;
      auto put = [](uint4* p, const uint4& v) {
        if (STREAM_OUT) st_stream(p, v);
        else st_keep(p, v);
      };
      if (role == kRoleQ) {
        put(qrow + olo, pack_pairs(ylo));
        put(qrow + olo + PPH, pack_pairs(yhi));
        if (SAVE) {
          st_stream(qprow + olo, xlo);
          st_stream(qprow + olo + PPH, xhi);
        }
      } else if (role == kRoleK) {
        if (!POOL || slot >= 0) {
          put(krow + olo, pack_pairs(ylo));
          put(krow + olo + PPH, pack_pairs(yhi));
        }
        if (SAVE) {
          st_stream(kprow + olo, xlo);
          st_stream(kprow + olo + PPH, xhi);
        }
      } else if (!POOL || slot >= 0) {
        put(vrow + olo, BIAS ? pack_pairs(lo) : xlo);
        put(vrow + olo + PPH, BIAS ? pack_pairs(hi) : xhi);
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

// ------------------------------------------------------------ backward ----

// STEPS > 0: exactly STEPS chunk pairs per consumer thread (the host picks the
// instance); with the norm and no bias the weight-gradient sums are then kept
// per step (a thread's step always has the same role) and routed to the q / k
// sums once at the end: half the multiply-adds of updating both every time,
// which the issue-bound consumers show (T = 16384 backward 161.5 -> 157.0 us).
// NORM off: g = R^T d is the whole gradient, and the saved inputs are neither
// staged nor read (three sections per stage instead of five). BIAS: the norm's
// input is x + b (bias staged in shared memory after the ring), and db = sum
// over tokens of the packed gradient. A thread owns the same chunk pairs of
// the same token slot in every tile and keeps their running sums in registers
// (the host keeps steps <= kBiasMaxSteps); at the end the token slots' sums
// are added in a fixed order into the CTA's row of db_partials.
template <int HD, bool SECTIONED, bool ROPE, bool NORM, bool BIAS, int NCW, int CPS, int STEPS>
__global__ void __maxnreg__(stream_max_regs(NCW, CPS)) qkvp_bwd_stream_kernel(const BwdArgs a) {
  griddep_wait();
  using G = Geom<HD>;
  constexpr int CPH = G::CPH, HALF = G::HALF, NCT = NCW * 32;
  constexpr int MAXM = BIAS ? kBiasMaxSteps : (STEPS ? STEPS : kStreamMaxSteps);
  constexpr bool PERSTEP = STEPS > 0 && NORM && !BIAS;  // weight-gradient sums per step, routed at the end
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float s_red[NORM ? NCW : 1][2][HD];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + StreamSmem::kBarriers);
  uint64_t* empty = full + kMaxStages;
  float* s_w = reinterpret_cast<float*>(smem + StreamSmem::kWeights);
  // (an instance for a fixed step count has it as a constant)
  const int tpt = a.sg.tpt, stages = a.sg.stages, steps = STEPS ? STEPS : a.sg.steps, stage_bytes = a.sg.stage_bytes;
  float4* s_b = reinterpret_cast<float4*>(smem + StreamSmem::bias(HD, tpt, stages, stage_bytes));
  // Stage sections (16-byte chunks): dq, dk, dv[, q_pre, k_pre], each [tpt][heads][CPH].
  const int qc = a.n_q * CPH, kc = a.n_kv * CPH;
  const int sec_dk = tpt * qc, sec_dv = sec_dk + tpt * kc, sec_qp = sec_dv + tpt * kc, sec_kp = sec_qp + tpt * qc;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    mbar_init_fence();
  }
  if (NORM) fill_split_weights<HD>(a.w_q, a.w_k, s_w);
  if (NORM && BIAS) fill_bias<HD>(a.bias, a.cpt / 2, s_b);
  __syncthreads();

  if (threadIdx.x >= NCT) {
    stream_producer<HALF, ROPE, false, false, NORM>(
        smem, HD, tpt, stages, stage_bytes, a.sg.n_tiles, a.T, a.pos, a.rope, nullptr, nullptr, 0, 0, nullptr, a.err,
        true, [&](unsigned char* dst, int64_t t0, int ntok, uint64_t* bar, uint64_t pol) {
          const uint32_t qb = (uint32_t)qc * 16u, kb = (uint32_t)kc * 16u;
          mbar_expect_tx(bar, (uint32_t)ntok * (NORM ? 2 * qb + 3 * kb : qb + 2 * kb));
          uint4* d = reinterpret_cast<uint4*>(dst);
          bulk_load(d, a.dq + t0 * qc, ntok * qb, bar, pol);
          bulk_load(d + sec_dk, a.dk + t0 * kc, ntok * kb, bar, pol);
          bulk_load(d + sec_dv, a.dv + t0 * kc, ntok * kb, bar, pol);
          if (NORM) {
            bulk_load(d + sec_qp, a.q_pre + t0 * qc, ntok * qb, bar, pol);
            bulk_load(d + sec_kp, a.k_pre + t0 * kc, ntok * kb, bar, pol);
          }
        });
    return;
  }

  // Unit j of a token = chunk pair (lo = chunk e of packed head h, hi = chunk
  // e + PPH), as in the forward.
  constexpr int PPH = CPH / 2, LOG_PPH = G::LOG_CPH - 1;
  const int ct = threadIdx.x, lane = ct & 31;
  const int upt = a.cpt / 2;
  const int tpg = NCT / tpt;
  const int tl = ct / tpg;
  const int ig = ct - tl * tpg;
  const int e = ig & (PPH - 1);
  // Per step: stage chunk of d_lo (low 16 bits) and of x_lo (high 16 bits);
  // 2 role bits and 1 parity bit (of the output head) per step.
  uint32_t offs[MAXM];
  uint32_t roles = 0, odds = 0;
#pragma unroll
  for (int m = 0; m < MAXM; ++m) {
    int role = kRoleV;
    uint32_t oh = 0;
    const bool in_row = m < steps && ig + tpg * m < upt;
    if (in_row)
      classify<SECTIONED>((uint32_t)(ig + tpg * m) >> LOG_PPH, a.n_q, a.n_kv, a.group, a.gs_magic, role, oh);
    uint32_t d_off, x_off;
    if (!in_row) {
      d_off = x_off = 0;  // any chunk of the stage; the step is skipped
    } else if (role == kRoleQ) {
      d_off = (tl * a.n_q + oh) * CPH + e;
      x_off = sec_qp + d_off;
    } else if (role == kRoleK) {
      d_off = sec_dk + (tl * a.n_kv + oh) * CPH + e;
      x_off = sec_kp + (tl * a.n_kv + oh) * CPH + e;
    } else {
      d_off = sec_dv + (tl * a.n_kv + oh) * CPH + e;
      x_off = d_off;  // unused
    }
    offs[m] = d_off | (x_off << 16);
    roles |= (uint32_t)role << (2 * m);
    odds |= (oh & 1u) << m;
  }
  const unsigned char* data = smem + StreamSmem::data(HD, tpt, stages);
  float2 aql[4], aqh[4], akl[4], akh[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) aql[i] = aqh[i] = akl[i] = akh[i] = f2(0.f, 0.f);
  float2 psl[PERSTEP ? MAXM : 1][4], psh[PERSTEP ? MAXM : 1][4];
#pragma unroll
  for (int m = 0; m < (PERSTEP ? MAXM : 1); ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i) psl[m][i] = psh[m][i] = f2(0.f, 0.f);
  float2 dbl[BIAS ? MAXM : 1][4], dbh[BIAS ? MAXM : 1][4];  // bias-gradient sums (BIAS)
#pragma unroll
  for (int m = 0; m < (BIAS ? MAXM : 1); ++m)
#pragma unroll
    for (int i = 0; i < 4; ++i) dbl[m][i] = dbh[m][i] = f2(0.f, 0.f);

  int s = 0;
  uint32_t phase = 0;
  for (int64_t tile = blockIdx.x; tile < a.sg.n_tiles; tile += gridDim.x) {
    const bool got = mbar_wait(&full[s], phase, a.err);
    if (!__all_sync(0xffffffffu, got)) break;
    const int64_t t = tile * tpt + tl;
    const bool valid = t < a.T;
    const uint4* sx = reinterpret_cast<const uint4*>(data + (size_t)s * stage_bytes);
    const float* tab = reinterpret_cast<const float*>(smem + StreamSmem::tables(HD) + s * StreamSmem::table_stride(HD, tpt));
    float2 c2[4], s2[4];
    if (ROPE) {
      load_pairs(tab + tl * HALF + 8 * e, c2);
      load_pairs(tab + tpt * HALF + tl * HALF + 8 * e, s2);
    }
    uint4* drow = a.dpacked + t * a.row_stride16;

#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
      if (m >= steps) break;
      const int j = ig + tpg * m;
      const int role = (int)((roles >> (2 * m)) & 3u);
      const bool odd = (odds >> m) & 1u;
      const int dl = (int)(offs[m] & 0xffffu), xl = (int)(offs[m] >> 16);
      // odd output heads read hi first (different shared-memory banks)
      const uint4 d1 = sx[odd ? dl + PPH : dl], d2 = sx[odd ? dl : dl + PPH];
      uint4 x1 = d1, x2 = d2;
      if (NORM) {
        x1 = sx[odd ? xl + PPH : xl];
        x2 = sx[odd ? xl : xl + PPH];
      }
      const uint4 dlo = odd ? d2 : d1, dhi = odd ? d1 : d2;
      float2 dl2[4], dh2[4], xl2[4], xh2[4], wlo[4], whi[4], dxlo[4], dxhi[4], gxlo[4], gxhi[4];
      float r;
      unpack_pairs(dlo, dl2);
      unpack_pairs(dhi, dh2);
      if (NORM) {
        unpack_pairs(odd ? x2 : x1, xl2);
        unpack_pairs(odd ? x1 : x2, xh2);
        if (BIAS) {
          float2 blo[4], bhi[4];
          load_bias_unit(s_b, upt, j < upt ? j : 0, blo, bhi);
          add_bias_pairs(xl2, blo);
          add_bias_pairs(xh2, bhi);
        }
        load_split_weights<HD>(s_w, role, e, wlo);
        load_split_weights<HD>(s_w, role, e + PPH, whi);
      }
      pair_backward<CPH, ROPE, NORM>(dl2, dh2, xl2, xh2, wlo, whi, a.eps, a.inv_head_dim, c2, s2, dxlo, dxhi,
                                     gxlo, gxhi, r);
      const bool live = valid && j < upt;
      const int plo = (j >> LOG_PPH) * CPH + e;  // packed-row chunk of lo
      if (PERSTEP) {
        // Selects and predicated stores instead of a branch per step: the
        // steps stay one block of straight-line code, so the arithmetic of
        // one step fills the latencies of the other (T = 16384 backward
        // 156.1 -> 155.2 us on GB300).
        const float2 r2 = f2(r, r);  // v units add g x r too; they are dropped when the sums are routed
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 nl = __ffma2_rn(gxlo[i], r2, psl[PERSTEP ? m : 0][i]);
          const float2 nh = __ffma2_rn(gxhi[i], r2, psh[PERSTEP ? m : 0][i]);
          psl[PERSTEP ? m : 0][i] = live ? nl : psl[PERSTEP ? m : 0][i];
          psh[PERSTEP ? m : 0][i] = live ? nh : psh[PERSTEP ? m : 0][i];
        }
        if (live) {
          st_keep(drow + plo, role == kRoleV ? dlo : pack_pairs(dxlo));
          st_keep(drow + plo + PPH, role == kRoleV ? dhi : pack_pairs(dxhi));
        }
        continue;
      }
      if (!live) continue;
      if (NORM) {
        const float rq = role == kRoleQ ? r : 0.f, rk = role == kRoleK ? r : 0.f;
        const float2 rq2 = f2(rq, rq), rk2 = f2(rk, rk);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          aql[i] = __ffma2_rn(gxlo[i], rq2, aql[i]);
          aqh[i] = __ffma2_rn(gxhi[i], rq2, aqh[i]);
          akl[i] = __ffma2_rn(gxlo[i], rk2, akl[i]);
          akh[i] = __ffma2_rn(gxhi[i], rk2, akh[i]);
        }
      }
      if (BIAS) {
        const int mb = BIAS ? m : 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          dbl[mb][i] = __fadd2_rn(dbl[mb][i], role == kRoleV ? dl2[i] : dxlo[i]);
          dbh[mb][i] = __fadd2_rn(dbh[mb][i], role == kRoleV ? dh2[i] : dxhi[i]);
        }
      }
      st_keep(drow + plo, role == kRoleV ? dlo : pack_pairs(dxlo));
      st_keep(drow + plo + PPH, role == kRoleV ? dhi : pack_pairs(dxhi));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (++s == stages) {
      s = 0;
      phase ^= 1;
    }
  }

  if (BIAS) {
    // Token group g of the tile (threads with tl == g) holds the sums of token
    // slot g of every tile; the groups are added in order 0, 1, ... through the
    // ring's shared memory, idle now (it holds at least two stages of dq, dk,
    // dv, i.e. at least the bias row's cpt * 8 floats), then written as the
    // CTA's row of db_partials.
    float* red = reinterpret_cast<float*>(smem + StreamSmem::data(HD, tpt, stages));
    asm volatile("bar.sync 1, %0;" ::"r"(NCT) : "memory");  // every consumer is done with the ring
    for (int g = 0; g < tpt; ++g) {
      if (tl == g) {
#pragma unroll
        for (int m = 0; m < MAXM; ++m) {
          const int j = ig + tpg * m;
          if (m >= steps || j >= upt) break;
          const int plo = (j >> LOG_PPH) * CPH + e;
          float2* lo = reinterpret_cast<float2*>(red + 8 * plo);
          float2* hi = reinterpret_cast<float2*>(red + 8 * (plo + PPH));
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            lo[i] = g == 0 ? dbl[m][i] : __fadd2_rn(lo[i], dbl[m][i]);
            hi[i] = g == 0 ? dbh[m][i] : __fadd2_rn(hi[i], dbh[m][i]);
          }
        }
      }
      asm volatile("bar.sync 1, %0;" ::"r"(NCT) : "memory");
    }
    float* row = a.db_partials + (int64_t)blockIdx.x * a.cpt * 8;
    for (int i = ct; i < a.cpt * 8; i += NCT) row[i] = red[i];
  }
  if (!NORM) return;

  if (PERSTEP) {  // route each step's sums to its role's accumulators
#pragma unroll
    for (int m = 0; m < (PERSTEP ? MAXM : 1); ++m) {
      const int role = (int)((roles >> (2 * m)) & 3u);
      const float2 fq = f2(role == kRoleQ ? 1.f : 0.f, role == kRoleQ ? 1.f : 0.f);
      const float2 fk = f2(role == kRoleK ? 1.f : 0.f, role == kRoleK ? 1.f : 0.f);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        aql[i] = __ffma2_rn(psl[m][i], fq, aql[i]);
        aqh[i] = __ffma2_rn(psh[m][i], fq, aqh[i]);
        akl[i] = __ffma2_rn(psl[m][i], fk, akl[i]);
        akh[i] = __ffma2_rn(psh[m][i], fk, akh[i]);
      }
    }
  }
  // Weight-grad partials: lanes of a warp with the same e (lane % PPH), then
  // the warps, in a fixed order (deterministic).
  float ql[8], qh[8], kl[8], kh[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    ql[2 * i] = aql[i].x; ql[2 * i + 1] = aql[i].y;
    qh[2 * i] = aqh[i].x; qh[2 * i + 1] = aqh[i].y;
    kl[2 * i] = akl[i].x; kl[2 * i + 1] = akl[i].y;
    kh[2 * i] = akh[i].x; kh[2 * i + 1] = akh[i].y;
  }
#pragma unroll
  for (int o = PPH; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      ql[i] += __shfl_xor_sync(0xffffffffu, ql[i], o);
      qh[i] += __shfl_xor_sync(0xffffffffu, qh[i], o);
      kl[i] += __shfl_xor_sync(0xffffffffu, kl[i], o);
      kh[i] += __shfl_xor_sync(0xffffffffu, kh[i], o);
    }
  }
  const int warp = ct >> 5;
  if (lane < PPH) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      s_red[warp][0][lane * 8 + i] = ql[i];
      s_red[warp][0][(lane + PPH) * 8 + i] = qh[i];
      s_red[warp][1][lane * 8 + i] = kl[i];
      s_red[warp][1][(lane + PPH) * 8 + i] = kh[i];
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(NCT) : "memory");  // consumer warps only
  for (int i = ct; i < 2 * HD; i += NCT) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) sum += s_red[w][i / HD][i % HD];
    a.partials[(int64_t)blockIdx.x * 2 * HD + i] = sum;
  }
  if (BIAS || a.flags == nullptr) return;  // the finalize kernel adds the rows

  // Fold: the CTA that finishes last (warp_publish_and_elect) adds every CTA's
  // partial row into dw_q and dw_k. Thread (o, sl) adds column o of rows
  // sl, sl + S, sl + 2S, ... (S slices of the rows), straight from L2 in
  // batches of 80 independent loads (one batch for a grid of up to 160 CTAs
  // at head_dim 64, two at 128: each batch is one L2 round trip in the
  // kernel's tail), into four running sums (row i of the slice
  // into sum i % 4), combined in order; then the slices in order. A fixed order
  // throughout, so the result does not depend on which CTA folds. (Float64
  // adds are slow on this part; float32 over at most 1024 rows is far inside
  // the weight-gradient tolerance.)
  __shared__ int s_last;
  __threadfence();  // this thread's partial-row stores, before the flag
  asm volatile("bar.sync 1, %0;" ::"r"(NCT) : "memory");
  if (ct < 32) {
    const bool won = warp_publish_and_elect(a.flags, a.flags + gridDim.x, blockIdx.x, gridDim.x, a.call_id);
    if (ct == 0) s_last = won ? 1 : 0;
  }
  asm volatile("bar.sync 1, %0;" ::"r"(NCT) : "memory");
  if (!s_last) return;
  fence_acq_rel_gpu();
  constexpr int OUT = 2 * HD, S = NCT / OUT > 0 ? NCT / OUT : 1, kBatch = 80;
  float* stage = reinterpret_cast<float*>(smem + StreamSmem::data(HD, tpt, stages));  // the idle ring
  const int nrows = gridDim.x;
  const int o = ct % OUT, sl = ct / OUT;
  if (sl < S) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const float* col = a.partials + o;
    for (int i0 = 0; sl + S * i0 < nrows; i0 += kBatch) {
      float v[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int row = sl + S * (i0 + k);
        v[k] = row < nrows ? __ldcg(col + (int64_t)row * OUT) : 0.f;
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) acc[k & 3] += v[k];  // kBatch is a multiple of 4: row i into sum i % 4
    }
    stage[sl * OUT + o] = ((acc[0] + acc[1]) + acc[2]) + acc[3];
  }
  asm volatile("bar.sync 1, %0;" ::"r"(NCT) : "memory");
  for (int i = ct; i < OUT; i += NCT) {
    float total = stage[i];
    for (int k = 1; k < S; ++k) total += stage[k * OUT + i];
    float* dst = i < HD ? a.dw_q + i : a.dw_k + (i - HD);
    *dst = a.accumulate ? *dst + total : total;
  }
}

}  // namespace qkvp
