// Per-head Newton-Schulz of a fused QKV update on the tensor cores (sm_103a).
//
// "[muon] Per-head Newton-Schulz for fused QKV projections" (DeepSpeed), What
// this PR does: a fused weight's dim 0 is cut into head_dim-row blocks (the
// same blocks in the sectioned and the interleaved packing, so the packing
// never enters), each block is orthogonalised on its own and multiplied by
// max(1, head_dim / in_features) ** 0.5. The iteration is Muon's published
// quintic Newton-Schulz: X = G / (||G||_F + eps), then five times
//     A = X X^T,   B = b A + c A A,   X = a X + B X,
// with (a, b, c) = (3.4445, -4.7750, 2.0315). (The published code transposes a
// tall block first only to work on the smaller Gram matrix; a X + B X with
// A = X X^T is the same polynomial in X either way.)
//
// Work split. A unit is 128 consecutive weight rows, two 64-row heads or one
// 128-row head (the tensor cores' M = 128). One cluster of nc CTAs takes one
// unit; CTA r keeps columns [r cs, (r + 1) cs) of it resident in shared memory
// for the whole iteration (bf16, 128-byte-swizzled boxes of 64 columns, loaded
// once by TMA). Each step:
//   1. Gram partial P_r = X_r X_r^T: tcgen05, K = cs, into TMEM columns 0-127.
//   2. A = sum over the cluster of P_r: every thread pushes its row's 64
//      columns of the partial (straight from TMEM via registers) to the CTA
//      that owns the row (CTA r owns rows [128 r / nc, 128 (r + 1) / nc)),
//      with st.async into that CTA's receive buffer, counted in bytes on its
//      mbarrier; the owner sums the nc partials of its rows in rank order,
//      rounds them to bf16 and pushes them the same way into the A tile of
//      every CTA of the cluster. No remote loads, no fences, no barrier
//      round trips: each CTA arms its two barriers with the bytes it expects.
//   3. A A: tcgen05, K = 128, into TMEM columns 128-255 (TMEM: 256 columns
//      when cs <= 256, else 512; the three products reuse the same columns
//      one after the other).
//   4. B = b A + c A A, rounded to bf16, in place of A.
//   5. B X_r with X_r as the MN-major B operand: tcgen05, N = cs, into TMEM
//      columns 0 .. cs-1.
//   6. X_r = a X_r + B X_r, rounded to bf16, in place; after the last step
//      times the scale, then TMA-stored to the output. (a stays an fp32
//      factor: folded into B's diagonal it would be rounded to bf16 too,
//      0.2 % off, which is what X gets when B is small.)
// With 64-row heads only the two diagonal 64 x 64 blocks of A are reduced and
// written; the rest of the A tile stays 0, so B is block diagonal and the two
// heads of a unit never mix. Before the first step each block's squared norm
// is summed the same way (row sums, then over the cluster) and X is scaled in
// place to X / (norm + eps).
//
// B X is committed in two sections of the slice's columns, and the next
// step's Gram starts on section 0 while the epilogue still updates section 1.
//
// Roles: warp 0 issues the TMA load; warp 1 owns TMEM and one of its threads
// issues every MMA; warps 2-9 are the epilogue: warp w reads TMEM lanes
// 32 (w % 4) .. 32 (w % 4) + 31 (= weight rows of the unit) and one half of
// the columns. The grid is always launched as an explicit cluster (st.async
// needs one, even for one CTA); without one the kernel does nothing and sets
// an error bit. Every wait is bounded (2 s); after a timeout the device error
// word is set and every thread still passes every barrier, without waiting.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "pipeline.cuh"
#include "tcgen05.cuh"

namespace qkvp {
namespace {

constexpr int kNsThreads = 320, kNsEpiThreads = 256, kNsEpiBar = 1;
constexpr int kBox = kNsUnitRows * 128;  // bytes of one 128-row x 64-column bf16 box
// Receive buffer of a row owner: nc slots of ceil(128 / nc) rows x 64 fp32
// columns; nc ceil(128 / nc) is at most 140 (nc = 14) for nc <= 16.
constexpr int kRecvBytes = 140 * 64 * 4;
constexpr float kNsA = 3.4445f, kNsB = -4.7750f, kNsC = 2.0315f;
constexpr int kNsSteps = 5;

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a swizzled box.
__device__ __forceinline__ int swz(int row, int chunk) { return row * 128 + ((chunk ^ (row & 7)) << 4); }

// Bounded wait that gives up at once when another thread of the CTA already
// gave up (*fail): after one timeout the rest of the kernel runs through its
// barriers without waiting.
template <bool CLUSTER>
__device__ __forceinline__ bool ns_wait(uint64_t* bar, uint32_t parity, int* err, volatile int* fail) {
  auto test = [&]() { return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (test()) return true;
  const uint64_t t0 = global_ns();
  while (!test()) {
    if (*fail) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      *fail = 1;
      atomicOr(err, kErrWaitTimeout);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace

__global__ void __launch_bounds__(kNsThreads, 1)
    qkvp_newton_schulz_kernel(const __grid_constant__ CUtensorMap tmap_m, const __grid_constant__ CUtensorMap tmap_out,
                              const NsArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t bar_load, bar_gram, bar_aready, bar_sq, bar_bready, bar_fin;
  // Section s of the slice written (one arrive per epilogue warp; the Gram of
  // the next step starts on section 0 while section 1 is being written) and
  // B X of section s done
  __shared__ __align__(8) uint64_t bar_xsec[2], bar_bx[2];
  __shared__ __align__(8) uint64_t bar_efull, bar_afull;  // completed by arrivals from every CTA of the cluster
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail;
  __shared__ float s_red[8], s_inv[2];
  __shared__ __align__(16) float2 s_nrecv[kNsMaxCluster];  // the cluster's block-norm partials

  if (!is_explicit_cluster()) {  // the exchange needs a cluster launch (the host always makes one)
    if (threadIdx.x == 0) atomicOr(a.err, kErrNotCluster);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t nc = (uint32_t)a.nc, rank = cluster_ctarank();
  const int unit = blockIdx.x / a.nc;
  const int cs = a.cs, nbox = cs >> 6, hd = a.head_dim;
  const int npass = hd == 64 ? 1 : 2;  // exchange passes per Gram (64 columns each)
  // Sections: boxes [0, sb) and [sb, nbox) when the slice has 4 boxes or more
  // (the Gram accumulator, TMEM columns 0-127, then lies in section 0's part
  // of the last B X), else one section.
  const int nsec = nbox >= 4 ? 2 : 1, sb = nsec == 2 ? nbox >> 1 : nbox;
  // Phases: every waiter below waits each phase of a barrier in order and can
  // never be more than one phase behind it, so a parity names one phase.
  // bar_xsec[s] completes once for the normalised input (phase 0) and once per
  // step's update (phase it + 1); the Gram of step it waits phase it.
  unsigned char* xs = smem;                 // nbox boxes: this CTA's columns of the unit
  unsigned char* ab = smem + nbox * kBox;   // 2 boxes: A, then B in place (128 x 128)
  float* R = reinterpret_cast<float*>(ab + 2 * kBox);  // receive buffer: [nc][rmax][64] fp32
  const int rmax = (kNsUnitRows + a.nc - 1) / a.nc;
  const int r0 = (int)(kNsUnitRows * rank / nc), r1 = (int)(kNsUnitRows * (rank + 1) / nc);  // rows owned

  if (threadIdx.x == 0) {
    mbar_init(&bar_load, 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&bar_xsec[k], kNsEpiThreads / 32);
      mbar_init(&bar_bx[k], 1);
    }
    mbar_init(&bar_gram, 1);
    mbar_init(&bar_aready, 1);
    mbar_init(&bar_sq, 1);
    mbar_init(&bar_bready, 1);
    mbar_init(&bar_fin, 1);
    mbar_init(&bar_efull, 1);  // armed once per phase by this CTA, completed by bytes from the cluster
    mbar_init(&bar_afull, 1);
    s_fail = 0;
    mbar_init_fence();
  }
  // The A tile starts at 0: with 64-row heads its off-diagonal blocks stay 0.
  for (int i = threadIdx.x; i < 2 * kBox / 16; i += kNsThreads) reinterpret_cast<uint4*>(ab)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_cta();
  if (warp == 1) tmem_alloc(&s_tmem, (uint32_t)a.tmem_cols);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ loads
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar_load, (uint32_t)(nbox * kBox));
      for (int j = 0; j < nbox; ++j)
        tma_load_2d(xs + j * kBox, &tmap_m, (int)rank * cs + 64 * j, unit * kNsUnitRows, &bar_load);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMAs
    if (lane == 0) {
      const uint32_t id_sq = umma_idesc_bf16(128, 128);
      for (int it = 0; it < kNsSteps; ++it) {
        // P = X_r X_r^T, section by section as the epilogue finishes them
        bool ok = true;
        for (int sec = 0; sec < nsec && ok; ++sec) {
          ok = ns_wait<false>(&bar_xsec[sec], it & 1, a.err, &s_fail);
          tc_fence_after();
          for (int j = sec * sb; j < (sec == 0 ? sb : nbox); ++j) {
            const uint64_t d = umma_desc_sw128(xs + j * kBox);
#pragma unroll
            for (int k = 0; k < 4; ++k) umma_bf16(tmem, d + 2 * k, d + 2 * k, id_sq, (j | k) != 0);
          }
        }
        if (!ok) break;
        umma_commit(&bar_gram);
        // A is complete in this CTA (the epilogue has seen every exchange pass
        // of this step finish; waiting on the cluster barrier here could skip
        // a phase when a step has two passes)
        if (!ns_wait<false>(&bar_aready, it & 1, a.err, &s_fail)) break;
        tc_fence_after();
        fence_proxy_async_cta();  // A arrived by st.async (generic proxy); the MMA reads it
        for (int j = 0; j < 2; ++j) {  // A A (A is symmetric: both operands are its rows)
          const uint64_t d = umma_desc_sw128(ab + j * kBox);
#pragma unroll
          for (int k = 0; k < 4; ++k) umma_bf16(tmem + 128, d + 2 * k, d + 2 * k, id_sq, (j | k) != 0);
        }
        umma_commit(&bar_sq);
        if (!ns_wait<false>(&bar_bready, it & 1, a.err, &s_fail)) break;
        tc_fence_after();
        for (int sec = 0; sec < nsec; ++sec) {  // B X_r, one section (at most 256 columns) at a time
          const int n0 = 64 * sec * sb, n = 64 * (sec == 0 ? sb : nbox - sb);
          const uint32_t id = umma_idesc_bf16_bmn(128, n);
          const uint64_t bd = umma_desc_sw128_mn(xs + (n0 >> 6) * kBox, kBox);
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            const uint64_t ad = umma_desc_sw128(ab + (s >> 2) * kBox) + 2 * (s & 3);
            umma_bf16(tmem + n0, ad, bd + (uint64_t)(128 * s), id, s != 0);  // +2048 B: 16 rows of X
          }
          umma_commit(&bar_bx[sec]);
        }
      }
      umma_commit(&bar_fin);  // arrives once everything issued above has completed
      mbar_wait(&bar_fin, 0, a.err);
    }
  } else {
    // --------------------------------------------------------- epilogue
    const int et = threadIdx.x - 64, q = warp & 3, h = (warp - 2) >> 2, row = 32 * q + lane;
    const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
    const uint32_t efull = smem_addr(&bar_efull), afull = smem_addr(&bar_afull);
    uint32_t pass = 0;

    // ---- block norms: row sums of squares, then over the cluster
    ns_wait<false>(&bar_load, 0, a.err, &s_fail);
    const int half_ch = nbox * 4;  // 16-byte chunks per row in one column half
    float ss = 0.f;
    for (int ch = h * half_ch; ch < (h + 1) * half_ch; ++ch) {
      float f[8];
      unpack8(*reinterpret_cast<const uint4*>(xs + (ch >> 3) * kBox + swz(row, ch & 7)), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) s_red[warp - 2] = ss;
    named_sync(kNsEpiBar, kNsEpiThreads);
    if (warp == 2) {  // the cluster exchange of the block norms: lane r talks to CTA r
      float lo = 0.f, hi = 0.f;  // rows 0-63, rows 64-127 of this CTA's columns
      for (int i = 0; i < 8; ++i) {
        if (((i + 2) & 3) < 2)
          lo += s_red[i];
        else
          hi += s_red[i];
      }
      if (lane == 0) mbar_arrive_expect_tx(&bar_efull, 8u * nc);
      if ((uint32_t)lane < nc)
        st_async_u2(cluster_map(smem_addr(&s_nrecv[rank]), lane), __float_as_uint(lo), __float_as_uint(hi),
                    cluster_map(efull, lane));
      float tlo = 0.f, thi = 0.f;
      if (ns_wait<true>(&bar_efull, pass & 1, a.err, &s_fail) && (uint32_t)lane < nc) {
        tlo = s_nrecv[lane].x;
        thi = s_nrecv[lane].y;
      }
      tlo = warp_sum(tlo);  // the same order in every CTA of the cluster
      thi = warp_sum(thi);
      if (lane == 0) {
        if (hd == 64) {
          s_inv[0] = 1.f / (sqrtf(tlo) + a.eps);
          s_inv[1] = 1.f / (sqrtf(thi) + a.eps);
        } else {
          s_inv[0] = s_inv[1] = 1.f / (sqrtf(tlo + thi) + a.eps);
        }
      }
    }
    ++pass;  // bar_efull: phase 0 was the norms; bar_afull starts with the first Gram
    uint32_t apass = 0;
    named_sync(kNsEpiBar, kNsEpiThreads);
    {
      const float inv = s_inv[row >> 6];
      for (int j = 0; j < nbox; ++j) {  // box j: this warp's rows, 32 columns
        uint4* pch[4];
        uint4 xv[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          pch[kk] = reinterpret_cast<uint4*>(xs + j * kBox + swz(row, 4 * h + kk));
          xv[kk] = *pch[kk];
        }
        const float2 inv2 = f2(inv, inv);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          float2 x2[4];
          unpack_pairs(xv[kk], x2);
#pragma unroll
          for (int i = 0; i < 4; ++i) x2[i] = __fmul2_rn(x2[i], inv2);
          *pch[kk] = pack_pairs(x2);
        }
        if (j == sb - 1 || j == nbox - 1) {  // end of a section
          fence_proxy_async_cta();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_xsec[j == nbox - 1 ? nsec - 1 : 0]);
        }
      }
    }

    for (int it = 0; it < kNsSteps; ++it) {
      // ---- 1-2: Gram partial -> exchange -> A (bf16) in every CTA
      ns_wait<false>(&bar_gram, it & 1, a.err, &s_fail);
      tc_fence_after();
      for (int p = 0; p < npass; ++p) {
        if (et == 0) {  // the bytes this CTA receives in this pass
          mbar_arrive_expect_tx(&bar_efull, (uint32_t)(nc * (r1 - r0) * 256));
          mbar_arrive_expect_tx(&bar_afull, (uint32_t)(kNsUnitRows * 64 * 2));
        }
        {  // push this row's 32 columns of the partial to the row's owner
          uint32_t v[32];
          tmem_ld32_issue(trow + (uint32_t)((hd == 64 ? 64 * (q >> 1) : 64 * p) + 32 * h), v);
          const uint32_t o = (uint32_t)(((row + 1) * (int)nc - 1) / kNsUnitRows);  // owner of this row
          const int lo_row = (int)(kNsUnitRows * o / nc);
          const uint32_t dst = cluster_map(smem_addr(R + ((int)rank * rmax + row - lo_row) * 64 + 32 * h), o);
          const uint32_t bar = cluster_map(efull, o);
          tmem_wait_ld32(v);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            st_async_f4(dst + 16 * i,
                        make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                    __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])),
                        bar);
        }
        ns_wait<true>(&bar_efull, pass & 1, a.err, &s_fail);
        // this CTA's rows: the nc partials summed in rank order, then pushed as
        // bf16 into the A tile of every CTA of the cluster
        for (int idx = et; idx < (r1 - r0) * 16; idx += kNsEpiThreads) {
          const int li = idx >> 4, c4 = idx & 15, i = r0 + li;
          const float* src = R + li * 64 + 4 * c4;
          float4 s4 = *reinterpret_cast<const float4*>(src);
          for (uint32_t r = 1; r < nc; ++r) {
            const float4 t = *reinterpret_cast<const float4*>(src + (int)r * rmax * 64);
            s4.x += t.x;
            s4.y += t.y;
            s4.z += t.z;
            s4.w += t.w;
          }
          const int col = (hd == 64 ? 64 * (i >> 6) : 64 * p) + 4 * c4;
          const uint32_t d = smem_addr(ab + (col >> 6) * kBox + swz(i, (col & 63) >> 3) + (col & 7) * 2);
          const uint32_t lo = pack2(s4.x, s4.y), hi2 = pack2(s4.z, s4.w);
          for (uint32_t r = 0; r < nc; ++r) st_async_u2(cluster_map(d, r), lo, hi2, cluster_map(afull, r));
        }
        ns_wait<true>(&bar_afull, apass & 1, a.err, &s_fail);  // A complete in this CTA
        ++pass;
        ++apass;
      }
      if (et == 0) mbar_arrive(&bar_aready);

      // ---- 3-4: B = b A + c A A, in place of A
      ns_wait<false>(&bar_sq, it & 1, a.err, &s_fail);
      tc_fence_after();
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {  // 32 columns of A A, and of A, at a time
        uint32_t sq[32];
        tmem_ld32_issue(trow + (uint32_t)(128 + 64 * h + 32 * half), sq);
        uint4* pch[4];
        uint4 av[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          pch[k] = reinterpret_cast<uint4*>(ab + h * kBox + swz(row, 4 * half + k));
          av[k] = *pch[k];
        }
        tmem_wait_ld32(sq);
        const float2 b2 = f2(kNsB, kNsB), c2 = f2(kNsC, kNsC);
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // on pairs: c (A A) + b A
          float2 a2[4];
          unpack_pairs(av[k], a2);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            a2[i] = __ffma2_rn(c2, f2(__uint_as_float(sq[8 * k + 2 * i]), __uint_as_float(sq[8 * k + 2 * i + 1])),
                               __fmul2_rn(b2, a2[i]));
          *pch[k] = pack_pairs(a2);
        }
      }
      tc_fence_before();
      fence_proxy_async_cta();
      named_sync(kNsEpiBar, kNsEpiThreads);
      if (et == 0) mbar_arrive(&bar_bready);

      // ---- 5-6: X = a X + B X (after the last step: times the scale, then stored)
      const bool last = it == kNsSteps - 1;
      const float fa = last ? a.scale * kNsA : kNsA, fd = last ? a.scale : 1.f;
      const float2 fa2 = f2(fa, fa), fd2 = f2(fd, fd);
      // 32 columns from c: X = a X + B X. The TMEM load is issued first, the
      // four shared-memory loads of X go out while it is in flight, and only
      // then are the new values computed and stored.
      auto update = [&](int c) {
        uint32_t d[32];
        tmem_ld32_issue(trow + (uint32_t)c, d);
        uint4* pch[4];
        uint4 xv[4];
        unsigned char* xb = xs + (c >> 6) * kBox;
        const int k0 = (c & 63) >> 3;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          pch[kk] = reinterpret_cast<uint4*>(xb + swz(row, k0 + kk));
          xv[kk] = *pch[kk];
        }
        tmem_wait_ld32(d);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // on pairs: a x + d (a x + s d after the last step)
          float2 x2[4];
          unpack_pairs(xv[kk], x2);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float2 d2 = f2(__uint_as_float(d[8 * kk + 2 * i]), __uint_as_float(d[8 * kk + 2 * i + 1]));
            if (last) d2 = __fmul2_rn(fd2, d2);
            x2[i] = __ffma2_rn(fa2, x2[i], d2);
          }
          *pch[kk] = pack_pairs(x2);
        }
      };
      for (int sec = 0; sec < nsec; ++sec) {
        ns_wait<false>(&bar_bx[sec], it & 1, a.err, &s_fail);
        tc_fence_after();
        for (int j = sec * sb; j < (sec == 0 ? sb : nbox); ++j) {  // box j: this warp's rows, 32 columns
          update(64 * j + 32 * h);
        }
        tc_fence_before();
        fence_proxy_async_cta();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_xsec[sec]);
      }
      if (last && et == 0) {  // store each section of the result as soon as every warp has written it
        for (int sec = 0; sec < nsec; ++sec) {
          ns_wait<false>(&bar_xsec[sec], kNsSteps & 1, a.err, &s_fail);
          for (int j = sec * sb; j < (sec == 0 ? sb : nbox); ++j)
            tma_store_2d(&tmap_out, xs + j * kBox, (int)rank * cs + 64 * j, unit * kNsUnitRows);
        }
        bulk_commit();
        bulk_wait_all();
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while another may still touch its shared memory
  if (warp == 1) tmem_dealloc(tmem, (uint32_t)a.tmem_cols);
}

const void* ns_kernel() { return reinterpret_cast<const void*>(&qkvp_newton_schulz_kernel); }
int ns_smem_bytes(int cs) {
  const int need = (cs / 64) * kBox + 2 * kBox + kRecvBytes + 1024;
  // 228 KiB per SM, 1 KiB reserved per CTA: 118 KiB admits one CTA per SM,
  // 78 KiB at most two
  const int floor = ns_tmem_cols(cs) == 512 ? 118 * 1024 : 78 * 1024;
  return need > floor ? need : floor;
}
int ns_threads() { return kNsThreads; }

}  // namespace qkvp
