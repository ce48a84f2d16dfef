// Per-head Newton-Schulz of a fused QKV update on the tensor cores (sm_103a).
//
// "[muon] Per-head Newton-Schulz for fused QKV projections" (DeepSpeed), What
// this PR does: a fused weight's dim 0 is cut into head_dim-row blocks (the
// same blocks in the sectioned and the interleaved packing, so the packing
// never enters), each block is orthogonalised on its own and multiplied by
// max(1, head_dim / in_features) ** 0.5. The iteration is Muon's published
// quintic Newton-Schulz: X = G / (||G||_F + eps), then five times
//     A = X X^T,   B = b A + c A A,   X = a X + B X,
// with (a, b, c) = (3.4445, -4.7750, 2.0315).
//
// Evaluation through the Gram matrix. With P_k = a I + b A_k + c A_k^2 a step
// is X_{k+1} = P_k X_k, hence A_{k+1} = X_{k+1} X_{k+1}^T = P_k A_k P_k: every
// matrix of the iteration is a polynomial in A_0 = X_0 X_0^T (symmetric, and
// all of them commute), and
//     X_5 = M X_0,   M = P_4 P_3 P_2 P_1 P_0.
// So the weight is read twice instead of once per step, and the five steps run
// on head_dim x head_dim matrices:
//   1. qkvp_ns_gram_kernel: partial Gram matrices G_u G_u^T over column ranges
//      of each 128-row unit (two 64-row heads or one 128-row head), streamed
//      through shared memory by TMA, fp32 accumulation in tensor memory;
//   2. qkvp_ns_poly_kernel: per unit, the partials summed in a fixed order, the
//      block norms (trace of each head's diagonal block), then the fourteen
//      dependent 128 x 128 products of the steps on the tensor cores, and
//      M * (1 / (||G|| + eps)) * factor written out;
//   3. qkvp_ns_apply_kernel: out = M G, unit by unit and box by box of 64
//      columns, streamed through shared memory, stored by TMA.
// With 64-row heads every matrix of a unit is block diagonal (the two heads
// never mix): the products only compute the two 64 x 64 diagonal blocks and the
// rest of every matrix stays exactly 0.
//
// Precision. M has the eigenvalue a^5 (about 488) on every direction in which
// the block is (nearly) rank deficient, so the small eigenvalues that carry the
// result are differences of numbers that large: held in bf16 (or tf32) the
// steps lose them. Every matrix operand of the steps is therefore held as the
// sum of two bf16 numbers (hi = bf16(v), lo = bf16(v - hi): about 16
// significant bits) and a product is three bf16 MMAs (hi hi + hi lo + lo hi)
// with fp32 accumulation; M is applied the same way (hi G + lo G). The result is
// much closer to the exact iteration than the published bf16 iteration is.
//
// Every wait is bounded (2 s); after a timeout the device error word is set and
// every thread still passes every barrier, without waiting.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "pipeline.cuh"
#include "tcgen05.cuh"

namespace qkvp {
namespace {

constexpr int kBox = kNsUnitRows * 128;  // bytes of one 128-row x 64-column bf16 box
constexpr int kPlane = 2 * kBox;         // one bf16 plane of a 128 x 128 matrix: two boxes
constexpr float kNsA = 3.4445f, kNsB = -4.7750f, kNsC = 2.0315f;
constexpr int kNsSteps = 5;

constexpr int kGramThreads = 192, kGramStages = 4;
constexpr int kPolyThreads = 320, kPolyEpiWarps = 8;
constexpr int kApplyThreads = 320, kApplyStages = 9, kApplyAcc = 8;

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a swizzled box.
__device__ __forceinline__ int swz(int row, int chunk) { return row * 128 + ((chunk ^ (row & 7)) << 4); }

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return reinterpret_cast<unsigned char*>(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

// Bounded wait that gives up at once when another thread of the CTA already
// gave up (*fail): after one timeout the rest of the kernel runs through its
// barriers without waiting.
__device__ __forceinline__ bool ns_wait(uint64_t* bar, uint32_t parity, int* err, volatile int* fail) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*fail) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      *fail = 1;
      atomicOr(err, kErrWaitTimeout);
      return false;
    }
  }
  return true;
}

// ns_wait by lane 0 of the calling warp, its result shared with the whole warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* err, volatile int* fail) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = ns_wait(bar, parity, err, fail) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ void bulk_wait_read_but1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

// The 32 fp32 columns of this warp's TMEM lanes starting at `addr`.
__device__ __forceinline__ void tmem_ld32f(uint32_t addr, float (&v)[32]) {
  uint32_t r[32];
  tmem_ld32_issue(addr, r);
  tmem_wait_ld32(r);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Eight consecutive values of row r, from matrix column c (a multiple of 8),
// into the hi and lo bf16 planes of a 128 x 128 matrix: hi = bf16(v),
// lo = bf16(v - hi), both rounded to nearest even.
__device__ __forceinline__ void put8_split(unsigned char* hi, unsigned char* lo, int r, int c, const float* v) {
  const int off = (c >> 6) * kBox + swz(r, (c & 63) >> 3);
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 hb = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    const float2 hf = __bfloat1622float2(hb);
    h[i] = *reinterpret_cast<const uint32_t*>(&hb);
    l[i] = pack2(v[2 * i] - hf.x, v[2 * i + 1] - hf.y);
  }
  *reinterpret_cast<uint4*>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

// D (+)= X Y^T on the tensor cores (issued by the calling thread), X and Y
// held as bf16 hi/lo planes (three MMAs per K step of 16: hi hi, hi lo, lo hi),
// fp32 in TMEM columns d ..
// d + 127; K steps [k0, k1) of the HD / 16 (the first step of 0 overwrites D).
// All matrices of the iteration are symmetric, so Y's rows serve as its
// columns. With 128-row heads a plane is the 128 x 128 matrix (two boxes).
// With 64-row heads it is stacked: row r holds the 64 columns of its own
// head's block (one box), so D[r][n] is the wanted X_h Y_h^T entry when rows r
// and n are in the same head h (columns 64 h..) and a cross-head value, never
// read, otherwise.
template <int HD>
__device__ __forceinline__ void ns_product(uint32_t d, const unsigned char* xh, const unsigned char* xl,
                                           const unsigned char* yh, const unsigned char* yl, int k0, int k1) {
  const uint32_t id = umma_idesc_bf16(128, 128);
  for (int ks = k0; ks < k1; ++ks) {
    const int j = ks >> 2, kk = ks & 3;
    const uint64_t ah = umma_desc_sw128(xh + j * kBox) + 2 * kk, al = umma_desc_sw128(xl + j * kBox) + 2 * kk;
    const uint64_t bh = umma_desc_sw128(yh + j * kBox) + 2 * kk, bl = umma_desc_sw128(yl + j * kBox) + 2 * kk;
    umma_bf16(d, ah, bh, id, ks != 0);
    umma_bf16(d, ah, bl, id, 1);
    umma_bf16(d, al, bh, id, 1);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Bulk copy of `bytes` (a multiple of 16) from this CTA's shared memory to global memory.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src)),
               "r"(bytes)
               : "memory");
}

}  // namespace

// ----------------------------------------------------------------- Gram ----
// CTA b: unit b / split, boxes [p nb / split, (p + 1) nb / split) of it with
// p = b % split. Warp 0 loads, warp 1 owns TMEM (128 columns) and issues the
// MMAs, warps 2-5 write the partial: row r's columns of its own head block
// (rows padded to head_dim + 4 floats).
__global__ void __launch_bounds__(kGramThreads)
    qkvp_ns_gram_kernel(const __grid_constant__ CUtensorMap tmap_m, const NsArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* ring = align1024(smem_raw);
  __shared__ __align__(8) uint64_t full[kGramStages], empty[kGramStages], done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x / a.split, part = blockIdx.x % a.split;
  const int j0 = (int)((int64_t)part * a.nb / a.split), j1 = (int)((int64_t)(part + 1) * a.nb / a.split);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGramStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    s_fail = 0;
    mbar_init_fence();
  }
  if (warp == 1) tmem_alloc(&s_tmem, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  // The update may come from, and the partials be read by, the kernels before
  // this one. The dependents are let go only after that wait: the apply kernel
  // starts reading the update before its own wait.
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      for (int j = j0, i = 0; j < j1; ++j, ++i) {
        const int s = i % kGramStages;
        if (i >= kGramStages && !ns_wait(&empty[s], ((i / kGramStages) - 1) & 1, a.err, &s_fail)) break;
        mbar_arrive_expect_tx(&full[s], kBox);
        tma_load_2d(ring + s * kBox, &tmap_m, 64 * j, unit * kNsUnitRows, &full[s]);
      }
    }
  } else if (warp == 1) {
    const uint32_t id = umma_idesc_bf16(128, 128);
    for (int j = j0, i = 0; j < j1; ++j, ++i) {
      const int s = i % kGramStages;
      if (!warp_wait(&full[s], (i / kGramStages) & 1, a.err, &s_fail)) break;
      tc_fence_after();
      const uint64_t d = umma_desc_sw128(ring + s * kBox);
#pragma unroll
      for (int k = 0; k < 4; ++k) umma_bf16_warp(tmem, d + 2 * k, d + 2 * k, id, (i | k) != 0);
      umma_commit_warp(&empty[s]);
    }
    umma_commit_warp(&done);
  } else {
    const int q = warp & 3, r = 32 * q + lane;
    const int c0 = a.head_dim == 64 ? 64 * (q >> 1) : 0;  // the row's head block starts at this column
    ns_wait(&done, 0, a.err, &s_fail);
    tc_fence_after();
    float4* dst = reinterpret_cast<float4*>(a.partial + ((size_t)blockIdx.x * kNsUnitRows + r) *
                                                            ns_partial_stride(a.head_dim));
    for (int c = 0; c < a.head_dim; c += 32) {
      float v[32];
      tmem_ld32f(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(c0 + c), v);
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[(c >> 2) + i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 128);
}

// ----------------------------------------------------------- polynomial ----
// One CTA per unit. Shared memory: the hi and lo planes of A (A_k, and Q_k =
// P_k A_k between the products), P_k and M_k, first used to stage the unit's
// Gram partials (bulk copies, up to kStage of them at a time). TMEM: T0
// (columns 0-127: S = A A, then A_{k+1} = Q P), T1 (128-255: Q = P A), T2
// (256-383: M_{k+1} = P M). Warp 1 issues the MMAs: per step S; Q and the first
// half of P M's K steps (all of them for 64-row heads); A' and the rest, so
// that P M fills the tensor pipe while the epilogue writes Q and A'. Warps 2-9
// are the epilogue: warp w holds TMEM lanes (= matrix rows) 32 (w % 4) .. + 31
// and half of each row's HD columns of its head block (HD / 2 per thread), and
// keeps its A_k in fp32 registers for b A + c A A.
template <int HD>
__global__ void __launch_bounds__(kPolyThreads, 1) qkvp_ns_poly_kernel(const NsArgs a) {
  constexpr int W = HD / 2;                   // columns per epilogue thread
  constexpr int kPl = (HD / 64) * kBox;       // bytes of one plane
  constexpr int kNk = HD / 16;                // K steps of a product
  constexpr int kKh = HD == 64 ? kNk : kNk / 2;  // K steps of P M issued after Q
  constexpr int kStride = ns_partial_stride(HD);
  constexpr int kPart = kNsUnitRows * kStride * 4;  // bytes of one staged partial
  constexpr int kStage = ns_poly_stage_parts(HD);
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = align1024(smem_raw);
  unsigned char *Ah = base, *Al = base + kPl, *Ph = base + 2 * kPl, *Pl = base + 3 * kPl;
  unsigned char *Mh = base + 4 * kPl, *Ml = base + 5 * kPl;
  // MMA -> epilogue (one commit each) and epilogue -> MMA (one arrival per epilogue warp)
  __shared__ __align__(8) uint64_t bar_s, bar_q, bar_m, bar_a, bar_e1, bar_e2, bar_e2m, bar_e3, bar_stage;
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail;
  __shared__ float s_diag[kNsUnitRows];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x;

  if (threadIdx.x == 0) {
    mbar_init(&bar_s, 1);
    mbar_init(&bar_q, 1);
    mbar_init(&bar_m, 1);
    mbar_init(&bar_a, 1);
    mbar_init(&bar_e1, kPolyEpiWarps);
    mbar_init(&bar_e2, kPolyEpiWarps);
    mbar_init(&bar_e2m, kPolyEpiWarps);
    mbar_init(&bar_e3, kPolyEpiWarps);
    mbar_init(&bar_stage, 1);
    s_fail = 0;
    mbar_init_fence();
  }
  if (warp == 1) tmem_alloc(&s_tmem, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t T0 = tmem, T1 = tmem + 128, T2 = tmem + 256;
  griddep_launch_dependents();
  griddep_wait();  // the Gram partials

  if (warp == 1) {
    if (lane == 0) {
      for (int k = 0; k < kNsSteps; ++k) {
        const bool last = k == kNsSteps - 1;
        if (!ns_wait(&bar_e3, k & 1, a.err, &s_fail)) break;  // A_k in the A planes
        tc_fence_after();
        ns_product<HD>(T0, Ah, Al, Ah, Al, 0, kNk);  // S = A A
        umma_commit(&bar_s);
        if (!ns_wait(&bar_e1, k & 1, a.err, &s_fail)) break;  // P_k written
        tc_fence_after();
        if (!last) {
          ns_product<HD>(T1, Ph, Pl, Ah, Al, 0, kNk);  // Q = P A
          umma_commit(&bar_q);
        }
        if (k > 0 && !ns_wait(&bar_e2m, (k - 1) & 1, a.err, &s_fail)) break;  // M_k written
        tc_fence_after();
        ns_product<HD>(T2, Ph, Pl, Mh, Ml, 0, last ? kNk : kKh);  // M_{k+1} = P M
        if (!last) {
          if (!ns_wait(&bar_e2, k & 1, a.err, &s_fail)) break;  // Q in the A planes
          tc_fence_after();
          ns_product<HD>(T0, Ah, Al, Ph, Pl, 0, kNk);  // A_{k+1} = Q P
          umma_commit(&bar_a);
          ns_product<HD>(T2, Ph, Pl, Mh, Ml, kKh, kNk);
        }
        umma_commit(&bar_m);
      }
    }
  } else if (warp >= 2) {
    const int q = warp & 3, h2 = (warp - 2) >> 2, r = 32 * q + lane;
    const int cp = W * h2;                                  // first plane column of this thread
    const int tc = (HD == 64 ? 64 * (q >> 1) : 0) + cp;     // its first TMEM column
    const int dj = (r % HD) - cp;                           // the diagonal's index in them, if in [0, W)
    const uint32_t trow = (uint32_t)(32 * q) << 16;
    float A[W];

    // fp32 tensor-memory columns tc .. tc + W - 1 of region t
    auto ld = [&](uint32_t t, float (&v)[W]) {
#pragma unroll
      for (int c = 0; c < W; c += 32) {
        float u[32];
        tmem_ld32f(t + trow + (uint32_t)(tc + c), u);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[c + i] = u[i];
      }
    };
    auto put = [&](unsigned char* hi, unsigned char* lo, const float (&v)[W]) {
#pragma unroll
      for (int c = 0; c < W; c += 8) put8_split(hi, lo, r, cp + c, v + c);
    };
    // this warp's writes are visible to the MMAs (and its TMEM reads done)
    auto signal = [&](uint64_t* bar) {
      tc_fence_before();
      fence_proxy_async_cta();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
    };
    // 1 / (||G_h|| + eps) of this row's head from the diagonal of its Gram
    // block: every warp of the head sums it in the same order
    auto inv_norm = [&]() {
      const int hb = r - r % HD;
      float t = 0.f;
#pragma unroll
      for (int i = 0; i < HD / 32; ++i) t += s_diag[hb + 32 * i + lane];
      t = warp_sum(t);
      return 1.f / (sqrtf(t) + a.eps);
    };

    // ---- A_0: the partials staged and summed in order, the block norms, the scaling
    {
      const int sp = a.split;
      const float* gsrc = a.partial + (size_t)unit * sp * kNsUnitRows * kStride;
      for (int p0 = 0, round = 0; p0 < sp; p0 += kStage, ++round) {
        const int n = sp - p0 < kStage ? sp - p0 : kStage;
        if (round > 0) named_sync(1, kPolyEpiWarps * 32);  // every thread is done with the last round
        if (threadIdx.x == 64) {
          mbar_arrive_expect_tx(&bar_stage, (uint32_t)(n * kPart));
          bulk_load(base, gsrc + (size_t)p0 * kNsUnitRows * kStride, (uint32_t)(n * kPart), &bar_stage,
                    policy_evict_first());
        }
        ns_wait(&bar_stage, round & 1, a.err, &s_fail);
        for (int i = 0; i < n; ++i) {
          const float4* src = reinterpret_cast<const float4*>(base + i * kPart + (r * kStride + cp) * 4);
#pragma unroll
          for (int c = 0; c < W / 4; ++c) {
            const float4 v = src[c];
            if (p0 + i == 0) {
              A[4 * c] = v.x;
              A[4 * c + 1] = v.y;
              A[4 * c + 2] = v.z;
              A[4 * c + 3] = v.w;
            } else {
              A[4 * c] += v.x;
              A[4 * c + 1] += v.y;
              A[4 * c + 2] += v.z;
              A[4 * c + 3] += v.w;
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < W; ++i)
        if (i == dj) s_diag[r] = A[i];
      named_sync(1, kPolyEpiWarps * 32);  // s_diag complete; the staging area is free
      const float inv = inv_norm();
#pragma unroll
      for (int i = 0; i < W; ++i) A[i] = (A[i] * inv) * inv;
      put(Ah, Al, A);
      float e[W];  // M_0 = I
#pragma unroll
      for (int i = 0; i < W; ++i) e[i] = i == dj ? 1.f : 0.f;
      put(Mh, Ml, e);
      signal(&bar_e3);  // phase 0: A_0 and M_0
    }

    for (int k = 0; k < kNsSteps; ++k) {
      const bool last = k == kNsSteps - 1;
      float v[W];
      // ---- P = a I + b A + c S
      ns_wait(&bar_s, k & 1, a.err, &s_fail);
      tc_fence_after();
      ld(T0, v);
#pragma unroll
      for (int i = 0; i < W; ++i) {
        v[i] = fmaf(kNsC, v[i], kNsB * A[i]);
        if (i == dj) v[i] += kNsA;
      }
      put(Ph, Pl, v);
      signal(&bar_e1);
      if (!last) {
        // ---- Q = P A into the A planes
        ns_wait(&bar_q, k & 1, a.err, &s_fail);
        tc_fence_after();
        ld(T1, v);
        put(Ah, Al, v);
        signal(&bar_e2);
        // ---- A_{k+1} = Q P
        ns_wait(&bar_a, k & 1, a.err, &s_fail);
        tc_fence_after();
        ld(T0, A);
        put(Ah, Al, A);
        signal(&bar_e3);
      }
      // ---- M_{k+1} = P M
      ns_wait(&bar_m, k & 1, a.err, &s_fail);
      tc_fence_after();
      ld(T2, v);
      if (!last) {
        put(Mh, Ml, v);
        signal(&bar_e2m);
      } else {
        // M (1 / (||G|| + eps)) * factor as the apply pass's image: the hi and
        // lo planes of the block-diagonal 128 x 128 matrix, 64 KiB from base
        // (the A and P planes, no longer read by any MMA)
        const float f = inv_norm() * a.scale;
#pragma unroll
        for (int i = 0; i < W; ++i) v[i] *= f;
        tc_fence_before();
        if (HD == 64) {  // the off-diagonal blocks are 0
          for (int i = threadIdx.x - 64; i < 4 * kBox / 16; i += kPolyEpiWarps * 32)
            reinterpret_cast<uint4*>(base)[i] = make_uint4(0, 0, 0, 0);
          named_sync(1, kPolyEpiWarps * 32);
        }
        const int c0 = (HD == 64 ? 64 * (r >> 6) : 0) + cp;
#pragma unroll
        for (int c = 0; c < W; c += 8) put8_split(base, base + 2 * kBox, r, c0 + c, v + c);
        fence_proxy_async_cta();
        named_sync(1, kPolyEpiWarps * 32);
        if (threadIdx.x == 64) {
          bulk_store(a.mh + (size_t)unit * (4 * kBox / 16), base, 4 * kBox);
          bulk_commit();
          bulk_wait_all();
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- apply ----
// Persistent: CTA c takes the boxes [c n / grid, (c + 1) n / grid) of the
// n = units * nb boxes of 128 rows x 64 columns, in unit-major order. Warp 0
// loads the boxes of G; warp 1 loads the unit's M image (64 KiB, when the unit
// changes, after its MMAs on the previous one are done: meanwhile the loads of
// G run on) and issues out_box = (M_hi + M_lo) G_box (K = the unit's 128 rows,
// G as the MN-major B operand) into one of 8 accumulators of 64 TMEM columns;
// warps 2-5 round the result to bf16, write it over the G box it came from and
// store it by TMA (32 rows per warp), then hand the ring slot back once the
// store has read it.
__global__ void __launch_bounds__(kApplyThreads, 1)
    qkvp_ns_apply_kernel(const __grid_constant__ CUtensorMap tmap_m, const __grid_constant__ CUtensorMap tmap_out,
                         const NsArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* mimg = align1024(smem_raw);    // hi plane, lo plane
  unsigned char* ring = mimg + 2 * kPlane;      // kApplyStages boxes
  __shared__ __align__(8) uint64_t full[kApplyStages], empty[kApplyStages], tfull[kApplyAcc], tempty[kApplyAcc];
  __shared__ __align__(8) uint64_t bar_mh, mh_free;
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n = (int64_t)a.units * a.nb;
  const int64_t i0 = n * blockIdx.x / gridDim.x, i1 = n * (blockIdx.x + 1) / gridDim.x;
  const int cnt = (int)(i1 - i0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kApplyStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    for (int b = 0; b < kApplyAcc; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(&bar_mh, 1);
    mbar_init(&mh_free, 1);
    s_fail = 0;
    mbar_init_fence();
  }
  if (warp == 1) tmem_alloc(&s_tmem, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // The first boxes of G go out before the wait for the polynomial kernel
      // (G itself was ready before the Gram kernel let its dependents go);
      // the rest of the kernel waits for M.
      const uint64_t pol = policy_evict_first();  // the last read of G
      for (int t = 0; t < cnt; ++t) {
        if (t == kApplyStages) griddep_wait();
        const int64_t i = i0 + t;
        const int u = (int)(i / a.nb), j = (int)(i % a.nb);
        const int s = t % kApplyStages;
        if (t >= kApplyStages && !ns_wait(&empty[s], ((t / kApplyStages) - 1) & 1, a.err, &s_fail)) break;
        mbar_arrive_expect_tx(&full[s], kBox);
        tma_load_2d_hint(ring + s * kBox, &tmap_m, 64 * j, u * kNsUnitRows, &full[s], pol);
      }
    }
  } else if (warp == 1) {
    griddep_wait();  // M from the polynomial kernel
    const uint32_t id = umma_idesc_bf16_bmn(128, 64);
    int cur = -1, nchg = 0;
    for (int t = 0; t < cnt; ++t) {
      const int u = (int)((i0 + t) / a.nb);
      if (u != cur) {  // the unit's M image, once the MMAs on the previous one are done
        if (nchg > 0) {
          umma_commit_warp(&mh_free);
          if (!warp_wait(&mh_free, (nchg - 1) & 1, a.err, &s_fail)) break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar_mh, 2 * kPlane);
          bulk_load(mimg, a.mh + (size_t)u * (2 * kPlane / 16), 2 * kPlane, &bar_mh, policy_evict_normal());
        }
        if (!warp_wait(&bar_mh, nchg & 1, a.err, &s_fail)) break;
        cur = u;
        ++nchg;
      }
      const int s = t % kApplyStages, b = t % kApplyAcc;
      if (!warp_wait(&full[s], (t / kApplyStages) & 1, a.err, &s_fail)) break;
      if (t >= kApplyAcc && !warp_wait(&tempty[b], ((t / kApplyAcc) - 1) & 1, a.err, &s_fail)) break;
      tc_fence_after();
      const uint64_t bd = umma_desc_sw128_mn(ring + s * kBox, kBox);
#pragma unroll
      for (int p = 0; p < 2; ++p) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = umma_desc_sw128(mimg + p * kPlane + (kk >> 2) * kBox) + 2 * (kk & 3);
          umma_bf16_warp(tmem + 64 * b, ad, bd + (uint64_t)(128 * kk), id, (p | kk) != 0);  // +2048 B: 16 rows of G
        }
      }
      umma_commit_warp(&tfull[b]);
    }
  } else {
    griddep_wait();  // the output may still be read by the kernels before this one
    // two groups of four warps take alternate boxes, so that one group's
    // stores drain while the other converts
    const int q = warp & 3, g = (warp - 2) >> 2, r = 32 * q + lane;
    const uint32_t trow = (uint32_t)(32 * q) << 16;
    int prev = -1;
    for (int t = g; t < cnt; t += 2) {
      const int64_t i = i0 + t;
      const int u = (int)(i / a.nb), j = (int)(i % a.nb);
      const int s = t % kApplyStages, b = t % kApplyAcc;
      if (!ns_wait(&tfull[b], (t / kApplyAcc) & 1, a.err, &s_fail)) break;
      tc_fence_after();
      float v0[32], v1[32];
      tmem_ld32f(tmem + trow + (uint32_t)(64 * b), v0);
      tmem_ld32f(tmem + trow + (uint32_t)(64 * b + 32), v1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[b]);
      unsigned char* box = ring + s * kBox;  // the G box this result came from (the MMAs are done with it)
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const float* v = ch < 4 ? v0 + 8 * ch : v1 + 8 * (ch - 4);
        *reinterpret_cast<uint4*>(box + swz(r, ch)) =
            make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
      }
      fence_proxy_async_cta();
      __syncwarp();
      if (lane == 0) {
        const int row0 = u * kNsUnitRows + 32 * q;
        if (row0 < a.rows) tma_store_2d(&tmap_out, box + 32 * q * 128, 64 * j, row0);
        bulk_commit();
        if (prev >= 0) {  // this warp's previous box's store has read its slot: hand it back
          bulk_wait_read_but1();
          mbar_arrive(&empty[prev % kApplyStages]);
        }
      }
      prev = t;
      __syncwarp();
    }
    if (lane == 0) bulk_wait_all();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

const void* ns_gram_kernel() { return reinterpret_cast<const void*>(&qkvp_ns_gram_kernel); }
const void* ns_poly_kernel(int head_dim) {
  return head_dim == 64 ? reinterpret_cast<const void*>(&qkvp_ns_poly_kernel<64>)
                        : reinterpret_cast<const void*>(&qkvp_ns_poly_kernel<128>);
}
const void* ns_apply_kernel() { return reinterpret_cast<const void*>(&qkvp_ns_apply_kernel); }
int ns_gram_smem_bytes() { return kGramStages * kBox + 1024; }
int ns_poly_smem_bytes(int head_dim) {
  const int planes = 6 * (head_dim / 64) * kBox;
  const int stage = ns_poly_stage_parts(head_dim) * kNsUnitRows * ns_partial_stride(head_dim) * 4;
  return (planes > stage ? planes : stage) + 1024;
}
int ns_apply_smem_bytes() { return 2 * kPlane + kApplyStages * kBox + 1024; }
int ns_gram_threads() { return kGramThreads; }
int ns_poly_threads() { return kPolyThreads; }
int ns_apply_threads() { return kApplyThreads; }

}  // namespace qkvp
