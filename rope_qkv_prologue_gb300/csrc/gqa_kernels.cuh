// Forward and backward kernels of the packed-QKV prologue for the GQA packings.
//
// Work decomposition. A token's packed row is cpt = heads * head_dim / 8
// 16-byte chunks. The (token, chunk) pairs of the whole batch are numbered
// t * cpt + j and cut into work items of kThreads * U consecutive chunks; a
// CTA takes items round-robin (grid = a multiple of the SM count, capped by
// the number of items). Thread `tid` handles chunks u * kThreads + tid of the
// item, so:
//   * a warp covers 32 consecutive chunks = 32 / CPH whole heads (item and
//     head boundaries are multiples of CPH), hence every chunk of a thread
//     sits at the same position e = tid % CPH inside its head and the thread
//     keeps the 8 weights of that position in registers;
//   * the RMSNorm sum of squares of a head is a 3-step (CPH = 8) xor-shuffle
//     reduction inside the CPH-lane group;
//   * the rotate-half partner of element d is element d +- head_dim/2, held by
//     lane (lane ^ CPH/2) at the same position of its chunk: one xor-shuffle.
// cos / sin depend only on (token, frequency): an item first writes them for
// the few tokens it touches into shared memory, and all of its heads read
// them back.
//
// Every global access is a 16-byte vector access; a warp's loads and stores
// cover whole 128-byte head rows (coalesced).
#pragma once

#include "common.cuh"
#include "qkv_prologue.h"

namespace qkvp {

template <int HD>
struct Geom {
  static constexpr int CPH = HD / 8;   // 16-byte chunks per head
  static constexpr int HALF = HD / 2;  // RoPE frequencies
  static constexpr int LOG_CPH = HD == 64 ? 3 : 4;
  static_assert(HD == 64 || HD == 128, "head_dim 64 or 128");
};

// Which output head a packed chunk belongs to.
template <bool SECTIONED>
__device__ __forceinline__ void classify(uint32_t hp, int n_q, int n_kv, int group,
                                         uint32_t gs_magic, int& role, uint32_t& oh) {
  if (SECTIONED) {
    // [n_q q heads | n_kv k heads | n_kv v heads]
    if (hp < (uint32_t)n_q) {
      role = kRoleQ;
      oh = hp;
    } else if (hp < (uint32_t)(n_q + n_kv)) {
      role = kRoleK;
      oh = hp - n_q;
    } else {
      role = kRoleV;
      oh = hp - n_q - n_kv;
    }
  } else {
    // [n_kv groups][group q heads, 1 k head, 1 v head]
    const uint32_t g = small_div(hp, gs_magic);
    const uint32_t s = hp - g * (uint32_t)(group + 2);
    role = s < (uint32_t)group ? kRoleQ : (s == (uint32_t)group ? kRoleK : kRoleV);
    oh = role == kRoleQ ? g * group + s : g;
  }
}

// cos and signed sin of frequencies f0 .. f0+7 of table row tl, as pairs;
// ssin = sign * sin.
template <int HALF>
__device__ __forceinline__ void read_cos_sin(const float* s_cos, const float* s_sin, uint32_t tl, int f0,
                                             float sign, float2 (&c)[4], float2 (&ssin)[4]) {
  float2 sn[4];
  load_pairs(s_cos + tl * HALF + f0, c);
  load_pairs(s_sin + tl * HALF + f0, sn);
  const float2 sg = f2(sign, sign);
#pragma unroll
  for (int i = 0; i < 4; ++i) ssin[i] = __fmul2_rn(sn[i], sg);
}

// Fill the shared cos/sin table for tokens t_first .. t_first + ntok - 1.
template <int HALF>
__device__ __forceinline__ void fill_rope_table(const int32_t* pos, const RopeTable& rope,
                                                int64_t t_first, int ntok, float* s_cos,
                                                float* s_sin) {
  for (int i = threadIdx.x; i < ntok * HALF; i += kThreads) {
    const int tl = i / HALF;
    const int f = i % HALF;
    float c, s;
    rope_cos_sin(pos[t_first + tl], rope.turns[f], rope.scale, &c, &s);
    s_cos[i] = c;
    s_sin[i] = s;
  }
}

// ------------------------------------------------------------- forward ----

template <int HD, bool SECTIONED, bool ROPE, bool SAVE, bool POOL, bool NORM, bool BIAS>
__global__ void __launch_bounds__(kThreads, 2) qkvp_fwd_kernel(const FwdArgs a) {
  griddep_wait();
  using G = Geom<HD>;
  constexpr int CPH = G::CPH, HALF = G::HALF, U = kFwdChunksPerThread;
  extern __shared__ __align__(16) unsigned char smem[];
  float* s_cos = reinterpret_cast<float*>(smem);
  float* s_sin = s_cos + a.max_tok * HALF;
  int32_t* s_slot = reinterpret_cast<int32_t*>(s_sin + a.max_tok * HALF);

  const int tid = threadIdx.x;
  const int e = tid & (CPH - 1);
  const float sign = e < CPH / 2 ? -1.f : 1.f;
  const int f0 = (e & (CPH / 2 - 1)) * 8;
  float2 wq[4], wk[4];
  if (NORM) {
    load_pairs(a.w_q + 8 * e, wq);
    load_pairs(a.w_k + 8 * e, wk);
  }

  const int64_t total = a.T * a.cpt;
  for (int64_t item = blockIdx.x; item < a.n_items; item += gridDim.x) {
    const int64_t c0 = item * a.item_chunks;
    const int nch = (int)min(a.item_chunks, total - c0);
    const int64_t t_first = c0 / a.cpt;
    const int s0 = (int)(c0 - t_first * a.cpt);
    const int ntok = (int)((c0 + nch - 1) / a.cpt - t_first + 1);

    uint4 xv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int cl = u * kThreads + tid;
      xv[u] = make_uint4(0u, 0u, 0u, 0u);
      if (cl < nch) {
        const uint32_t n = (uint32_t)(cl + s0);
        const uint32_t tl = small_div(n, a.cpt_magic);
        const uint32_t j = n - tl * (uint32_t)a.cpt;
        xv[u] = ld_stream(a.packed + (t_first + tl) * a.row_stride16 + j);
      }
    }

    __syncthreads();  // readers of the previous item's table are done
    if (ROPE) fill_rope_table<HALF>(a.pos, a.rope, t_first, ntok, s_cos, s_sin);
    if (POOL) {
      for (int i = tid; i < ntok; i += kThreads) {
        const int32_t pg = a.page[t_first + i], of = a.offset[t_first + i];
        int bad = 0;
        if (pg < 0 || pg >= a.num_pages) bad |= QKVP_DEV_BAD_PAGE;
        if (of < 0 || of >= a.page_size) bad |= QKVP_DEV_BAD_OFFSET;
        if (bad && a.dev_status) atomicOr(a.dev_status, bad);
        s_slot[i] = bad ? -1 : pg * a.page_size + of;
      }
    }
    __syncthreads();

#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int cl = u * kThreads + tid;
      const bool valid = cl < nch;
      const uint32_t n = (uint32_t)((valid ? cl : 0) + s0);
      const uint32_t tl = small_div(n, a.cpt_magic);
      const uint32_t j = n - tl * (uint32_t)a.cpt;
      int role;
      uint32_t oh;
      classify<SECTIONED>(j >> G::LOG_CPH, a.n_q, a.n_kv, a.group, a.gs_magic, role, oh);

      float2 x[4], w[4], c[4], ssin[4], y[4];
      unpack_pairs(xv[u], x);
      if (BIAS) {
        float2 b[4];
        load_pairs(a.bias + 8 * j, b);
        add_bias_pairs(x, b);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = NORM ? (role == kRoleQ ? wq[i] : wk[i]) : f2(1.f, 1.f);
      if (ROPE) read_cos_sin<HALF>(s_cos, s_sin, tl, f0, sign, c, ssin);
      chunk_forward<CPH, ROPE, NORM>(x, w, a.eps, a.inv_head_dim, c, ssin, y);
      if (!valid) continue;

      const int64_t t = t_first + tl;
      const uint4 out = pack_pairs(y);
      const uint4 vout = BIAS ? pack_pairs(x) : xv[u];  // v: the (biased) input
      if (role == kRoleQ) {
        const int64_t idx = (t * a.n_q + oh) * CPH + e;
        st_keep(a.q + idx, out);
        if (SAVE) st_stream(a.q_pre + idx, xv[u]);
      } else if (POOL) {
        const int32_t slot = s_slot[tl];
        if (slot >= 0) {
          const int64_t idx = ((int64_t)slot * a.n_kv + oh) * CPH + e;
          if (role == kRoleK) st_keep(a.k_pool + idx, out);
          else st_keep(a.v_pool + idx, vout);
        }
      } else {
        const int64_t idx = (t * a.n_kv + oh) * CPH + e;
        if (role == kRoleK) {
          st_keep(a.k + idx, out);
          if (SAVE) st_stream(a.k_pre + idx, xv[u]);
        } else {
          st_keep(a.v + idx, vout);
        }
      }
    }
  }
}

// ------------------------------------------------------------ backward ----
//
// For an output chunk of the packed gradient at (token t, position j): find
// its head; v heads copy dv; q/k heads read the gradient d of the roped output
// and the saved pre-norm input x, and compute
//   g  = R(theta)^T d                      (rotate by -theta; or g = d on NoPE)
//   r  = (mean(x^2) + eps)^-1/2
//   dx = r w g - x (r^3 / D) sum_d(x w g)
//   dw += g x r                             (per thread, fp32 registers)
// The CTA reduces its dw partial sums in a fixed order and writes one row of
// `partials`; qkvp_dw_finalize_kernel adds the rows in float64.
// Without the norm: dx = g, no dw, and the saved inputs are not read. With a
// qkv bias the norm's input is x + b, and the bias gradient db = sum over
// tokens of dx: the host then makes every work item one whole token, so a
// thread always holds the same packed chunks and adds them into the CTA's row
// of float sums in shared memory (no two threads share a chunk; the order is
// fixed), written out as one row of `db_partials`.

template <int HD, bool SECTIONED, bool ROPE, bool NORM, bool BIAS>
__global__ void __launch_bounds__(kThreads, 2) qkvp_bwd_kernel(const BwdArgs a) {
  griddep_wait();
  using G = Geom<HD>;
  constexpr int CPH = G::CPH, HALF = G::HALF, U = kBwdChunksPerThread;
  extern __shared__ __align__(16) unsigned char smem[];
  float* s_cos = reinterpret_cast<float*>(smem);
  float* s_sin = s_cos + a.max_tok * HALF;
  float* s_db = s_sin + a.max_tok * HALF;  // [cpt * 8] (BIAS)
  __shared__ float s_red[kThreads / 32][2][HD];

  const int tid = threadIdx.x;
  const int e = tid & (CPH - 1);
  const float sign = e < CPH / 2 ? 1.f : -1.f;  // R(theta)^T: the partner term flips sign
  const int f0 = (e & (CPH / 2 - 1)) * 8;
  float2 wq[4], wk[4], accq[4], acck[4];
  if (NORM) {
    load_pairs(a.w_q + 8 * e, wq);
    load_pairs(a.w_k + 8 * e, wk);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) accq[i] = acck[i] = f2(0.f, 0.f);
  if (BIAS) {
    for (int i = tid; i < a.cpt * 8; i += kThreads) s_db[i] = 0.f;
  }

  const int64_t total = a.T * a.cpt;
  for (int64_t item = blockIdx.x; item < a.n_items; item += gridDim.x) {
    const int64_t c0 = item * a.item_chunks;
    const int nch = (int)min(a.item_chunks, total - c0);
    const int64_t t_first = c0 / a.cpt;
    const int s0 = (int)(c0 - t_first * a.cpt);
    const int ntok = (int)((c0 + nch - 1) / a.cpt - t_first + 1);

    uint4 dv[U], xv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int cl = u * kThreads + tid;
      dv[u] = xv[u] = make_uint4(0u, 0u, 0u, 0u);
      if (cl < nch) {
        const uint32_t n = (uint32_t)(cl + s0);
        const uint32_t tl = small_div(n, a.cpt_magic);
        const uint32_t j = n - tl * (uint32_t)a.cpt;
        int role;
        uint32_t oh;
        classify<SECTIONED>(j >> G::LOG_CPH, a.n_q, a.n_kv, a.group, a.gs_magic, role, oh);
        const int64_t t = t_first + tl;
        if (role == kRoleQ) {
          const int64_t idx = (t * a.n_q + oh) * CPH + e;
          dv[u] = ld_stream(a.dq + idx);
          if (NORM) xv[u] = ld_stream(a.q_pre + idx);
        } else {
          const int64_t idx = (t * a.n_kv + oh) * CPH + e;
          if (role == kRoleK) {
            dv[u] = ld_stream(a.dk + idx);
            if (NORM) xv[u] = ld_stream(a.k_pre + idx);
          } else {
            dv[u] = ld_stream(a.dv + idx);
          }
        }
      }
    }

    __syncthreads();
    if (ROPE) fill_rope_table<HALF>(a.pos, a.rope, t_first, ntok, s_cos, s_sin);
    __syncthreads();

#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int cl = u * kThreads + tid;
      const bool valid = cl < nch;
      const uint32_t n = (uint32_t)((valid ? cl : 0) + s0);
      const uint32_t tl = small_div(n, a.cpt_magic);
      const uint32_t j = n - tl * (uint32_t)a.cpt;
      int role;
      uint32_t oh;
      classify<SECTIONED>(j >> G::LOG_CPH, a.n_q, a.n_kv, a.group, a.gs_magic, role, oh);

      float2 d[4], x[4], w[4], c[4], ssin[4], dx[4], gx[4];
      float r;
      unpack_pairs(dv[u], d);
      unpack_pairs(xv[u], x);
      if (NORM && BIAS) {
        float2 b[4];
        load_pairs(a.bias + 8 * j, b);
        add_bias_pairs(x, b);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = NORM ? (role == kRoleQ ? wq[i] : wk[i]) : f2(1.f, 1.f);
      if (ROPE) read_cos_sin<HALF>(s_cos, s_sin, tl, f0, sign, c, ssin);
      chunk_backward<CPH, ROPE, NORM>(d, x, w, a.eps, a.inv_head_dim, c, ssin, dx, gx, r);
      if (!valid) continue;

      if (NORM) {
        const float rq = role == kRoleQ ? r : 0.f, rk = role == kRoleK ? r : 0.f;
        const float2 rq2 = f2(rq, rq), rk2 = f2(rk, rk);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          accq[i] = __ffma2_rn(gx[i], rq2, accq[i]);
          acck[i] = __ffma2_rn(gx[i], rk2, acck[i]);
        }
      }
      if (BIAS) {  // one token per item: chunk j is this thread's on every item
        float* p = s_db + 8 * j;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 g = role == kRoleV ? d[i] : dx[i];
          p[2 * i] += g.x;
          p[2 * i + 1] += g.y;
        }
      }
      const int64_t t = t_first + tl;
      st_keep(a.dpacked + t * a.row_stride16 + j, role == kRoleV ? dv[u] : pack_pairs(dx));
    }
  }

  if (BIAS) {
    __syncthreads();
    for (int i = tid; i < a.cpt * 8; i += kThreads) a.db_partials[(int64_t)blockIdx.x * a.cpt * 8 + i] = s_db[i];
  }
  if (!NORM) return;

  // Weight-grad partials: lanes of a warp with the same e, then the warps.
  float aq[8], ak[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    aq[2 * i] = accq[i].x; aq[2 * i + 1] = accq[i].y;
    ak[2 * i] = acck[i].x; ak[2 * i + 1] = acck[i].y;
  }
#pragma unroll
  for (int o = CPH; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      aq[i] += __shfl_xor_sync(0xffffffffu, aq[i], o);
      ak[i] += __shfl_xor_sync(0xffffffffu, ak[i], o);
    }
  }
  const int lane = tid & 31, warp = tid >> 5;
  if (lane < CPH) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      s_red[warp][0][lane * 8 + i] = aq[i];
      s_red[warp][1][lane * 8 + i] = ak[i];
    }
  }
  __syncthreads();
  for (int i = tid; i < 2 * HD; i += kThreads) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) sum += s_red[w][i / HD][i % HD];
    a.partials[(int64_t)blockIdx.x * 2 * HD + i] = sum;
  }
}

}  // namespace qkvp
